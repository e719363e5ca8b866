"""Host logic of bench.py that needs no GPU: the DRAM traffic it reports comes
from the committed ncu record only while the kernel sources hash to the value
recorded with it, and the decode layer's traffic is its two kernels' summed."""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCES = ("qg_ffn.cu", "qg_stack.cu", "qg_norm.cuh", "qg_common.cuh")


def _bench():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench

    return bench


def _tree(tmp_path, records):
    csrc = tmp_path / "block_quantized_decode_rmsnorm_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for i, f in enumerate(SOURCES):
        (csrc / f).write_text(f"// source {i}\n")
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(records))
    return csrc


def test_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    bench = _bench()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    csrc = _tree(tmp_path, {})
    h = bench.kernel_source_hash()
    recs = {"ffn_up_kernel": {"dram_bytes_per_launch": 7000, "source_sha256": h},
            "gemv_prefetch_kernel": {"dram_bytes_per_launch": 3000, "source_sha256": h}}
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(recs))
    assert bench.ncu_traffic("ffn_up_kernel") == 7000
    assert bench.ncu_traffic("layer_pair") == 10000
    assert bench.ncu_traffic("decode_stack_kernel") is None  # no record
    # any change to a hashed source voids every record taken before it
    (csrc / "qg_common.cuh").write_text("// source 3, edited\n")
    assert bench.kernel_source_hash() != h
    assert bench.ncu_traffic("ffn_up_kernel") is None
    assert bench.ncu_traffic("layer_pair") is None


def test_layer_pair_needs_both_records(tmp_path, monkeypatch):
    bench = _bench()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _tree(tmp_path, {})
    h = bench.kernel_source_hash()
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(
        json.dumps({"ffn_up_kernel": {"dram_bytes_per_launch": 7000, "source_sha256": h}}))
    assert bench.ncu_traffic("layer_pair") is None


def test_committed_record_covers_the_decode_kernels():
    """The committed record names the kernels the bench looks up, each with its
    capture command and a byte count within 1 % of the algorithmic bytes."""
    recs = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
    algorithmic = {"ffn_up_kernel": 7825120, "gemv_prefetch_kernel": 3911392}
    for k, a in algorithmic.items():
        r = recs[k]
        assert "ncu" in r["command"] and "--clock-control none" in r["command"]
        assert abs(r["dram_bytes_per_launch"] - a) / a < 0.01
    assert recs["decode_stack_kernel"]["dram_read"] > 24 * 11_698_176 * 0.99
