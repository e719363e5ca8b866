#!/usr/bin/env python
"""Benchmark of the Q8_0 decode path on GB300.

Headline workload: the decode feed-forward block of a 0.8B-shaped model (hidden
1024, stacked gate|up 7168 x 1024, down 1024 x 3584, Q8_0 weights), batch 1.
One step = one decode step's worth of that block: L chained layers (default 24)
with distinct weights, replayed as one CUDA graph.  Each layer is two launches
(--path two, the default): RMSNorm + Q8_0 of x + stacked gate|up + SiLU*u + Q8_0
of h in one kernel, then the down GEMV with the residual folded in.  --path four
runs the same layer unfused (4 launches), --path one as one launch per layer.
The weights of one step (L x 11.7 MB) exceed the L2 cache, so every step streams
them from HBM.

Metric: achieved HBM GB/s = algorithmic bytes of the step / step time.  The line
also carries the roofline of the layer (its two launches overlap, so the unit is
the layer: both projections' bytes over the step time per layer, with both
kernels' DRAM traffic and the gate|up kernel timed alone as context), an
end-to-end number through pinned host buffers (input read and result written by
the first and last layers, the host waiting every step), the CPU oracle timed on
the host, the SM clocks sampled during the timed region, and (unless --quick) the
other workloads' kernel rates: Q8_0 GEMV 256x1024, bf16 projection 18432x2560,
output-head GEMV 262144x1024 at batch 1/2/4/8, the bf16 and Q8_0 prompt
contractions for 512 rows, and the int8 mma.sync rate.

--impl reference times the CPU oracle (the only reference this method has) on
the same workload and prints the same line with "impl": "reference".
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Q8_0 decode GEMV achieved HBM GB/s (% of GB300 peak); prefill int8 TOPS"
HIDDEN, FFN = 1024, 3584
EPS = 1e-6
# algorithmic bytes of one FFN layer: both weights (values + binary16 scales),
# the input row x (f32), the RMSNorm gain (f32) and the output row (f32)
W_GU_BYTES = 2 * FFN * HIDDEN + 2 * FFN * (HIDDEN // 32) * 2
W_DN_BYTES = HIDDEN * FFN + HIDDEN * (FFN // 32) * 2
LAYER_BYTES = W_GU_BYTES + W_DN_BYTES + 3 * HIDDEN * 4
# fused gate|up launch: weights, x and gamma in (f32), h out (f32) and its Q8_0 codes + scales
GU_KERNEL_BYTES = W_GU_BYTES + 2 * HIDDEN * 4 + FFN * 4 + FFN + (FFN // 32) * 2
# persistent stack kernel over n layers: every layer's weights and gain, the input and the output row
def STACK_KERNEL_BYTES(n: int) -> int:
    return n * (W_GU_BYTES + W_DN_BYTES + HIDDEN * 4) + 2 * HIDDEN * 4


# one-launch layer: both weights, x in, gamma, x out, the cleared buffer, h and its codes and scales
LAYER_KERNEL_BYTES = W_GU_BYTES + W_DN_BYTES + 4 * HIDDEN * 4 + FFN * 4 + FFN + (FFN // 32) * 2


def workload_name(layers: int) -> str:
    return (f"decode FFN, 0.8B-shaped (hidden {HIDDEN}, stacked gate|up {2 * FFN}x{HIDDEN}, down {HIDDEN}x{FFN}, "
            f"Q8_0), batch 1, {layers} chained layers with distinct weights per step")


def peaks():
    p = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}
    f = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(f):
        m = json.load(open(f))
        for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
            if k in m:
                p[k] = float(m[k])
        p["source"] = "measured"
    return p


# --------------------------------------------------------------------------
# clocks during the timed region (NVML read-only queries)
# --------------------------------------------------------------------------
REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
           0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
           0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}


class ClockSampler:
    """Polls the SM clock and the clock-event reasons of this process's GPU."""

    def __init__(self, torch, dev: int):
        self.ok = False
        self.samples = []
        self.reasons = 0
        self.max_mhz = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            pr = torch.cuda.get_device_properties(dev)
            bus = f"{getattr(pr, 'pci_domain_id', 0):08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
                if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(dev), ctypes.byref(h)) != 0:
                    return
            self.nv, self.h = nv, h
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._reason_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self.ok = True
        except (OSError, AttributeError):
            self.ok = False

    def _read(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0:
            self.samples.append(clk.value)
        if self._reason_fn(self.h, ctypes.byref(rs)) == 0:
            self.reasons |= rs.value

    def start(self):
        self.samples, self.reasons = [], 0
        self._stop = threading.Event()
        if not self.ok:
            return
        self._read()

        def loop():
            while not self._stop.wait(0.002):
                self._read()

        self._t = threading.Thread(target=loop, daemon=True)
        self._t.start()

    def stop(self):
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"], "samples": 0}
        self._stop.set()
        self._t.join()
        self._read()
        names = [n for b, n in REASONS.items() if self.reasons & b and b != 0x1]
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None, "sm_max_mhz": self.max_mhz,
                "reasons": names, "samples": len(self.samples)}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    import platform
    import subprocess

    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def gpu_processes():
    """Compute processes on the GPUs as nvidia-smi lists them ("pid, name, memory"),
    or None when the query is unavailable."""
    import subprocess

    try:
        r = subprocess.run(["nvidia-smi", "--query-compute-apps=pid,process_name,used_memory", "--format=csv,noheader"],
                           capture_output=True, text=True, timeout=20)
    except (OSError, subprocess.SubprocessError):
        return None
    if r.returncode != 0:
        return None
    return [ln.strip() for ln in r.stdout.splitlines() if ln.strip()]


def other_processes(procs):
    if procs is None:
        return None
    me = str(os.getpid())
    return [p for p in procs if p.split(",")[0].strip() != me]


# --------------------------------------------------------------------------
# distributed plumbing (one process per GPU; no collective on the data path)
# --------------------------------------------------------------------------
class Dist:
    """One process per GPU under torchrun: barrier and max-over-ranks timing.
    NCCL on GPUs; gloo (tensors on the host) when asked, which is how the
    multi-rank logic is exercised on a CPU-only machine."""

    def __init__(self, torch, backend: str = "nccl"):
        self.torch = torch
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        self.device = "cuda" if backend == "nccl" else "cpu"
        if self.world > 1:
            import torch.distributed as dist

            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        t = self.torch.tensor([v], dtype=self.torch.float64, device=self.device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def job_rate(world: int, steps: int, unit_bytes: int, max_elapsed_s: float) -> float:
    """Whole-job GB/s: every rank processes `steps` units of `unit_bytes`; the
    job takes as long as its slowest rank."""
    return world * steps * unit_bytes / max_elapsed_s / 1e9


# --------------------------------------------------------------------------
# the workload on the GPU
# --------------------------------------------------------------------------
def make_layers(torch, n_layers: int, seed: int = 0):
    from block_quantized_decode_rmsnorm_gb300 import api, synth

    layers = []
    for l in range(n_layers):
        c = synth.ffn_case(seed, HIDDEN, FFN, layer=l)
        layers.append(api.FFNLayer(torch.from_numpy(c["gamma"]).cuda(),
                                   api.q8_weight_from_numpy(c["gu_qs"], c["gu_d"]),
                                   api.q8_weight_from_numpy(c["dn_qs"], c["dn_d"])))
        if l == 0:
            x0 = c["x"]
    return layers, x0


_WARM_STREAM = []


def capture(torch, fn):
    """Record fn() (which launches on the current stream) into a CUDA graph.

    The warm-up run goes to one side stream kept for the whole process.  With a
    new side stream for every capture (event waits both ways with the replay
    stream), every decode-step graph of the process, old and new, ran at
    119-120 instead of 102.5 us from the eighth such stream on (measured on
    GB300, reproducible, independent of CUDA_DEVICE_MAX_CONNECTIONS; no clock or
    throttle change)."""
    if not _WARM_STREAM:
        _WARM_STREAM.append(torch.cuda.Stream())
    s = _WARM_STREAM[0]
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm the launch paths outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_graph(torch, g, iters: int) -> float:
    """Seconds per replay, CUDA events on the replay stream."""
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3 / iters


def replay_trials(torch, g, per: int, trials: int = 20) -> dict:
    """Seconds per launch over `trials` separately timed replays of g (each
    replay `per` launches): median, 10th and 90th percentiles."""
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(trials):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) / 1e3 / per)
    ts.sort()
    return {"median": statistics.median(ts), "p10": ts[round(0.1 * (trials - 1))],
            "p90": ts[round(0.9 * (trials - 1))], "trials": trials}


def cold_and_warm(torch, launch, ws, wbytes: int) -> dict:
    """Per-launch time of launch(w): cold, over the rotating copies ws (>= 4x L2,
    one graph), and warm, 20 launches on ws[0] (only where a copy fits in half
    of L2), each over 20 timed replays."""
    g = capture(torch, lambda: [launch(w) for w in ws])
    st = replay_trials(torch, g, len(ws))
    del g
    out = {"us": st["median"] * 1e6, "us_p10": st["p10"] * 1e6, "us_p90": st["p90"] * 1e6,
           "trials": st["trials"], "copies": len(ws)}
    if 2 * wbytes <= torch.cuda.get_device_properties(0).L2_cache_size:
        gw = capture(torch, lambda: [launch(ws[0]) for _ in range(20)])
        out["us_warm_l2"] = replay_trials(torch, gw, 20)["median"] * 1e6
        del gw
    return out


def l2_copies(torch, bytes_one: int) -> int:
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    return max(2, -(-4 * l2 // bytes_one))


def replicate_q8(torch, api, w0, copies: int):
    """`copies` distinct device copies of a packed weight, carved from one allocation."""
    qs = torch.empty((copies,) + tuple(w0.qs.shape), dtype=w0.qs.dtype, device="cuda")
    d = torch.empty((copies,) + tuple(w0.d.shape), dtype=w0.d.dtype, device="cuda")
    qs.copy_(w0.qs.unsqueeze(0).expand_as(qs))
    d.copy_(w0.d.unsqueeze(0).expand_as(d))
    return [api.Q8Weight(qs[i], d[i]) for i in range(copies)]


def hbm_read_probe(torch) -> dict:
    """The library's pure-read probe over a 2 GiB buffer (16x the L2): GB/s of
    one read, median of 10 timed launches after 3 untimed."""
    from block_quantized_decode_rmsnorm_gb300 import api

    nbytes = 2 << 30
    buf = torch.empty((nbytes,), dtype=torch.uint8, device="cuda")
    buf.fill_(1)
    sink = api.qg_measure_hbm_read(buf)
    for _ in range(3):
        api.qg_measure_hbm_read(buf, sink)
    torch.cuda.synchronize()
    ts = []
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        api.qg_measure_hbm_read(buf, sink)
        e1.record()
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) / 1e3)
    del buf, sink
    torch.cuda.empty_cache()
    return {"GB/s": nbytes / statistics.median(ts) / 1e9, "bytes": nbytes,
            "note": "qg_measure_hbm_read: every SM streams the buffer once with the GEMV kernels' 32-byte loads"}


def config_summary(torch, pk, probe_gbs: float, variants: bool = False) -> tuple:
    """One short entry per workload of the method besides the headline step:
    per-launch time (median of 20 timed graph replays over rotating weight copies
    >= 4x L2), the rate and its fraction of the measured peak (copy peak for HBM
    work, and of the read probe; the measured bf16 dense peak for tensor work).
    With `variants`, also every tile width and alternative kernel, returned
    separately."""
    from block_quantized_decode_rmsnorm_gb300 import api, synth

    cfg, var = {}, {}
    hbm = pk["hbm_gbs"]

    def hbm_entry(r, algo):
        gbs = algo / (r["us"] / 1e6) / 1e9
        e = {"us": round(r["us"], 3), "us_p90": round(r["us_p90"], 3), "GB/s": round(gbs, 1),
             "frac_copy_peak": round(gbs / hbm, 4), "frac_read_probe": round(gbs / probe_gbs, 4)}
        if "us_warm_l2" in r:
            e["us_warm_l2"] = round(r["us_warm_l2"], 3)
        return e

    def gemv(n, k, batch):
        qs, d = synth.q8_0_weight_planes(0, synth.S_W0, n, k)
        w0 = api.q8_weight_from_numpy(qs, d)
        copies = l2_copies(torch, w0.nbytes)
        ws = replicate_q8(torch, api, w0, copies)
        x = torch.from_numpy(synth.f32_normal(0, synth.S_X, (batch, k))).cuda()
        xq, xd = api.quantize_act_q8_0(x)
        y = torch.empty((batch, n), dtype=torch.float32, device="cuda")
        r = cold_and_warm(torch, lambda w: api.qgemv_q8_0(w, xq, xd, y=y), ws, w0.nbytes)
        algo = w0.nbytes + batch * (k + (k // 32) * 2) + batch * n * 4
        del ws
        return r, algo, copies

    # 1: Q8_0 GEMV 256x1024, and an empty kernel chain of the same launch shape
    # (the staging GEMV: rows spread over one wave, ceil(256 / SMs) rows and one
    # warp per row per CTA)
    r, algo, copies = gemv(256, 1024, 1)
    e = hbm_entry(r, algo)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rpc = -(-256 // sms)
    gf = capture(torch, lambda: api.qg_measure_launch_chain(copies, -(-256 // rpc), 32 * min(rpc, 8)))
    e["launch_floor_us"] = round(replay_trials(torch, gf, copies)["median"] * 1e6, 3)
    del gf
    cfg["1_gemv_256x1024"] = e
    # 4: output head 262144x1024, batch 1, 2, 4, 8
    for b in (1, 2, 4, 8):
        r, algo, _ = gemv(262144, 1024, b)
        cfg[f"4_head_262144x1024_b{b}"] = hbm_entry(r, algo)

    # next step 4: the headline step with the activation rotated in the fused
    # gate|up kernel (qg_decode_ffn_q8_0_rotated), 24 layers, one graph
    layers, x0 = make_layers(torch, 24)
    buf = api.FFNBuffers.allocate(HIDDEN, FFN, "cuda")
    xr = torch.from_numpy(x0).cuda()
    gr = capture(torch, lambda: [api.qg_decode_ffn_q8_0_rotated(xr, xr, ly, buf, EPS) for ly in layers])
    for _ in range(5):
        gr.replay()
    t_r = time_graph(torch, gr, 100)  # back-to-back replays, as the headline step
    del gr, layers
    gbs = 24 * LAYER_BYTES / t_r / 1e9
    cfg["next4_rotated_decode_step_24_layers"] = {"us": round(t_r * 1e6, 2), "GB/s": round(gbs, 1),
                                                  "frac_copy_peak": round(gbs / hbm, 4),
                                                  "timing": "100 back-to-back replays of the 24-layer graph"}

    # 3: bf16 gate|up 18432x2560, RMSNorm in front, SiLU*u behind
    bc = synth.bf16_case(0)
    w0 = api.bf16_from_bits(bc["w"])
    copies = l2_copies(torch, w0.numel() * 2)
    ws = [w0] + [w0.clone() for _ in range(copies - 1)]
    xb, gb = api.bf16_from_bits(bc["x"]), api.bf16_from_bits(bc["gamma"])
    yb = torch.empty((w0.shape[0] // 2,), dtype=torch.float32, device="cuda")
    r = cold_and_warm(torch, lambda w: api.qgemv_bf16(w, xb, gb, EPS, epilogue="silu_mul", y=yb), ws,
                      w0.numel() * 2)
    cfg["3_bf16_18432x2560"] = hbm_entry(r, w0.numel() * 2 + 2 * 2 * w0.shape[1] + yb.numel() * 4)

    # next step 3: the same projection for a 512-row prompt on tcgen05 (row norms + projection)
    xp = api.bf16_from_bits(synth.bf16_normal_bits(0, synth.S_X + 7, (512, w0.shape[1])))
    xh = torch.empty_like(xp)
    yp16 = torch.empty((512, w0.shape[0] // 2), dtype=torch.float32, device="cuda")
    flops = 2 * 512 * w0.shape[0] * w0.shape[1]
    bf16_fns = [("next3_prefill_bf16_512x18432x2560",
                 lambda w: api.qgemm_bf16_prefill(w, xp, gb, EPS, epilogue="silu_mul", y=yp16, xhat=xh))]
    if variants:
        bf16_fns.append(("prefill_bf16_512x18432x2560_gemm_only",
                         lambda w: api.qgemm_bf16_prefill(w, xh, None, EPS, epilogue="silu_mul", y=yp16)))
    for i, (name, fn) in enumerate(bf16_fns):
        r = cold_and_warm(torch, fn, ws, w0.numel() * 2)
        tf = flops / (r["us"] / 1e6) / 1e12
        (cfg if i == 0 else var)[name] = {"us": round(r["us"], 3), "TFLOP/s": round(tf, 1),
                                          "frac_bf16_dense_peak": round(tf / pk["bf16_tflops"], 4)}
    del ws, xp, xh, yp16

    # 5: prompt contraction 512x7168x1024 (wide tcgen05 tiles); int8 mma.sync rate as context
    api.qg_measure_mma_s8(100)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    mops = api.qg_measure_mma_s8(20000)
    e1.record()
    torch.cuda.synchronize()
    mma_tops = mops / (e0.elapsed_time(e1) / 1e3) / 1e12
    pc = synth.prefill_case(0)
    wp = api.q8_weight_from_numpy(pc["w_qs"], pc["w_d"])
    copies = l2_copies(torch, wp.nbytes)
    wps = replicate_q8(torch, api, wp, copies)
    xdev = torch.from_numpy(pc["x"]).cuda()
    yp = torch.empty((512, 7168), dtype=torch.float32, device="cuda")
    ops = 2 * 512 * 7168 * 1024
    wps2 = [api.qg_q8_0_pack_f16(w) for w in wps]
    x2 = api.quantize_act_q8_0_f16(xdev)
    w2bytes = wps2[0].codes.numel() * 2 + wps2[0].scales_t.numel() * 4
    runs = [("5_prefill_512x7168x1024", lambda w: api.qgemm_q8_0_prefill_tc2(w, x2, y=yp), wps2, w2bytes, cfg)]
    if variants:
        xq, xd = api.quantize_act_q8_0(xdev)
        xt = api.quantize_act_q8_0_tiles(xdev)
        runs.append(("prefill_wide_with_act_quant",
                     lambda w: api.qgemm_q8_0_prefill_tc2(w, api.quantize_act_q8_0_f16(xdev, out=x2), y=yp), wps2,
                     w2bytes, var))
        for bn in (128, 192):
            runs.append((f"prefill_wide_bn{bn}", lambda w, bn=bn: api.qgemm_q8_0_prefill_tc2(w, x2, y=yp, tile_n=bn),
                         wps2, w2bytes, var))
        runs.append(("prefill_tile_records", lambda w: api.qgemm_q8_0_prefill_tc(w, xt, y=yp), wps, wp.nbytes, var))
        for bn in (64, 96, 128):
            runs.append((f"prefill_tile_records_bn{bn}",
                         lambda w, bn=bn: api.qgemm_q8_0_prefill_tc(w, xt, y=yp, tile_n=bn), wps, wp.nbytes, var))
        runs.append(("prefill_mma_sync", lambda w: api.qgemm_q8_0_prefill(w, xq, xd, y=yp), wps, wp.nbytes, var))
    for name, fn, ws_, nb_, dst in runs:
        r = cold_and_warm(torch, fn, ws_, nb_)
        tops = ops / (r["us"] / 1e6) / 1e12
        dst[name] = {"us": round(r["us"], 3), "TOPS": round(tops, 1),
                     "frac_f16_dense_peak": round(tops / pk["bf16_tflops"], 4),
                     "x_mma_s8_rate": round(tops / mma_tops, 3)}
    cfg["5_prefill_512x7168x1024"]["mma_s8_rate_tops"] = round(mma_tops, 1)
    del wps, wps2
    torch.cuda.empty_cache()
    return cfg, var


def ncu_traffic(kernel_key: str):
    """DRAM bytes per launch of a kernel from the committed ncu summary (for
    "layer_pair", the decode layer's two kernels summed), or None when a kernel
    source changed since the capture or a record is missing."""
    f = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(f):
        return None
    recs = json.load(open(f))
    if kernel_key == "layer_pair":
        parts = [ncu_traffic(k) for k in ("ffn_up_kernel", "gemv_prefetch_kernel")]
        return None if None in parts else sum(parts)
    rec = recs.get(kernel_key)
    if not rec:
        return None
    if rec.get("source_sha256") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("qg_ffn.cu", "qg_stack.cu", "qg_norm.cuh", "qg_common.cuh"):
        with open(os.path.join(ROOT, "block_quantized_decode_rmsnorm_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _oracle_layers(job) -> tuple:
    """One host thread: oracle FFN layers of the step until `seconds` pass.
    Returns (layers done, seconds)."""
    seconds, n_layers = job
    import oracle
    from block_quantized_decode_rmsnorm_gb300 import synth

    oracle.build()
    cases = [synth.ffn_case(0, HIDDEN, FFN, layer=l) for l in range(min(n_layers, 4))]
    x = cases[0]["x"].copy()
    done, t0 = 0, time.perf_counter()
    while True:
        c = cases[done % len(cases)]
        r = oracle.decode_ffn(x, c["gamma"], EPS, c["gu_qs"], c["gu_d"], c["dn_qs"], c["dn_d"])
        x = r["out"]
        done += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return done, el


def cpu_baseline(seconds: float, n_layers: int, all_cores: bool = True) -> dict:
    """The oracle, as it stands, on this host: FFN layers of the step until the
    time budget is spent, on one host thread; and the same loop in one process
    per host core (spawned, so no GPU state is inherited), summed."""
    done, el = _oracle_layers((seconds, n_layers))
    out = {"value": done * LAYER_BYTES / el / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle", "cpu_model": cpu_model(),
           "sample": f"{done} FFN layers (hidden {HIDDEN}, ffn {FFN}) of the {n_layers}-layer step in {el:.1f} s, "
                     "plain C oracle, one host thread"}
    if all_cores:
        import multiprocessing as mp

        n = os.cpu_count() or 1
        with mp.get_context("spawn").Pool(n) as pool:
            res = pool.map(_oracle_layers, [(seconds, n_layers)] * n)
        total, span = sum(r[0] for r in res), max(r[1] for r in res)
        out["all_cores"] = {"value": total * LAYER_BYTES / span / 1e9, "unit": "GB/s", "cores": n,
                            "sample": f"{total} FFN layers in {span:.1f} s, the same oracle loop in {n} processes "
                                      "(one per host core), layers summed"}
    return out


def run_ours(args):
    import torch

    from block_quantized_decode_rmsnorm_gb300 import api, build

    dist = Dist(torch)
    dev = dist.local if dist.world > 1 else 0
    torch.cuda.set_device(dev)
    build()
    pk = peaks()
    L = args.layers
    layers, x0_np = make_layers(torch, L)
    buf = api.FFNBuffers.allocate(HIDDEN, FFN, "cuda")
    x = torch.from_numpy(x0_np).cuda()

    path = args.path
    if path == "stack":
        launches_per_step = -(-L // api._lib.load().qg_decode_stack_max_layers())
    else:
        launches_per_step = {"one": 1, "two": 2, "four": 4}[path] * L + (1 if path == "one" else 0)  # + the finish
    stack = api.LayerStack(HIDDEN, FFN, "cuda") if path == "one" else None
    dstack = api.DecodeStack(layers) if path == "stack" else None
    x_out = x
    if dstack is not None:
        x_out = torch.empty_like(x)  # each replay reads x and writes x_out
    if stack is not None:
        for layer in layers:  # down weights in the column-block layout, packed once at load time
            api.prepare_one_launch(layer)
        stack.load(x)
        torch.cuda.synchronize()
        x, x_out = stack.r[0], stack.out  # each replay reads r[0] and writes out

    def step():
        if dstack is not None:
            dstack.run(x, x_out, EPS)
            return
        if stack is not None:
            stack.run(layers, buf, EPS)
            return
        for layer in layers:
            if path == "two":
                api.qg_decode_ffn_q8_0(x, layer, buf, EPS)
            else:
                api.decode_ffn_q8_0(x, layer, buf, EPS)

    g = capture(torch, step)
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(torch, dev)
    procs_before = other_processes(gpu_processes())
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    e0.record()
    for _ in range(args.steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    procs_after = other_processes(gpu_processes())
    dist.barrier()
    elapsed = dist.max(e0.elapsed_time(e1) / 1e3)
    step_bytes = L * LAYER_BYTES
    value = job_rate(dist.world, args.steps, step_bytes, elapsed)

    # dominant kernel, timed alone (L back-to-back launches in a graph, events on the launching stream)
    if path == "stack":
        # the persistent kernel is the whole step: time it over back-to-back replays
        t_k = time_graph(torch, g, max(5, args.steps // 4)) / launches_per_step
        kbytes = STACK_KERNEL_BYTES(min(L, api._lib.load().qg_decode_stack_max_layers()))
        kname, kkey = ("decode_stack_kernel (every layer in one cooperative launch: RMSNorm + Q8_0 + gate|up + SiLU*u "
                       "+ Q8_0 + down + residual, hand-offs through value+epoch words)"), "decode_stack_kernel"
    elif path == "one":
        # the layer kernel is the step's only kernel but the one-block finish
        t_k = time_graph(torch, g, max(5, args.steps // 4)) / L
        kbytes, kname, kkey = LAYER_KERNEL_BYTES, ("ffn_up_kernel<1,true> (one-launch layer: RMSNorm + Q8_0 + "
                                                   "gate|up + SiLU*u + Q8_0 + split-K down + residual)"), "layer_kernel"
    else:
        # A layer's launches overlap under programmatic dependent launch (each one
        # stages its weights while its predecessor computes), so no launch has a
        # duration of its own inside the step.  The unit is the layer (the
        # algorithmic bytes of both projections), its time the timed region's
        # step time over the layers, both kernels' DRAM bytes its traffic.
        t_k = elapsed / args.steps / L
        kbytes = LAYER_BYTES
        if path == "two":
            kname, kkey = ("decode layer: ffn_up_kernel<1> (RMSNorm + Q8_0 + gate|up 7168x1024 + SiLU*u + Q8_0), "
                           "then gemv_prefetch_kernel<4> (down 1024x3584 + residual)"), "layer_pair"
        else:
            kname, kkey = "decode layer, four launches (rmsnorm_quantize, gate|up GEMV, quantize, down GEMV)", None
        if path == "two":
            # context: the gate|up kernel alone, L back-to-back launches in a graph
            h1, hq1, hd1 = buf.h[0], buf.hq[0], buf.hd[0]
            gu_graph = capture(torch, lambda: [api.qg_ffn_up_q8_0(x, l.gamma, l.gate_up, EPS, h=h1, hq=hq1, hd=hd1)
                                               for l in layers])
            t_alone = time_graph(torch, gu_graph, max(5, args.steps // 4)) / L
            del gu_graph
            kernel_alone = {"kernel": "ffn_up_kernel<1>", "us": t_alone * 1e6,
                            "GB/s": GU_KERNEL_BYTES / t_alone / 1e9,
                            "frac": GU_KERNEL_BYTES / t_alone / 1e9 / pk["hbm_gbs"],
                            "algorithmic_bytes_per_launch": GU_KERNEL_BYTES, "traffic": ncu_traffic("ffn_up_kernel"),
                            "note": "back to back, each launch waits on its own weight staging: the kernel releases its "
                                    "dependent after its wait, which is what the decode layer wants"}
    # the floor's measured inputs: an empty kernel chain of the step's launch count
    # and launch shape (one CTA per SM), and the step's bytes at the measured peaks
    n_chain = max(2, launches_per_step)
    g_floor = capture(torch, lambda: api.qg_measure_launch_chain(n_chain, min(152, torch.cuda.get_device_properties(
        dev).multi_processor_count), 256))
    edge_us = replay_trials(torch, g_floor, n_chain)["median"] * 1e6
    del g_floor
    floor = {"empty_launch_us": round(edge_us, 3), "launches_per_step": launches_per_step,
             "hbm_us_per_step_copy_peak": round(L * LAYER_BYTES / pk["hbm_gbs"] / 1e3, 2)}
    achieved = kbytes / t_k / 1e9
    per_layer = path in ("two", "four")
    roofline = {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "peak_source": pk["source"],
                ("algorithmic_bytes_per_layer" if per_layer else "algorithmic_bytes_per_launch"): kbytes,
                ("us_per_layer" if per_layer else "launch_us"): t_k * 1e6,
                "traffic": ncu_traffic(kkey) if kkey else None}
    if path == "two":
        roofline["kernel_alone"] = kernel_alone

    # end to end through host buffers, every step: x taken from pinned host memory,
    # the step, the result left in pinned host memory, and the host waiting for it;
    # a step is one graph launch.  On the two-launch path the first layer reads x
    # from the host buffer and the last layer writes its output into the host
    # buffer directly (qg_decode_ffn_q8_0_out); the other paths copy x in and the
    # result out with copies captured in the graph.
    x_host = torch.from_numpy(x0_np.copy()).pin_memory()
    out_host = torch.empty_like(x_host).pin_memory()
    direct = path in ("two", "stack") and stack is None

    def e2e_step():
        if dstack is not None:
            dstack.run(x_host, out_host, EPS)
            return
        if direct:
            src = x_host
            for i, layer in enumerate(layers):
                dst = out_host if i == len(layers) - 1 else x
                api.qg_decode_ffn_q8_0_out(src, dst, layer, buf, EPS)
                src = dst
            return
        x.copy_(x_host, non_blocking=True)
        step()
        out_host.copy_(x_out, non_blocking=True)

    g_e2e = capture(torch, e2e_step)
    for _ in range(max(3, args.warmup)):
        g_e2e.replay()
        torch.cuda.current_stream().synchronize()
    dist.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        g_e2e.replay()
        torch.cuda.current_stream().synchronize()
    e2e_el = dist.max(time.perf_counter() - t0)
    e2e = {"value": job_rate(dist.world, args.steps, step_bytes, e2e_el), "unit": "GB/s",
           "h2d_bytes_per_step": HIDDEN * 4, "d2h_bytes_per_step": HIDDEN * 4,
           "ms_per_step": e2e_el / args.steps * 1e3,
           "transfer": ("first layer reads x from pinned host memory, last layer writes its result into pinned "
                        "host memory (kernels over the host link, no copy operations)") if direct else
                       "cudaMemcpyAsync host->device and device->host, captured in the step's graph"}

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": workload_name(L), "layers": L, "batch": 1, "bytes_per_step": step_bytes,
                   "frac_of_hbm_peak": value / dist.world / pk["hbm_gbs"],
                   "l2": f"inputs larger than L2: {step_bytes / 1e6:.0f} MB of weights per step, "
                         f"L2 {torch.cuda.get_device_properties(dev).L2_cache_size / 1e6:.0f} MB",
                   "graph": f"one CUDA graph per step, {launches_per_step} launches, programmatic dependent launch",
                   "path": {"stack": "every layer in one persistent cooperative launch (qg_decode_stack_q8_0)",
                            "one": "one launch per layer (qg_decode_layer_q8_0: split-K down, cluster partials summed by the next layer) + finish",
                            "two": "two launches per layer (qg_decode_ffn_q8_0)",
                            "four": "four launches per layer (decode_ffn_q8_0)"}[path],
                   "parallelism": f"replicas x{dist.world} (independent decode streams, no collective)"},
        "roofline": roofline, "e2e": e2e, "gpu_launches": launches_per_step * args.steps, "clocks": clocks,
        "other_gpu_processes": {"before": procs_before, "after": procs_after}, "step_floor_inputs": floor,
    }
    if not args.quick:
        probe = hbm_read_probe(torch)
        cfgs, var = config_summary(torch, pk, probe["GB/s"], args.variants)
        line["hbm_read_probe"] = {"GB/s": round(probe["GB/s"], 1), "frac_copy_peak": round(probe["GB/s"] / pk["hbm_gbs"], 4)}
        line["roofline"]["frac_read_probe"] = line["roofline"]["achieved"] / probe["GB/s"]
        floor["hbm_us_per_step_read_probe"] = round(L * LAYER_BYTES / probe["GB/s"] / 1e3, 2)
        line["configs"] = cfgs
        if var:
            line["variants"] = var
    if dist.rank == 0 and dist.world == 1:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds, L)
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


def run_workload(args):
    """One workload's kernel alone, launched eagerly warmup + steps times (for
    profiling one kernel, e.g. under ncu); prints its mean launch time."""
    import torch

    from block_quantized_decode_rmsnorm_gb300 import api, build, synth

    torch.cuda.set_device(0)
    build()
    w = args.workload
    if w == "prefill":
        pc = synth.prefill_case(0)
        wt = api.q8_weight_from_numpy(pc["w_qs"], pc["w_d"])
        xt = api.quantize_act_q8_0_tiles(torch.from_numpy(pc["x"]).cuda())
        y = torch.empty((pc["x"].shape[0], pc["w_qs"].shape[0]), dtype=torch.float32, device="cuda")
        fn = lambda: api.qgemm_q8_0_prefill_tc(wt, xt, y=y)
        name = "prompt contraction 512x7168x1024, tcgen05"
    elif w == "prefill_wide":
        pc = synth.prefill_case(0)
        w2 = api.qg_q8_0_pack_f16(api.q8_weight_from_numpy(pc["w_qs"], pc["w_d"]))
        x2 = api.quantize_act_q8_0_f16(torch.from_numpy(pc["x"]).cuda())
        y = torch.empty((pc["x"].shape[0], pc["w_qs"].shape[0]), dtype=torch.float32, device="cuda")
        fn = lambda: api.qgemm_q8_0_prefill_tc2(w2, x2, y=y)
        name = "prompt contraction 512x7168x1024, tcgen05 wide tiles"
    elif w.startswith("head"):
        b = int(w[4:])
        qs, d = synth.q8_0_weight_planes(0, synth.S_W0, 262144, 1024)
        wt = api.q8_weight_from_numpy(qs, d)
        xq, xd = api.quantize_act_q8_0(torch.from_numpy(synth.f32_normal(0, synth.S_X, (b, 1024))).cuda())
        y = torch.empty((b, 262144), dtype=torch.float32, device="cuda")
        fn = lambda: api.qgemv_q8_0(wt, xq, xd, y=y)
        name = f"output head 262144x1024, batch {b}"
    elif w == "prefill_bf16":
        bc = synth.bf16_case(0)
        wb, gb = api.bf16_from_bits(bc["w"]), api.bf16_from_bits(bc["gamma"])
        xb = api.bf16_from_bits(synth.bf16_normal_bits(0, synth.S_X + 7, (512, bc["w"].shape[1])))
        xh = torch.empty_like(xb)
        y = torch.empty((512, bc["w"].shape[0] // 2), dtype=torch.float32, device="cuda")
        fn = lambda: api.qgemm_bf16_prefill(wb, xb, gb, EPS, epilogue="silu_mul", y=y, xhat=xh)
        name = "bf16 gate|up 18432x2560 + RMSNorm + SiLU*u, 512-row prompt, tcgen05"
    else:  # bf16
        bc = synth.bf16_case(0)
        wb, xb, gb = api.bf16_from_bits(bc["w"]), api.bf16_from_bits(bc["x"]), api.bf16_from_bits(bc["gamma"])
        y = torch.empty((bc["w"].shape[0] // 2,), dtype=torch.float32, device="cuda")
        fn = lambda: api.qgemv_bf16(wb, xb, gb, EPS, epilogue="silu_mul", y=y)
        name = "bf16 gate|up 18432x2560 + RMSNorm + SiLU*u"
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    print(json.dumps({"workload": name, "launches": args.steps,
                      "us_per_launch": e0.elapsed_time(e1) * 1e3 / args.steps,
                      "note": "eager back-to-back launches of one kernel, warm L2; for profiling, not the bench line"}),
          flush=True)


def run_reference(args):
    """The CPU oracle as the reference arm: same workload, metric and unit."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import oracle
    from block_quantized_decode_rmsnorm_gb300 import synth

    oracle.build()
    L = args.layers
    cases = [synth.ffn_case(0, HIDDEN, FFN, layer=l) for l in range(min(L, 4))]
    x = cases[0]["x"].copy()
    # one layer's time, then layers per step sized so the whole run ends in ~2 minutes
    t0 = time.perf_counter()
    oracle.decode_ffn(x, cases[0]["gamma"], EPS, cases[0]["gu_qs"], cases[0]["gu_d"], cases[0]["dn_qs"],
                      cases[0]["dn_d"])
    t_layer = max(time.perf_counter() - t0, 1e-4)
    per_step = max(1, min(L, int(120.0 / ((args.steps + args.warmup) * t_layer))))

    def step():
        nonlocal x
        for l in range(per_step):
            c = cases[l % len(cases)]
            x = oracle.decode_ffn(x, c["gamma"], EPS, c["gu_qs"], c["gu_d"], c["dn_qs"], c["dn_d"])["out"]

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = args.steps * per_step * LAYER_BYTES / el / 1e9
    sample = (f"{per_step} of the {L} FFN layers per step (hidden {HIDDEN}, ffn {FFN}), plain C oracle, "
              "one host thread")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(L), "layers": L, "batch": 1, "layers_per_step_sampled": per_step},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample,
                         "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=24)
    ap.add_argument("--quick", action="store_true", help="skip the other workloads' kernel rates")
    ap.add_argument("--variants", action="store_true",
                    help="also time every tile width and alternative kernel of the other workloads")
    ap.add_argument("--path", choices=["stack", "one", "two", "four"], default="two",
                    help="stack: every layer in one persistent launch; otherwise launches per decode layer: one "
                         "(split-K down inside the layer kernel), two, four")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--workload", choices=["prefill", "prefill_wide", "prefill_bf16", "head1", "head2", "head4", "head8", "bf16"],
                    help="time one workload's kernel alone (for profiling) instead of the bench step")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload:
        run_workload(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
