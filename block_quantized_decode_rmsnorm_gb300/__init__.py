"""GB300-native Q8_0 / bf16 decode matrix-vector path.

The compute lives in ``libqgemv.so`` (hand-written CUDA for sm_103a, C ABI in
``include/qgemv.h``); ``api`` is its torch-tensor binding and ``synth`` the
seeded input generator.  Importing the package loads neither torch nor the
library; the binding's names resolve on first use.
"""

_API_NAMES = {
    "qg_q8_0_pack", "quantize_act_q8_0", "rmsnorm_quantize", "qgemv_q8_0", "qgemv_bf16",
    "qgemm_q8_0_prefill", "qg_debug_block_dots_q8_0", "decode_ffn_q8_0", "qg_ffn_up_q8_0",
    "qg_decode_ffn_q8_0", "qg_decode_layer_q8_0", "qg_decode_layer_partials", "qg_decode_layer_finish", "LayerStack", "qg_decode_layers_q8_0_noalloc", "qg_q8_0_column_blocks", "prepare_one_launch", "quantize_act_q8_0_tiles", "qgemm_q8_0_prefill_tc", "ActTiles", "Q8Weight", "FFNLayer",
    "FFNBuffers", "q8_weight_from_numpy", "bf16_from_bits", "qgemm_bf16_prefill", "qg_measure_mma_s8",
    "qg_q8_0_pack_f16", "quantize_act_q8_0_f16", "qg_decode_ffn_q8_0_out", "qgemm_q8_0_prefill_tc2", "F16Codes",
}


def __getattr__(name):
    if name in _API_NAMES:
        from . import api

        return getattr(api, name)
    raise AttributeError(name)


def build(force: bool = False) -> str:
    """Compile libqgemv.so in-tree (nvcc, sm_103a)."""
    from .builder import build as _build

    return _build(force=force)
