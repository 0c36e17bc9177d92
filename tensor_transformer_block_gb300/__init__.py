"""GB300-native Megatron tensor-parallel transformer block.

The compute lives in ``libtpblock.so`` (hand-written sm_103a CUDA: tcgen05/TMEM
tensor-core GEMMs fed by TMA, fused GeLU / SwiGLU / residual epilogues, on-device shard reduction,
fused attention, LayerNorm).  This package is its ctypes binding (same function names as
the C header ``include/tpblock.h``), the in-tree build, a small convenience layer
that allocates outputs with torch (``block``), and the seeded synthetic inputs
(``inputs``).
"""
from ._binding import (  # noqa: F401
    HEADER_PATH, LIB_PATH, QKV_PLANES, STATUS, TP_BF16, TP_F32, TPError, header_functions, load_library,
    tp_attn_bwd, tp_attn_fwd, tp_attn_mlp_bwd, tp_attn_mlp_fwd, tp_attn_mlp_save_bytes, tp_attn_mlp_workspace_bytes,
    tp_attn_workspace_bytes, tp_debug_timeout_probe, tp_device_check,
    tp_gmlp_bwd, tp_gmlp_fwd, tp_gmlp_workspace_bytes, tp_gqa_bwd, tp_gqa_fwd, tp_gqa_workspace_bytes, tp_layer_bwd, tp_layer_fwd, tp_layer_save_bytes,
    tp_layer_workspace_bytes, tp_layernorm_bwd, tp_layernorm_fwd, tp_layernorm_workspace_bytes,
    tp_mlp_bwd, tp_mlp_fwd, tp_mlp_fwd_noalloc,
    tp_mlp_workspace_bytes, tp_set_gemm_tiling, tp_set_launch_overlap, tp_sp_layer_bwd, tp_sp_layer_fwd, tp_status_string,
    tp_sync_status, tp_timing_enable,
    tp_timing_kinds, tp_timing_name, tp_timing_read, tp_version, timing_report,
)

__version__ = "0.1.0"
