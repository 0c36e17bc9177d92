"""ctypes binding of libtpblock: one Python function per C entry point, same names.

Marshalling only: tensors become device pointers, sizes become int64, the stream
defaults to torch's current stream.  Before a call the binding checks that every
tensor is a contiguous CUDA tensor of the right dtype and at least the number of
elements the C call will touch (the C side only sees pointers and sizes).  A
non-zero status raises :class:`TPError`.  There is no fallback: if the shared
library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
# TPBLOCK_LIB selects another build of the library (the checked libtpblock_debug.so)
LIB_PATH = os.environ.get("TPBLOCK_LIB") or os.path.join(HERE, "libtpblock.so")
HEADER_PATH = os.path.join(os.path.dirname(HERE), "include", "tpblock.h")

TP_F32, TP_BF16 = 0, 1
QKV_PLANES = 3  # Q, K, V (fp16 values in 16-bit storage) per (token, head)
STATUS = {0: "TP_OK", 1: "TP_ERR_NULL", 2: "TP_ERR_SHAPE", 3: "TP_ERR_DTYPE", 4: "TP_ERR_WORKSPACE",
          5: "TP_ERR_CUDA", 6: "TP_ERR_TIMEOUT", 7: "TP_ERR_ALIGN", 8: "TP_ERR_DEVICE", 9: "TP_ERR_BOUNDS"}
_TORCH_DT = {TP_F32: torch.float32, TP_BF16: torch.bfloat16}

_lib = None

i64, i32, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
_SIGS = {
    "tp_version": ([], i32),
    "tp_status_string": ([i32], ctypes.c_char_p),
    "tp_device_check": ([], i32),
    "tp_sync_status": ([vp], i32),
    "tp_debug_timeout_probe": ([i64, vp], i32),
    "tp_mlp_workspace_bytes": ([i32, i64, i64, i64, i32], sz),
    "tp_mlp_fwd": ([i32, i64, i64, i64, i32, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
    "tp_mlp_bwd": ([i32, i64, i64, i64, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
    "tp_attn_workspace_bytes": ([i32, i64, i64, i64, i32, i32, i32], sz),
    "tp_attn_fwd": ([i32, i64, i64, i64, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
    "tp_attn_bwd": ([i32, i64, i64, i64, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz,
                     vp], i32),
    "tp_mlp_fwd_noalloc": ([i32, i64, i64, i64, i32, vp, vp, vp, vp, vp], i32),
    "tp_gmlp_workspace_bytes": ([i32, i64, i64, i64, i32], sz),
    "tp_gmlp_fwd": ([i32, i64, i64, i64, i32, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
    "tp_gmlp_bwd": ([i32, i64, i64, i64, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
    "tp_gqa_workspace_bytes": ([i32, i64, i64, i64, i32, i32, i32, i32], sz),
    "tp_gqa_fwd": ([i32, i64, i64, i64, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
    "tp_gqa_bwd": ([i32, i64, i64, i64, i32, i32, i32, i32, i32] + [vp] * 11 + [sz, vp], i32),
    "tp_layernorm_workspace_bytes": ([i32, i64, i64], sz),
    "tp_layernorm_fwd": ([i32, i64, i64, ctypes.c_float, vp, vp, vp, vp, vp, vp, vp], i32),
    "tp_layernorm_bwd": ([i32, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
    "tp_layer_save_bytes": ([i32, i64, i64, i64, i32, i32, i64, i32], sz),
    "tp_layer_workspace_bytes": ([i32, i64, i64, i64, i32, i32, i64, i32], sz),
    "tp_layer_fwd": ([i32, i64, i64, i64, i32, i32, i64, i32, i32, ctypes.c_float] + [vp] * 10 + [sz, vp, vp], i32),
    "tp_layer_bwd": ([i32, i64, i64, i64, i32, i32, i64, i32, i32] + [vp] * 8 + [sz] + [vp] * 10 + [vp, sz, vp],
                     i32),
    "tp_sp_layer_fwd": ([i32, i64, i64, i64, i32, i32, i64, i32, i32, ctypes.c_float] + [vp] * 10 + [sz, vp, vp], i32),
    "tp_sp_layer_bwd": ([i32, i64, i64, i64, i32, i32, i64, i32, i32] + [vp] * 8 + [sz] + [vp] * 10 + [vp, sz, vp],
                        i32),
    "tp_attn_mlp_save_bytes": ([i32, i64, i64, i64, i32, i32, i64, i32], sz),
    "tp_attn_mlp_workspace_bytes": ([i32, i64, i64, i64, i32, i32, i64, i32], sz),
    "tp_attn_mlp_fwd": ([i32, i64, i64, i64, i32, i32, i64, i32, i32] + [vp] * 6 + [sz, vp, vp], i32),
    "tp_attn_mlp_bwd": ([i32, i64, i64, i64, i32, i32, i64, i32, i32] + [vp] * 6 + [sz] + [vp] * 6 + [vp, sz, vp],
                        i32),
    "tp_set_gemm_tiling": ([i32], i32),
    "tp_set_launch_overlap": ([i32], i32),
    "tp_timing_enable": ([i32], i32),
    "tp_timing_kinds": ([], i32),
    "tp_timing_name": ([i32], ctypes.c_char_p),
    "tp_timing_read": ([i32, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double)], i32),
}


class TPError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__(f"{call} failed: {STATUS.get(status, status)} ({status_string(status)})")


def load_library(path: str | None = None) -> ctypes.CDLL:
    """dlopens libtpblock.so (built by ``build()``) and declares every signature."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"{path} is not built: run tensor_transformer_block_gb300.build.build() "
                          "(the block has no non-CUDA implementation)")
    lib = ctypes.CDLL(path)
    for name, (args, res) in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def header_functions() -> list[str]:
    """Names of the functions include/tpblock.h declares."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"\b(tp_[a-z0-9_]+)\s*\(", text)


def status_string(status: int) -> str:
    try:
        return load_library().tp_status_string(status).decode()
    except ImportError:
        return STATUS.get(status, "unknown status")


def _check(status: int, call: str) -> int:
    if status != 0:
        raise TPError(status, call)
    return status


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _p(t, name: str, dtype, numel: int | None, required: bool = True):
    """Device pointer of ``t`` after checking it (None -> NULL if optional)."""
    if t is None:
        if required:
            raise ValueError(f"{name} is required")
        return None
    if isinstance(t, int):  # raw device address supplied by the caller
        return t
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} has {t.numel()} elements, needs {numel}")
    return t.data_ptr()


def _ws(ws, need: int):
    if ws is None:
        return None, 0
    if isinstance(ws, int):
        return ws, need
    if not ws.is_cuda or not ws.is_contiguous():
        raise ValueError("ws must be a contiguous CUDA tensor")
    return ws.data_ptr(), ws.numel() * ws.element_size()


# ---------------------------------------------------------------- plain calls
def tp_version() -> int:
    return load_library().tp_version()


def tp_status_string(status: int) -> str:
    return load_library().tp_status_string(status).decode()


def tp_device_check() -> int:
    return load_library().tp_device_check()


def tp_sync_status(stream=None) -> int:
    return load_library().tp_sync_status(_stream(stream))


def tp_debug_timeout_probe(timeout_ns: int, stream=None) -> int:
    return _check(load_library().tp_debug_timeout_probe(timeout_ns, _stream(stream)), "tp_debug_timeout_probe")


# ---------------------------------------------------------------- MLP block
def tp_mlp_workspace_bytes(dtype: int, T: int, h: int, f: int, N: int) -> int:
    return load_library().tp_mlp_workspace_bytes(dtype, T, h, f, N)


def tp_mlp_fwd(dtype, T, h, f, N, X, W1s, W2s, Y_save, A_save, Z, ws=None, stream=None) -> int:
    dt = _TORCH_DT.get(dtype)
    act = T * f
    wptr, wbytes = _ws(ws, tp_mlp_workspace_bytes(dtype, T, h, f, N))
    return _check(load_library().tp_mlp_fwd(
        dtype, T, h, f, N, _p(X, "X", dt, T * h), _p(W1s, "W1s", dt, h * f), _p(W2s, "W2s", dt, f * h),
        _p(Y_save, "Y_save", dt, act, False), _p(A_save, "A_save", dt, act, False), _p(Z, "Z", dt, T * h),
        wptr, wbytes, _stream(stream)), "tp_mlp_fwd")


def tp_mlp_bwd(dtype, T, h, f, N, X, W1s, W2s, Y_save, A_save, dZ, dX, dW1s, dW2s, ws=None, stream=None) -> int:
    dt = _TORCH_DT.get(dtype)
    act = T * f
    wptr, wbytes = _ws(ws, tp_mlp_workspace_bytes(dtype, T, h, f, N))
    return _check(load_library().tp_mlp_bwd(
        dtype, T, h, f, N, _p(X, "X", dt, T * h), _p(W1s, "W1s", dt, h * f), _p(W2s, "W2s", dt, f * h),
        _p(Y_save, "Y_save", dt, act), _p(A_save, "A_save", dt, act), _p(dZ, "dZ", dt, T * h),
        _p(dX, "dX", dt, T * h), _p(dW1s, "dW1s", dt, h * f), _p(dW2s, "dW2s", dt, f * h),
        wptr, wbytes, _stream(stream)), "tp_mlp_bwd")


def tp_mlp_fwd_noalloc(dtype, T, h, f, N, X, W1s, W2s, Z, stream=None) -> int:
    """Z of the MLP block with the activation kept in the library's fixed device
    array (no allocation anywhere on the call's path)."""
    dt = _TORCH_DT.get(dtype)
    return _check(load_library().tp_mlp_fwd_noalloc(
        dtype, T, h, f, N, _p(X, "X", dt, T * h), _p(W1s, "W1s", dt, h * f), _p(W2s, "W2s", dt, f * h),
        _p(Z, "Z", dt, T * h), _stream(stream)), "tp_mlp_fwd_noalloc")


# ---------------------------------------------------------------- gated MLP block
def tp_gmlp_workspace_bytes(dtype: int, T: int, h: int, f: int, N: int) -> int:
    return load_library().tp_gmlp_workspace_bytes(dtype, T, h, f, N)


def tp_gmlp_fwd(dtype, T, h, f, N, X, Wgus, Wds, GU_save, A_save, Z, ws=None, stream=None) -> int:
    dt = _TORCH_DT.get(dtype)
    wptr, wbytes = _ws(ws, tp_gmlp_workspace_bytes(dtype, T, h, f, N))
    return _check(load_library().tp_gmlp_fwd(
        dtype, T, h, f, N, _p(X, "X", dt, T * h), _p(Wgus, "Wgus", dt, 2 * h * f), _p(Wds, "Wds", dt, f * h),
        _p(GU_save, "GU_save", dt, 2 * T * f, False), _p(A_save, "A_save", dt, T * f, False),
        _p(Z, "Z", dt, T * h), wptr, wbytes, _stream(stream)), "tp_gmlp_fwd")


def tp_gmlp_bwd(dtype, T, h, f, N, X, Wgus, Wds, GU_save, A_save, dZ, dX, dWgus, dWds, ws=None,
                stream=None) -> int:
    dt = _TORCH_DT.get(dtype)
    wptr, wbytes = _ws(ws, tp_gmlp_workspace_bytes(dtype, T, h, f, N))
    return _check(load_library().tp_gmlp_bwd(
        dtype, T, h, f, N, _p(X, "X", dt, T * h), _p(Wgus, "Wgus", dt, 2 * h * f), _p(Wds, "Wds", dt, f * h),
        _p(GU_save, "GU_save", dt, 2 * T * f), _p(A_save, "A_save", dt, T * f), _p(dZ, "dZ", dt, T * h),
        _p(dX, "dX", dt, T * h), _p(dWgus, "dWgus", dt, 2 * h * f), _p(dWds, "dWds", dt, f * h),
        wptr, wbytes, _stream(stream)), "tp_gmlp_bwd")


# ---------------------------------------------------------------- grouped-query attention
def tp_gqa_workspace_bytes(dtype: int, B: int, S: int, h: int, H: int, Hkv: int, d: int, N: int) -> int:
    return load_library().tp_gqa_workspace_bytes(dtype, B, S, h, H, Hkv, d, N)


def tp_gqa_fwd(dtype, B, S, h, H, Hkv, d, N, causal, X, Wqkv, Wo, QKV_save, O_save, LSE_save, Z, ws=None,
               stream=None) -> int:
    dt = _TORCH_DT.get(dtype)
    T = B * S
    wptr, wbytes = _ws(ws, tp_gqa_workspace_bytes(dtype, B, S, h, H, Hkv, d, N))
    return _check(load_library().tp_gqa_fwd(
        dtype, B, S, h, H, Hkv, d, N, 1 if causal else 0, _p(X, "X", dt, T * h),
        _p(Wqkv, "Wqkv", dt, h * (H + 2 * Hkv) * d), _p(Wo, "Wo", dt, H * d * h),
        _p(QKV_save, "QKV_save", dt, T * (H + 2 * Hkv) * d, False), _p(O_save, "O_save", dt, T * H * d, False),
        _p(LSE_save, "LSE_save", torch.float32, B * H * S, False), _p(Z, "Z", dt, T * h), wptr, wbytes,
        _stream(stream)), "tp_gqa_fwd")


def tp_gqa_bwd(dtype, B, S, h, H, Hkv, d, N, causal, X, Wqkv, Wo, QKV_save, O_save, LSE_save, dZ, dX, dWqkv, dWo,
               ws=None, stream=None) -> int:
    dt = _TORCH_DT.get(dtype)
    T = B * S
    wptr, wbytes = _ws(ws, tp_gqa_workspace_bytes(dtype, B, S, h, H, Hkv, d, N))
    return _check(load_library().tp_gqa_bwd(
        dtype, B, S, h, H, Hkv, d, N, 1 if causal else 0, _p(X, "X", dt, T * h),
        _p(Wqkv, "Wqkv", dt, h * (H + 2 * Hkv) * d), _p(Wo, "Wo", dt, H * d * h),
        _p(QKV_save, "QKV_save", dt, T * (H + 2 * Hkv) * d), _p(O_save, "O_save", dt, T * H * d),
        _p(LSE_save, "LSE_save", torch.float32, B * H * S), _p(dZ, "dZ", dt, T * h), _p(dX, "dX", dt, T * h),
        _p(dWqkv, "dWqkv", dt, h * (H + 2 * Hkv) * d), _p(dWo, "dWo", dt, H * d * h), wptr, wbytes,
        _stream(stream)), "tp_gqa_bwd")


# ---------------------------------------------------------------- LayerNorm, pre-norm layer
def tp_layernorm_workspace_bytes(dtype: int, T: int, h: int) -> int:
    return load_library().tp_layernorm_workspace_bytes(dtype, T, h)


def tp_layernorm_fwd(dtype, T, h, eps, X, gamma, beta, Y, mean, rstd, stream=None) -> int:
    dt = _TORCH_DT.get(dtype)
    return _check(load_library().tp_layernorm_fwd(
        dtype, T, h, eps, _p(X, "X", dt, T * h), _p(gamma, "gamma", dt, h), _p(beta, "beta", dt, h),
        _p(Y, "Y", dt, T * h), _p(mean, "mean", torch.float32, T), _p(rstd, "rstd", torch.float32, T),
        _stream(stream)), "tp_layernorm_fwd")


def tp_layernorm_bwd(dtype, T, h, X, gamma, mean, rstd, dY, dR, dX, dgamma, dbeta, ws=None, stream=None) -> int:
    dt = _TORCH_DT.get(dtype)
    wptr, wbytes = _ws(ws, tp_layernorm_workspace_bytes(dtype, T, h))
    return _check(load_library().tp_layernorm_bwd(
        dtype, T, h, _p(X, "X", dt, T * h), _p(gamma, "gamma", dt, h), _p(mean, "mean", torch.float32, T),
        _p(rstd, "rstd", torch.float32, T), _p(dY, "dY", dt, T * h), _p(dR, "dR", dt, T * h, False),
        _p(dX, "dX", dt, T * h), _p(dgamma, "dgamma", dt, h), _p(dbeta, "dbeta", dt, h), wptr, wbytes,
        _stream(stream)), "tp_layernorm_bwd")


def tp_layer_save_bytes(dtype, B, S, h, H, d, f, N) -> int:
    return load_library().tp_layer_save_bytes(dtype, B, S, h, H, d, f, N)


def tp_layer_workspace_bytes(dtype, B, S, h, H, d, f, N) -> int:
    return load_library().tp_layer_workspace_bytes(dtype, B, S, h, H, d, f, N)


def _layer_fwd(name, dtype, B, S, h, H, d, f, N, causal, eps, X, ln1_g, ln1_b, Wqkv, Wo, ln2_g, ln2_b, W1s, W2s,
               save, Z, stream):
    dt = _TORCH_DT.get(dtype)
    T = B * S
    sptr, sbytes = _ws(save, tp_layer_save_bytes(dtype, B, S, h, H, d, f, N))
    return _check(getattr(load_library(), name)(
        dtype, B, S, h, H, d, f, N, 1 if causal else 0, eps, _p(X, "X", dt, T * h), _p(ln1_g, "ln1_g", dt, h),
        _p(ln1_b, "ln1_b", dt, h), _p(Wqkv, "Wqkv", dt, 3 * h * H * d), _p(Wo, "Wo", dt, H * d * h),
        _p(ln2_g, "ln2_g", dt, h), _p(ln2_b, "ln2_b", dt, h), _p(W1s, "W1s", dt, h * f), _p(W2s, "W2s", dt, f * h),
        sptr, sbytes, _p(Z, "Z", dt, T * h), _stream(stream)), name)


def _layer_bwd(name, dtype, B, S, h, H, d, f, N, causal, X, ln1_g, Wqkv, Wo, ln2_g, W1s, W2s, save, dZ, dX, dln1_g,
               dln1_b, dWqkv, dWo, dln2_g, dln2_b, dW1s, dW2s, ws, stream):
    dt = _TORCH_DT.get(dtype)
    T = B * S
    sptr, sbytes = _ws(save, tp_layer_save_bytes(dtype, B, S, h, H, d, f, N))
    wptr, wbytes = _ws(ws, tp_layer_workspace_bytes(dtype, B, S, h, H, d, f, N))
    return _check(getattr(load_library(), name)(
        dtype, B, S, h, H, d, f, N, 1 if causal else 0, _p(X, "X", dt, T * h), _p(ln1_g, "ln1_g", dt, h),
        _p(Wqkv, "Wqkv", dt, 3 * h * H * d), _p(Wo, "Wo", dt, H * d * h), _p(ln2_g, "ln2_g", dt, h),
        _p(W1s, "W1s", dt, h * f), _p(W2s, "W2s", dt, f * h), sptr, sbytes, _p(dZ, "dZ", dt, T * h),
        _p(dX, "dX", dt, T * h), _p(dln1_g, "dln1_g", dt, h), _p(dln1_b, "dln1_b", dt, h),
        _p(dWqkv, "dWqkv", dt, 3 * h * H * d), _p(dWo, "dWo", dt, H * d * h), _p(dln2_g, "dln2_g", dt, h),
        _p(dln2_b, "dln2_b", dt, h), _p(dW1s, "dW1s", dt, h * f), _p(dW2s, "dW2s", dt, f * h), wptr, wbytes,
        _stream(stream)), name)


def tp_layer_fwd(dtype, B, S, h, H, d, f, N, causal, eps, X, ln1_g, ln1_b, Wqkv, Wo, ln2_g, ln2_b, W1s, W2s,
                 save, Z, stream=None) -> int:
    return _layer_fwd("tp_layer_fwd", dtype, B, S, h, H, d, f, N, causal, eps, X, ln1_g, ln1_b, Wqkv, Wo, ln2_g,
                      ln2_b, W1s, W2s, save, Z, stream)


def tp_layer_bwd(dtype, B, S, h, H, d, f, N, causal, X, ln1_g, Wqkv, Wo, ln2_g, W1s, W2s, save, dZ, dX, dln1_g,
                 dln1_b, dWqkv, dWo, dln2_g, dln2_b, dW1s, dW2s, ws=None, stream=None) -> int:
    return _layer_bwd("tp_layer_bwd", dtype, B, S, h, H, d, f, N, causal, X, ln1_g, Wqkv, Wo, ln2_g, W1s, W2s,
                      save, dZ, dX, dln1_g, dln1_b, dWqkv, dWo, dln2_g, dln2_b, dW1s, dW2s, ws, stream)


def tp_sp_layer_fwd(dtype, B, S, h, H, d, f, N, causal, eps, X, ln1_g, ln1_b, Wqkv, Wo, ln2_g, ln2_b, W1s, W2s,
                    save, Z, stream=None) -> int:
    """The layer with X and Z sequence-sharded ([N][B][S/N][h])."""
    return _layer_fwd("tp_sp_layer_fwd", dtype, B, S, h, H, d, f, N, causal, eps, X, ln1_g, ln1_b, Wqkv, Wo, ln2_g,
                      ln2_b, W1s, W2s, save, Z, stream)


def tp_sp_layer_bwd(dtype, B, S, h, H, d, f, N, causal, X, ln1_g, Wqkv, Wo, ln2_g, W1s, W2s, save, dZ, dX, dln1_g,
                    dln1_b, dWqkv, dWo, dln2_g, dln2_b, dW1s, dW2s, ws=None, stream=None) -> int:
    """The layer's backward with X, dZ and dX sequence-sharded."""
    return _layer_bwd("tp_sp_layer_bwd", dtype, B, S, h, H, d, f, N, causal, X, ln1_g, Wqkv, Wo, ln2_g, W1s, W2s,
                      save, dZ, dX, dln1_g, dln1_b, dWqkv, dWo, dln2_g, dln2_b, dW1s, dW2s, ws, stream)


# ---------------------------------------------------------------- attention block
def tp_attn_workspace_bytes(dtype: int, B: int, S: int, h: int, H: int, d: int, N: int) -> int:
    return load_library().tp_attn_workspace_bytes(dtype, B, S, h, H, d, N)


def tp_attn_fwd(dtype, B, S, h, H, d, N, causal, X, Wqkv, Wo, QKV_save, O_save, LSE_save, Z, ws=None,
                stream=None) -> int:
    dt = _TORCH_DT.get(dtype)
    T = B * S
    wptr, wbytes = _ws(ws, tp_attn_workspace_bytes(dtype, B, S, h, H, d, N))
    return _check(load_library().tp_attn_fwd(
        dtype, B, S, h, H, d, N, int(causal), _p(X, "X", dt, T * h), _p(Wqkv, "Wqkv", dt, h * 3 * H * d),
        _p(Wo, "Wo", dt, H * d * h), _p(QKV_save, "QKV_save", dt, T * QKV_PLANES * H * d, False),
        _p(O_save, "O_save", dt, T * H * d, False), _p(LSE_save, "LSE_save", torch.float32, T * H, False),
        _p(Z, "Z", dt, T * h), wptr, wbytes, _stream(stream)), "tp_attn_fwd")


def tp_attn_bwd(dtype, B, S, h, H, d, N, causal, X, Wqkv, Wo, QKV_save, O_save, LSE_save, dZ, dX, dWqkv, dWo,
                ws=None, stream=None) -> int:
    dt = _TORCH_DT.get(dtype)
    T = B * S
    wptr, wbytes = _ws(ws, tp_attn_workspace_bytes(dtype, B, S, h, H, d, N))
    return _check(load_library().tp_attn_bwd(
        dtype, B, S, h, H, d, N, int(causal), _p(X, "X", dt, T * h), _p(Wqkv, "Wqkv", dt, h * 3 * H * d),
        _p(Wo, "Wo", dt, H * d * h), _p(QKV_save, "QKV_save", dt, T * QKV_PLANES * H * d),
        _p(O_save, "O_save", dt, T * H * d), _p(LSE_save, "LSE_save", torch.float32, T * H),
        _p(dZ, "dZ", dt, T * h), _p(dX, "dX", dt, T * h), _p(dWqkv, "dWqkv", dt, h * 3 * H * d),
        _p(dWo, "dWo", dt, H * d * h), wptr, wbytes, _stream(stream)), "tp_attn_bwd")


# ---------------------------------------------------------------- attention block then MLP block
def tp_attn_mlp_save_bytes(dtype, B, S, h, H, d, f, N) -> int:
    return load_library().tp_attn_mlp_save_bytes(dtype, B, S, h, H, d, f, N)


def tp_attn_mlp_workspace_bytes(dtype, B, S, h, H, d, f, N) -> int:
    return load_library().tp_attn_mlp_workspace_bytes(dtype, B, S, h, H, d, f, N)


def tp_attn_mlp_fwd(dtype, B, S, h, H, d, f, N, causal, X, Wqkv, Wo, W1s, W2s, save, Z, stream=None) -> int:
    """Z = MLP(Attn(X)); ``save`` receives what the backward needs."""
    dt = _TORCH_DT.get(dtype)
    T = B * S
    sptr, sbytes = _ws(save, tp_attn_mlp_save_bytes(dtype, B, S, h, H, d, f, N))
    return _check(load_library().tp_attn_mlp_fwd(
        dtype, B, S, h, H, d, f, N, 1 if causal else 0, _p(X, "X", dt, T * h), _p(Wqkv, "Wqkv", dt, 3 * h * H * d),
        _p(Wo, "Wo", dt, H * d * h), _p(W1s, "W1s", dt, h * f), _p(W2s, "W2s", dt, f * h), sptr, sbytes,
        _p(Z, "Z", dt, T * h), _stream(stream)), "tp_attn_mlp_fwd")


def tp_attn_mlp_bwd(dtype, B, S, h, H, d, f, N, causal, X, Wqkv, Wo, W1s, W2s, save, dZ, dX, dWqkv, dWo, dW1s, dW2s,
                    ws=None, stream=None) -> int:
    dt = _TORCH_DT.get(dtype)
    T = B * S
    sptr, sbytes = _ws(save, tp_attn_mlp_save_bytes(dtype, B, S, h, H, d, f, N))
    wptr, wbytes = _ws(ws, tp_attn_mlp_workspace_bytes(dtype, B, S, h, H, d, f, N))
    return _check(load_library().tp_attn_mlp_bwd(
        dtype, B, S, h, H, d, f, N, 1 if causal else 0, _p(X, "X", dt, T * h), _p(Wqkv, "Wqkv", dt, 3 * h * H * d),
        _p(Wo, "Wo", dt, H * d * h), _p(W1s, "W1s", dt, h * f), _p(W2s, "W2s", dt, f * h), sptr, sbytes,
        _p(dZ, "dZ", dt, T * h), _p(dX, "dX", dt, T * h), _p(dWqkv, "dWqkv", dt, 3 * h * H * d),
        _p(dWo, "dWo", dt, H * d * h), _p(dW1s, "dW1s", dt, h * f), _p(dW2s, "dW2s", dt, f * h), wptr, wbytes,
        _stream(stream)), "tp_attn_mlp_bwd")


def tp_set_gemm_tiling(mode: int) -> int:
    """0 automatic, 1 one CTA per 128x256 tile, 2 CTA pairs per 256x256 tile."""
    return _check(load_library().tp_set_gemm_tiling(mode), "tp_set_gemm_tiling")


def tp_set_launch_overlap(on: bool) -> int:
    """True (default): each kernel's prologue overlaps the previous kernel's tail
    (programmatic dependent launch); False: ordinary stream order."""
    return _check(load_library().tp_set_launch_overlap(1 if on else 0), "tp_set_launch_overlap")


# ---------------------------------------------------------------- kernel timing
def tp_timing_enable(on: bool) -> int:
    return _check(load_library().tp_timing_enable(1 if on else 0), "tp_timing_enable")


def tp_timing_kinds() -> int:
    return load_library().tp_timing_kinds()


def tp_timing_name(kind: int) -> str:
    r = load_library().tp_timing_name(kind)
    return r.decode() if r else ""


def tp_timing_read(kind: int) -> tuple[int, float]:
    n = ctypes.c_int64(0)
    t = ctypes.c_double(0.0)
    _check(load_library().tp_timing_read(kind, ctypes.byref(n), ctypes.byref(t)), "tp_timing_read")
    return int(n.value), float(t.value)


def timing_report() -> dict:
    """{kernel kind name: (launches, total event-measured ms)} for every kind launched."""
    out = {}
    for k in range(tp_timing_kinds()):
        n, ms = tp_timing_read(k)
        if n:
            out[tp_timing_name(k)] = (n, ms)
    return out
