"""Convenience layer over the C-ABI: allocates outputs and scratch with torch
(device memory is torch's job) and calls the libtpblock entry points.  No
arithmetic happens here; every step of the block runs in the CUDA library."""
from __future__ import annotations

import torch

from . import _binding as B

_DT = {torch.float32: B.TP_F32, torch.bfloat16: B.TP_BF16}


def _dtype(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise ValueError(f"unsupported dtype {t.dtype}")
    return _DT[t.dtype]


def workspace(nbytes: int, device) -> torch.Tensor:
    """A 256-byte aligned scratch buffer of at least ``nbytes`` bytes."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def mlp_forward(X, W1s, W2s, save: bool = True, ws=None, stream=None) -> dict:
    """Z = sum_i GeLU(X W1_i) W2_i.  With ``save`` the pre-activation Y and the
    activation A (both [N][T][f/N]) are returned for the backward."""
    N, h, fN = W1s.shape
    T = X.shape[0]
    f = N * fN
    dt = _dtype(X)
    dev = X.device
    Z = torch.empty(T, h, dtype=X.dtype, device=dev)
    Y = torch.empty(N, T, fN, dtype=X.dtype, device=dev) if save else None
    A = torch.empty(N, T, fN, dtype=X.dtype, device=dev) if save else None
    if ws is None:  # scratch for A when it is not saved, and split-K partials for small shapes
        ws = workspace(B.tp_mlp_workspace_bytes(dt, T, h, f, N), dev)
    B.tp_mlp_fwd(dt, T, h, f, N, X, W1s, W2s, Y, A, Z, ws, stream)
    return {"Z": Z, "Y": Y, "A": A}


def mlp_backward(X, W1s, W2s, Y, A, dZ, ws=None, stream=None, out=None) -> dict:
    """dX, dW1s, dW2s of L = <dZ, Z> for the block whose forward saved Y and A."""
    N, h, fN = W1s.shape
    T = X.shape[0]
    f = N * fN
    dt = _dtype(X)
    dev = X.device
    if out is None:
        out = {"dX": torch.empty(T, h, dtype=X.dtype, device=dev),
               "dW1s": torch.empty(N, h, fN, dtype=X.dtype, device=dev),
               "dW2s": torch.empty(N, fN, h, dtype=X.dtype, device=dev)}
    if ws is None:
        ws = workspace(B.tp_mlp_workspace_bytes(dt, T, h, f, N), dev)
    B.tp_mlp_bwd(dt, T, h, f, N, X, W1s, W2s, Y, A, dZ, out["dX"], out["dW1s"], out["dW2s"], ws, stream)
    return out


def gmlp_forward(X, Wgus, Wds, save: bool = True, ws=None, stream=None) -> dict:
    """Z = sum_i (silu(X Wg_i) * (X Wu_i)) Wd_i.  With ``save`` the gate and up
    pre-activations GU ([N][T][2][f/N]) and the activation A ([N][T][f/N]) are
    returned for the backward."""
    N, h, two, fN = Wgus.shape
    assert two == 2
    T = X.shape[0]
    f = N * fN
    dt = _dtype(X)
    dev = X.device
    Z = torch.empty(T, h, dtype=X.dtype, device=dev)
    GU = torch.empty(N, T, 2, fN, dtype=X.dtype, device=dev) if save else None
    A = torch.empty(N, T, fN, dtype=X.dtype, device=dev) if save else None
    if A is None and ws is None:
        ws = workspace(B.tp_gmlp_workspace_bytes(dt, T, h, f, N), dev)
    B.tp_gmlp_fwd(dt, T, h, f, N, X, Wgus, Wds, GU, A, Z, ws, stream)
    return {"Z": Z, "GU": GU, "A": A}


def gmlp_backward(X, Wgus, Wds, GU, A, dZ, ws=None, stream=None, out=None) -> dict:
    """dX, dWgus, dWds of L = <dZ, Z> for the gated block whose forward saved GU and A."""
    N, h, _, fN = Wgus.shape
    T = X.shape[0]
    f = N * fN
    dt = _dtype(X)
    dev = X.device
    if out is None:
        out = {"dX": torch.empty(T, h, dtype=X.dtype, device=dev),
               "dWgus": torch.empty_like(Wgus), "dWds": torch.empty_like(Wds)}
    if ws is None:
        ws = workspace(B.tp_gmlp_workspace_bytes(dt, T, h, f, N), dev)
    B.tp_gmlp_bwd(dt, T, h, f, N, X, Wgus, Wds, GU, A, dZ, out["dX"], out["dWgus"], out["dWds"], ws, stream)
    return out


def attn_forward(X, Wqkv, Wo, B_: int, S: int, causal: bool = True, save: bool = True, ws=None,
                 stream=None) -> dict:
    """Z = sum_i O_i Wo_i with O the per-head causal attention of X Wqkv_i."""
    N, h, _, hN, d = Wqkv.shape
    H = N * hN
    T = B_ * S
    dt = _dtype(X)
    dev = X.device
    Z = torch.empty(T, h, dtype=X.dtype, device=dev)
    QKV = torch.empty(N, T, B.QKV_PLANES * hN * d, dtype=X.dtype, device=dev) if save else None
    O = torch.empty(N, T, hN * d, dtype=X.dtype, device=dev) if save else None
    LSE = torch.empty(B_, H, S, dtype=torch.float32, device=dev) if save else None
    if ws is None:
        ws = workspace(B.tp_attn_workspace_bytes(dt, B_, S, h, H, d, N), dev)
    B.tp_attn_fwd(dt, B_, S, h, H, d, N, causal, X, Wqkv, Wo, QKV, O, LSE, Z, ws, stream)
    return {"Z": Z, "QKV": QKV, "O": O, "LSE": LSE}


def gqa_forward(X, Wqkv, Wo, H: int, Hkv: int, d: int, B_: int, S: int, causal: bool = True, ws=None,
                stream=None) -> dict:
    """Grouped-query attention block: Wqkv [N][h][(H/N + 2 Hkv/N) d]."""
    N, h, _ = Wqkv.shape
    T = B_ * S
    dt = _dtype(X)
    dev = X.device
    Z = torch.empty(T, h, dtype=X.dtype, device=dev)
    QKV = torch.empty(N, T, (H + 2 * Hkv) * d // N, dtype=X.dtype, device=dev)
    O = torch.empty(N, T, H * d // N, dtype=X.dtype, device=dev)
    LSE = torch.empty(B_, H, S, dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(B.tp_gqa_workspace_bytes(dt, B_, S, h, H, Hkv, d, N), dev)
    B.tp_gqa_fwd(dt, B_, S, h, H, Hkv, d, N, causal, X, Wqkv, Wo, QKV, O, LSE, Z, ws, stream)
    return {"Z": Z, "QKV": QKV, "O": O, "LSE": LSE}


def gqa_backward(X, Wqkv, Wo, QKV, O, LSE, dZ, H: int, Hkv: int, d: int, B_: int, S: int, causal: bool = True,
                 ws=None, stream=None) -> dict:
    N, h, _ = Wqkv.shape
    T = B_ * S
    dt = _dtype(X)
    dev = X.device
    out = {"dX": torch.empty(T, h, dtype=X.dtype, device=dev), "dWqkv": torch.empty_like(Wqkv),
           "dWo": torch.empty_like(Wo)}
    if ws is None:
        ws = workspace(B.tp_gqa_workspace_bytes(dt, B_, S, h, H, Hkv, d, N), dev)
    B.tp_gqa_bwd(dt, B_, S, h, H, Hkv, d, N, causal, X, Wqkv, Wo, QKV, O, LSE, dZ, out["dX"], out["dWqkv"], out["dWo"],
                 ws, stream)
    return out


def attn_backward(X, Wqkv, Wo, QKV, O, LSE, dZ, B_: int, S: int, causal: bool = True, ws=None, stream=None,
                  out=None) -> dict:
    N, h, _, hN, d = Wqkv.shape
    H = N * hN
    T = B_ * S
    dt = _dtype(X)
    dev = X.device
    if out is None:
        out = {"dX": torch.empty(T, h, dtype=X.dtype, device=dev),
               "dWqkv": torch.empty_like(Wqkv), "dWo": torch.empty_like(Wo)}
    if ws is None:
        ws = workspace(B.tp_attn_workspace_bytes(dt, B_, S, h, H, d, N), dev)
    B.tp_attn_bwd(dt, B_, S, h, H, d, N, causal, X, Wqkv, Wo, QKV, O, LSE, dZ, out["dX"], out["dWqkv"],
                  out["dWo"], ws, stream)
    return out


LN_EPS = 1e-5


def layernorm_forward(X, gamma, beta, eps: float = LN_EPS, stream=None) -> dict:
    """Y = gamma * (X - mean) / sqrt(var + eps) + beta per row, with the row statistics."""
    T, h = X.shape
    dev = X.device
    Y = torch.empty_like(X)
    mean = torch.empty(T, dtype=torch.float32, device=dev)
    rstd = torch.empty(T, dtype=torch.float32, device=dev)
    B.tp_layernorm_fwd(_dtype(X), T, h, eps, X, gamma, beta, Y, mean, rstd, stream)
    return {"Y": Y, "mean": mean, "rstd": rstd}


def layernorm_backward(X, gamma, mean, rstd, dY, dR=None, ws=None, stream=None) -> dict:
    """dX (+ dR), dgamma, dbeta of the LayerNorm whose forward gave mean and rstd."""
    T, h = X.shape
    dev = X.device
    dt = _dtype(X)
    out = {"dX": torch.empty_like(X), "dgamma": torch.empty_like(gamma), "dbeta": torch.empty_like(gamma)}
    if ws is None:
        ws = workspace(B.tp_layernorm_workspace_bytes(dt, T, h), dev)
    B.tp_layernorm_bwd(dt, T, h, X, gamma, mean, rstd, dY, dR, out["dX"], out["dgamma"], out["dbeta"], ws, stream)
    return out


def prenorm_layer_forward(X, p: dict, B_: int, S: int, causal: bool = True, eps: float = LN_EPS, save=None,
                          stream=None, seq_sharded: bool = False) -> dict:
    """H1 = X + Attn(LN1(X)), Z = H1 + MLP(LN2(H1)).  ``p`` holds ln1_g, ln1_b, Wqkv,
    Wo, ln2_g, ln2_b, W1s, W2s; the returned ``save`` buffer feeds the backward.
    With ``seq_sharded`` X and Z are in the sequence-parallel layout [N][B][S/N][h]."""
    N, h, _, hN, d = p["Wqkv"].shape
    H = N * hN
    f = N * p["W1s"].shape[2]
    dt = _dtype(X)
    if save is None:
        save = workspace(B.tp_layer_save_bytes(dt, B_, S, h, H, d, f, N), X.device)
    Z = torch.empty_like(X)
    fn = B.tp_sp_layer_fwd if seq_sharded else B.tp_layer_fwd
    fn(dt, B_, S, h, H, d, f, N, causal, eps, X, p["ln1_g"], p["ln1_b"], p["Wqkv"], p["Wo"], p["ln2_g"], p["ln2_b"],
       p["W1s"], p["W2s"], save, Z, stream)
    return {"Z": Z, "save": save}


def prenorm_layer_backward(X, p: dict, save, dZ, B_: int, S: int, causal: bool = True, ws=None, stream=None,
                           out=None, seq_sharded: bool = False) -> dict:
    N, h, _, hN, d = p["Wqkv"].shape
    H = N * hN
    f = N * p["W1s"].shape[2]
    dt = _dtype(X)
    if out is None:
        out = {"dX": torch.empty_like(X), "dln1_g": torch.empty_like(p["ln1_g"]),
               "dln1_b": torch.empty_like(p["ln1_b"]), "dWqkv": torch.empty_like(p["Wqkv"]),
               "dWo": torch.empty_like(p["Wo"]), "dln2_g": torch.empty_like(p["ln2_g"]),
               "dln2_b": torch.empty_like(p["ln2_b"]), "dW1s": torch.empty_like(p["W1s"]),
               "dW2s": torch.empty_like(p["W2s"])}
    if ws is None:
        ws = workspace(B.tp_layer_workspace_bytes(dt, B_, S, h, H, d, f, N), X.device)
    fn = B.tp_sp_layer_bwd if seq_sharded else B.tp_layer_bwd
    fn(dt, B_, S, h, H, d, f, N, causal, X, p["ln1_g"], p["Wqkv"], p["Wo"], p["ln2_g"], p["W1s"], p["W2s"], save, dZ,
       out["dX"], out["dln1_g"], out["dln1_b"], out["dWqkv"], out["dWo"], out["dln2_g"], out["dln2_b"], out["dW1s"],
       out["dW2s"], ws, stream)
    return out


def attn_mlp_forward(X, p: dict, B_: int, S: int, causal: bool = True, save=None, stream=None) -> dict:
    """Z = MLP(Attn(X)): the attention block then the MLP block in one call (the
    attention output stays in the library's save buffer, in fp16).  ``p`` holds
    Wqkv, Wo, W1s, W2s; the returned ``save`` buffer feeds the backward."""
    N, h, _, hN, d = p["Wqkv"].shape
    H = N * hN
    f = N * p["W1s"].shape[2]
    dt = _dtype(X)
    if save is None:
        save = workspace(B.tp_attn_mlp_save_bytes(dt, B_, S, h, H, d, f, N), X.device)
    Z = torch.empty_like(X)
    B.tp_attn_mlp_fwd(dt, B_, S, h, H, d, f, N, causal, X, p["Wqkv"], p["Wo"], p["W1s"], p["W2s"], save, Z, stream)
    return {"Z": Z, "save": save}


def attn_mlp_backward(X, p: dict, save, dZ, B_: int, S: int, causal: bool = True, ws=None, stream=None,
                      out=None) -> dict:
    N, h, _, hN, d = p["Wqkv"].shape
    H = N * hN
    f = N * p["W1s"].shape[2]
    dt = _dtype(X)
    if out is None:
        out = {"dX": torch.empty_like(X), "dWqkv": torch.empty_like(p["Wqkv"]), "dWo": torch.empty_like(p["Wo"]),
               "dW1s": torch.empty_like(p["W1s"]), "dW2s": torch.empty_like(p["W2s"])}
    if ws is None:
        ws = workspace(B.tp_attn_mlp_workspace_bytes(dt, B_, S, h, H, d, f, N), X.device)
    B.tp_attn_mlp_bwd(dt, B_, S, h, H, d, f, N, causal, X, p["Wqkv"], p["Wo"], p["W1s"], p["W2s"], save, dZ,
                      out["dX"], out["dWqkv"], out["dWo"], out["dW1s"], out["dW2s"], ws, stream)
    return out
