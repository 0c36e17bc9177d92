"""Seeded synthetic inputs for the tensor-parallel block, shared by the CUDA path's
tests/benchmark and by the fp64 oracle.

This module draws random numbers and arranges them in the shard-major layouts of
the boundary; it contains none of the block's arithmetic.  Draws are fp32 normals
from a CPU ``torch.Generator`` seeded once, in a fixed order (MLP: X, W1, W2, dZ;
gated MLP: X, W_gate, W_up, W_down, dZ; attention: X, Wqkv, Wo, dZ; layer: X, Wqkv,
Wo, W1, W2, dZ; pre-norm layer: X, ln1 gamma, ln1 beta, Wqkv, Wo, ln2 gamma, ln2
beta, W1, W2, dZ), scaled by the stated
standard deviation and cast to the workload's dtype once.  The GPU and the oracle
then consume the identical values (the oracle upcasts them to float64).

Weights are drawn unsharded in the pages' [in x out] orientation and then cut the
way the pages cut them:
  * W1 [h x f] -> W1s [N][h][f/N]           (column split)
  * W2 [f x h] -> W2s [N][f/N][h]           (row split; bit-identical to W2)
  * W_gate, W_up [h x f] -> Wgus [N][h][2][f/N]  (both split by columns; shard i
    holds its gate columns, then the same columns of W_up)
  * W_down [f x h] -> Wds [N][f/N][h]       (row split)
  * Wqkv [h x 3*H*d] (Q heads | K heads | V heads) -> [N][h][3][H/N][d]
  * Wo [H*d x h] -> [N][H/N*d][h]           (row split by head)
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

__all__ = ["Workload", "WORKLOADS", "mlp_inputs", "gmlp_inputs", "attn_inputs", "layer_inputs", "prenorm_inputs",
           "ln_inputs", "gqa_inputs", "split_qkv_gqa", "to_seq_shards", "from_seq_shards",
           "split_columns", "split_rows", "split_qkv_heads"]


@dataclass(frozen=True)
class Workload:
    """One of the synthetic workloads the block is checked and measured on."""
    name: str
    kind: str            # "mlp", "gmlp" (gated MLP), "attn", "gqa", "layer", "lnlayer" (pre-norm layer) or
                         # "splayer" (the pre-norm layer with sequence-sharded activations)
    dtype: str           # "f32" or "bf16"
    backward: bool
    T: int = 0           # tokens = B*S
    h: int = 0
    f: int = 0
    N: int = 1
    B: int = 1
    S: int = 0
    H: int = 0
    d: int = 0
    Hkv: int = 0         # key/value heads (grouped-query attention)
    causal: bool = True
    x_std: float = 1.0
    w_std: float = 0.02
    seed: int = 0

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k in self.__dataclass_fields__}


# The workloads: MLP fp32 forward; MLP bf16 fwd+bwd (small and h=4096);
# attention bf16 forward; full layer bf16 fwd+bwd; gated MLP bf16 fwd+bwd.
WORKLOADS = {
    "mlp_f32_T64_h256_f1024_N2": Workload("mlp_f32_T64_h256_f1024_N2", "mlp", "f32", False,
                                          T=64, h=256, f=1024, N=2),
    "mlp_bf16_T2048_h1024_f4096_N4": Workload("mlp_bf16_T2048_h1024_f4096_N4", "mlp", "bf16", True,
                                              T=2048, h=1024, f=4096, N=4),
    "mlp_bf16_T8192_h4096_f16384_N8": Workload("mlp_bf16_T8192_h4096_f16384_N8", "mlp", "bf16", True,
                                               T=8192, h=4096, f=16384, N=8),
    "attn_bf16_B2_S2048_h4096_H32_d128_N8": Workload("attn_bf16_B2_S2048_h4096_H32_d128_N8", "attn",
                                                     "bf16", False, T=4096, h=4096, N=8, B=2,
                                                     S=2048, H=32, d=128),
    "layer_bf16_B1_S4096_h8192_H64_d128_f28672_N8": Workload(
        "layer_bf16_B1_S4096_h8192_H64_d128_f28672_N8", "layer", "bf16", True,
        T=4096, h=8192, f=28672, N=8, B=1, S=4096, H=64, d=128),
    "lnlayer_bf16_B1_S4096_h8192_H64_d128_f28672_N8": Workload(
        "lnlayer_bf16_B1_S4096_h8192_H64_d128_f28672_N8", "lnlayer", "bf16", True,
        T=4096, h=8192, f=28672, N=8, B=1, S=4096, H=64, d=128),
    "splayer_bf16_B2_S2048_h8192_H64_d128_f28672_N8": Workload(
        "splayer_bf16_B2_S2048_h8192_H64_d128_f28672_N8", "splayer", "bf16", True,
        T=4096, h=8192, f=28672, N=8, B=2, S=2048, H=64, d=128),
    "gqa_bf16_B2_S2048_h4096_H32_Hkv8_d128_N8": Workload("gqa_bf16_B2_S2048_h4096_H32_Hkv8_d128_N8", "gqa",
                                                         "bf16", True, T=4096, h=4096, N=8, B=2, S=2048, H=32,
                                                         d=128, Hkv=8),
    "gmlp_bf16_T8192_h4096_f12288_N8": Workload("gmlp_bf16_T8192_h4096_f12288_N8", "gmlp", "bf16", True,
                                                T=8192, h=4096, f=12288, N=8),
}

_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def _draw(gen: torch.Generator, shape, std: float, dtype: str) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(_DT[dtype]).contiguous()


def split_columns(w: torch.Tensor, n: int) -> torch.Tensor:
    """[rows][cols] -> [n][rows][cols/n]: block i holds columns i*cols/n..(i+1)*cols/n-1."""
    rows, cols = w.shape
    return w.reshape(rows, n, cols // n).permute(1, 0, 2).contiguous()


def split_rows(w: torch.Tensor, n: int) -> torch.Tensor:
    """[rows][cols] -> [n][rows/n][cols] (same bytes as the input)."""
    rows, cols = w.shape
    return w.reshape(n, rows // n, cols).contiguous()


def split_qkv_heads(w: torch.Tensor, n: int, H: int, d: int) -> torch.Tensor:
    """[h][3*H*d] laid out (Q heads | K heads | V heads) -> [n][h][3][H/n][d]."""
    h = w.shape[0]
    return w.reshape(h, 3, n, H // n, d).permute(2, 0, 1, 3, 4).contiguous()


def mlp_inputs(T: int, h: int, f: int, N: int, dtype: str = "bf16", seed: int = 0,
               x_std: float = 1.0, w_std: float = 0.02, backward: bool = True) -> dict:
    """X [T][h], W1s [N][h][f/N], W2s [N][f/N][h] and (if ``backward``) dZ [T][h],
    all CPU tensors of ``dtype``."""
    if N < 1 or f % N:
        raise ValueError("N must divide f")
    gen = torch.Generator().manual_seed(seed)
    X = _draw(gen, (T, h), x_std, dtype)
    W1 = _draw(gen, (h, f), w_std, dtype)
    W2 = _draw(gen, (f, h), w_std, dtype)
    out = {"X": X, "W1s": split_columns(W1, N), "W2s": split_rows(W2, N)}
    if backward:
        out["dZ"] = _draw(gen, (T, h), 1.0, dtype)
    return out


def gmlp_inputs(T: int, h: int, f: int, N: int, dtype: str = "bf16", seed: int = 0,
                x_std: float = 1.0, w_std: float = 0.02, backward: bool = True) -> dict:
    """Gated MLP: X [T][h], Wgus [N][h][2][f/N], Wds [N][f/N][h] and (if
    ``backward``) dZ [T][h]; f is the width of each of the gate and up projections."""
    if N < 1 or f % N:
        raise ValueError("N must divide f")
    gen = torch.Generator().manual_seed(seed)
    X = _draw(gen, (T, h), x_std, dtype)
    Wg = _draw(gen, (h, f), w_std, dtype)
    Wu = _draw(gen, (h, f), w_std, dtype)
    Wd = _draw(gen, (f, h), w_std, dtype)
    out = {"X": X, "Wgus": torch.stack([split_columns(Wg, N), split_columns(Wu, N)], dim=2).contiguous(),
           "Wds": split_rows(Wd, N)}
    if backward:
        out["dZ"] = _draw(gen, (T, h), 1.0, dtype)
    return out


def attn_inputs(B: int, S: int, h: int, H: int, d: int, N: int, dtype: str = "bf16",
                seed: int = 0, x_std: float = 1.0, w_std: float = 0.02,
                backward: bool = True) -> dict:
    """X [B*S][h], Wqkv [N][h][3][H/N][d], Wo [N][H/N*d][h] and dZ [B*S][h]."""
    if N < 1 or H % N:
        raise ValueError("N must divide H")
    gen = torch.Generator().manual_seed(seed)
    X = _draw(gen, (B * S, h), x_std, dtype)
    Wqkv = _draw(gen, (h, 3 * H * d), w_std, dtype)
    Wo = _draw(gen, (H * d, h), w_std, dtype)
    out = {"X": X, "Wqkv": split_qkv_heads(Wqkv, N, H, d), "Wo": split_rows(Wo, N)}
    if backward:
        out["dZ"] = _draw(gen, (B * S, h), 1.0, dtype)
    return out


def layer_inputs(B: int, S: int, h: int, H: int, d: int, f: int, N: int, dtype: str = "bf16",
                 seed: int = 0, x_std: float = 1.0, w_std: float = 0.02) -> dict:
    """Inputs of the attention block followed by the MLP block."""
    if N < 1 or H % N or f % N:
        raise ValueError("N must divide H and f")
    gen = torch.Generator().manual_seed(seed)
    X = _draw(gen, (B * S, h), x_std, dtype)
    Wqkv = _draw(gen, (h, 3 * H * d), w_std, dtype)
    Wo = _draw(gen, (H * d, h), w_std, dtype)
    W1 = _draw(gen, (h, f), w_std, dtype)
    W2 = _draw(gen, (f, h), w_std, dtype)
    dZ = _draw(gen, (B * S, h), 1.0, dtype)
    return {"X": X, "Wqkv": split_qkv_heads(Wqkv, N, H, d), "Wo": split_rows(Wo, N),
            "W1s": split_columns(W1, N), "W2s": split_rows(W2, N), "dZ": dZ}


def split_qkv_gqa(Wq: torch.Tensor, Wk: torch.Tensor, Wv: torch.Tensor, n: int) -> torch.Tensor:
    """[h][H d], [h][Hkv d], [h][Hkv d] -> [n][h][(H/n + 2 Hkv/n) d]: shard i holds its
    query heads' columns, then its key heads', then its value heads'."""
    q, k, v = (w.reshape(w.shape[0], n, w.shape[1] // n) for w in (Wq, Wk, Wv))
    return torch.cat([q, k, v], dim=2).permute(1, 0, 2).contiguous()


def gqa_inputs(B: int, S: int, h: int, H: int, Hkv: int, d: int, N: int, dtype: str = "bf16", seed: int = 0,
               x_std: float = 1.0, w_std: float = 0.02, backward: bool = True) -> dict:
    """Grouped-query attention: X [B*S][h], Wqkv [N][h][(H/N + 2 Hkv/N) d] (W_Q, W_K,
    W_V drawn in that order), Wo [N][H/N*d][h], dZ [B*S][h]."""
    if N < 1 or H % Hkv or Hkv % N:
        raise ValueError("Hkv must divide H and N must divide Hkv")
    gen = torch.Generator().manual_seed(seed)
    X = _draw(gen, (B * S, h), x_std, dtype)
    Wq = _draw(gen, (h, H * d), w_std, dtype)
    Wk = _draw(gen, (h, Hkv * d), w_std, dtype)
    Wv = _draw(gen, (h, Hkv * d), w_std, dtype)
    Wo = _draw(gen, (H * d, h), w_std, dtype)
    out = {"X": X, "Wqkv": split_qkv_gqa(Wq, Wk, Wv, N), "Wo": split_rows(Wo, N)}
    if backward:
        out["dZ"] = _draw(gen, (B * S, h), 1.0, dtype)
    return out


def to_seq_shards(X: torch.Tensor, B: int, S: int, n: int) -> torch.Tensor:
    """[B*S][h] (token t = b*S + s) -> [n][B][S/n][h]: the sequence-parallel layout,
    shard c holding positions c*S/n .. (c+1)*S/n - 1 of every sequence."""
    return X.reshape(B, n, S // n, X.shape[-1]).permute(1, 0, 2, 3).contiguous()


def from_seq_shards(Xs: torch.Tensor) -> torch.Tensor:
    """Inverse of :func:`to_seq_shards`."""
    n, B, L, h = Xs.shape
    return Xs.permute(1, 0, 2, 3).reshape(B * n * L, h).contiguous()


def ln_inputs(T: int, h: int, dtype: str = "bf16", seed: int = 0, x_std: float = 1.0, x_mean: float = 0.0,
              ln_std: float = 0.1) -> dict:
    """LayerNorm alone: X [T][h] ~ N(x_mean, x_std^2), gamma ~ 1 + N(0, ln_std^2),
    beta ~ N(0, ln_std^2), upstream dY and residual gradient dR ~ N(0, 1)."""
    gen = torch.Generator().manual_seed(seed)
    X = (torch.randn(T, h, generator=gen) * x_std + x_mean).to(_DT[dtype])
    g = (_draw(gen, (h,), ln_std, "f32") + 1.0).to(_DT[dtype])
    b = _draw(gen, (h,), ln_std, dtype)
    dY = _draw(gen, (T, h), 1.0, dtype)
    dR = _draw(gen, (T, h), 1.0, dtype)
    return {"X": X, "gamma": g, "beta": b, "dY": dY, "dR": dR}


def prenorm_inputs(B: int, S: int, h: int, H: int, d: int, f: int, N: int, dtype: str = "bf16",
                   seed: int = 0, x_std: float = 1.0, w_std: float = 0.02, ln_std: float = 0.1) -> dict:
    """Inputs of the pre-norm layer: the layer's plus LayerNorm gamma ~ 1 + N(0, ln_std^2)
    and beta ~ N(0, ln_std^2), each [h] (perturbed from the usual 1 / 0 start so that
    they take part in every check)."""
    if N < 1 or H % N or f % N:
        raise ValueError("N must divide H and f")
    gen = torch.Generator().manual_seed(seed)
    X = _draw(gen, (B * S, h), x_std, dtype)
    g1 = (_draw(gen, (h,), ln_std, "f32") + 1.0).to(_DT[dtype])
    b1 = _draw(gen, (h,), ln_std, dtype)
    Wqkv = _draw(gen, (h, 3 * H * d), w_std, dtype)
    Wo = _draw(gen, (H * d, h), w_std, dtype)
    g2 = (_draw(gen, (h,), ln_std, "f32") + 1.0).to(_DT[dtype])
    b2 = _draw(gen, (h,), ln_std, dtype)
    W1 = _draw(gen, (h, f), w_std, dtype)
    W2 = _draw(gen, (f, h), w_std, dtype)
    dZ = _draw(gen, (B * S, h), 1.0, dtype)
    return {"X": X, "ln1_g": g1, "ln1_b": b1, "Wqkv": split_qkv_heads(Wqkv, N, H, d), "Wo": split_rows(Wo, N),
            "ln2_g": g2, "ln2_b": b2, "W1s": split_columns(W1, N), "W2s": split_rows(W2, N), "dZ": dZ}


def workload_inputs(w: Workload, **overrides) -> dict:
    """Inputs for a :class:`Workload` (shape fields may be overridden)."""
    p = {**w.as_dict(), **overrides}
    if p["kind"] == "mlp":
        return mlp_inputs(p["T"], p["h"], p["f"], p["N"], p["dtype"], p["seed"], p["x_std"],
                          p["w_std"], p["backward"])
    if p["kind"] == "gmlp":
        return gmlp_inputs(p["T"], p["h"], p["f"], p["N"], p["dtype"], p["seed"], p["x_std"],
                           p["w_std"], p["backward"])
    if p["kind"] == "gqa":
        return gqa_inputs(p["B"], p["S"], p["h"], p["H"], p["Hkv"], p["d"], p["N"], p["dtype"], p["seed"],
                          p["x_std"], p["w_std"], p["backward"])
    if p["kind"] == "attn":
        return attn_inputs(p["B"], p["S"], p["h"], p["H"], p["d"], p["N"], p["dtype"], p["seed"],
                           p["x_std"], p["w_std"], p["backward"])
    if p["kind"] in ("lnlayer", "splayer"):
        return prenorm_inputs(p["B"], p["S"], p["h"], p["H"], p["d"], p["f"], p["N"], p["dtype"],
                              p["seed"], p["x_std"], p["w_std"])
    return layer_inputs(p["B"], p["S"], p["h"], p["H"], p["d"], p["f"], p["N"], p["dtype"],
                        p["seed"], p["x_std"], p["w_std"])
