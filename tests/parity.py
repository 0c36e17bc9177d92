"""Parity criteria of the CUDA path against the fp64 oracle.

bf16 storage with fp32 accumulation: relative Frobenius error <= 5e-3 and, in
every output column, max |gpu - oracle| <= 2e-2 x that column's RMS in the oracle.
fp32: relative Frobenius error <= 1e-5.  Columns are the last axis; for a
shard-major [N][rows][cols] tensor each (shard, column) pair is one column of
the unsharded matrix, so statistics are taken over axis -2.
"""
from __future__ import annotations

import numpy as np

BF16_REL_FRO = 5e-3
BF16_COL_MAXABS = 2e-2
F32_REL_FRO = 1e-5


def errors(gpu, ref) -> dict:
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    if g.shape != r.shape:
        raise AssertionError(f"shape {g.shape} != oracle {r.shape}")
    if r.ndim == 1:
        g, r = g[:, None], r[:, None]
    g3 = g.reshape(-1, g.shape[-2], g.shape[-1])
    r3 = r.reshape(-1, r.shape[-2], r.shape[-1])
    fro = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300))
    rms = np.sqrt(np.mean(r3 * r3, axis=1))
    maxabs = np.max(np.abs(g3 - r3), axis=1)
    col = maxabs / np.maximum(rms, 1e-30)
    return {"rel_fro": fro, "col_ratio": float(np.max(col)), "finite": bool(np.all(np.isfinite(g)))}


def assert_bf16_parity(gpu, ref, name: str = "") -> dict:
    e = errors(gpu, ref)
    assert e["finite"], f"{name}: non-finite values"
    assert e["rel_fro"] <= BF16_REL_FRO, f"{name}: rel Frobenius {e['rel_fro']:.3e} > {BF16_REL_FRO}"
    assert e["col_ratio"] <= BF16_COL_MAXABS, f"{name}: column max-abs/RMS {e['col_ratio']:.3e} > {BF16_COL_MAXABS}"
    return e


def assert_f32_parity(gpu, ref, name: str = "") -> dict:
    e = errors(gpu, ref)
    assert e["finite"], f"{name}: non-finite values"
    assert e["rel_fro"] <= F32_REL_FRO, f"{name}: rel Frobenius {e['rel_fro']:.3e} > {F32_REL_FRO}"
    return e


# Stored intermediates (the saved pre-activation Y, the activation A, attention's
# Q/K/V and O) are fp32-accumulated values rounded once to bf16.  Round-to-nearest
# puts each within half a bf16 spacing, i.e. within 2^-8 of its magnitude; the
# criterion allows one spacing (2^-8 |x|) plus 1e-4 of the tensor RMS for the fp32
# accumulation.  It is element-wise, so it is stricter than the column criterion
# everywhere except in heavy-tailed columns, where output rounding alone can
# exceed 2e-2 x RMS.
ROUNDED_REL = 2.0 ** -8
ROUNDED_ABS_RMS = 1e-4


def assert_bf16_rounded(gpu, ref, name: str = "", rel: float = ROUNDED_REL, abs_rms: float = ROUNDED_ABS_RMS) -> dict:
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, f"{name}: shape {g.shape} != {r.shape}"
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    rms = float(np.sqrt(np.mean(r * r)))
    bound = rel * np.abs(r) + abs_rms * rms
    excess = np.abs(g - r) / bound
    worst = float(np.max(excess))
    assert worst <= 1.0, f"{name}: element error {worst:.3f} x the one-ulp bound (at {np.unravel_index(np.argmax(excess), g.shape)})"
    return {"worst": worst, **errors(g, r)}
