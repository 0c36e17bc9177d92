"""LayerNorm (+ residual gradient) and the pre-norm layer on the GPU against the fp64 oracle."""
import numpy as np
import pytest
import torch

import tensor_transformer_block_gb300 as tp
from oracle import tp_oracle as O
from parity import assert_attn_parity, assert_bf16_rounded, assert_f32_parity
from tensor_transformer_block_gb300 import block, inputs

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


@pytest.mark.parametrize("T,h,x_mean", [
    (333, 200, 0.0),      # ragged: 25 vectors per row, one partial warp
    (1, 8, 0.0),          # one row of one vector
    (4096, 8192, 0.0),    # the layer workload's rows
    (640, 8192, 40.0),    # rows with a large common offset: centring must not cancel
    (77, 8200, 0.0),      # two vectors per thread, ragged
    (96, 16384, 0.0),     # the largest row
])
def test_layernorm_fwd_bwd(T, h, x_mean):
    inp = inputs.ln_inputs(T, h, seed=T + h, x_mean=x_mean)
    d = {k: v.cuda() for k, v in inp.items()}
    f = block.layernorm_forward(d["X"], d["gamma"], d["beta"])
    g = block.layernorm_backward(d["X"], d["gamma"], f["mean"], f["rstd"], d["dY"], d["dR"])
    g0 = block.layernorm_backward(d["X"], d["gamma"], f["mean"], f["rstd"], d["dY"], None)
    torch.cuda.synchronize()
    assert tp.tp_sync_status() == 0
    r = {k: _np(v) for k, v in inp.items()}
    ref = O.layer_norm(r["X"], r["gamma"], r["beta"])
    # one rounding of an fp32 evaluation: Y within a bf16 spacing; statistics fp32
    assert_bf16_rounded(_np(f["Y"]), ref["y"], "Y")
    # fp32 mean of h bf16 values: within 1e-5 of the row's scale (|offset| + 1)
    assert np.max(np.abs(_np(f["mean"]) - ref["mean"])) <= 1e-5 * (abs(x_mean) + 1.0)
    assert_f32_parity(_np(f["rstd"]), ref["rstd"], "rstd")
    gb = O.layer_norm_backward(r["X"], r["gamma"], r["dY"])
    assert_bf16_rounded(_np(g["dX"]), gb["dx"] + r["dR"], "dX + dR")
    assert_bf16_rounded(_np(g0["dX"]), gb["dx"], "dX")
    assert_bf16_rounded(_np(g["dgamma"]), gb["dgamma"], "dgamma")
    assert_bf16_rounded(_np(g["dbeta"]), gb["dbeta"], "dbeta")
    assert torch.equal(g["dgamma"], g0["dgamma"]) and torch.equal(g["dbeta"], g0["dbeta"])


def test_layernorm_deterministic():
    inp = inputs.ln_inputs(1000, 4096, seed=3)
    d = {k: v.cuda() for k, v in inp.items()}
    f = block.layernorm_forward(d["X"], d["gamma"], d["beta"])
    a = block.layernorm_backward(d["X"], d["gamma"], f["mean"], f["rstd"], d["dY"], d["dR"])
    b = block.layernorm_backward(d["X"], d["gamma"], f["mean"], f["rstd"], d["dY"], d["dR"])
    torch.cuda.synchronize()
    for k in a:
        assert torch.equal(a[k], b[k]), k


def _layer(B, S, h, H, d, f, N, seed=0, zero_out=False):
    inp = inputs.prenorm_inputs(B, S, h, H, d, f, N, seed=seed)
    if zero_out:
        inp["Wo"] = torch.zeros_like(inp["Wo"])
        inp["W2s"] = torch.zeros_like(inp["W2s"])
    dev = {k: v.cuda() for k, v in inp.items()}
    fw = block.prenorm_layer_forward(dev["X"], dev, B, S)
    bw = block.prenorm_layer_backward(dev["X"], dev, fw["save"], dev["dZ"], B, S)
    torch.cuda.synchronize()
    assert tp.tp_sync_status() == 0
    return inp, {k: _np(v) for k, v in inp.items()}, fw, bw


def _args(r):
    return (r["X"], r["ln1_g"], r["ln1_b"], r["Wqkv"], r["Wo"], r["ln2_g"], r["ln2_b"], r["W1s"], r["W2s"])


def test_prenorm_layer_reduced():
    """LN1 -> attention (+X) -> LN2 -> MLP (+H1), forward and every gradient, at
    reduced size (B=2, S=256, h=1024, 8 heads of 128, f=4096, N=8)."""
    B, S, h, H, d, f, N = 2, 256, 1024, 8, 128, 4096, 8
    inp, r, fw, bw = _layer(B, S, h, H, d, f, N, seed=4)
    ref = O.prenorm_layer_forward(*_args(r), B, S)
    assert_attn_parity(_np(fw["Z"]), ref["Z"], "Z")
    g = O.prenorm_layer_backward(*_args(r), r["dZ"], B, S)
    assert_attn_parity(_np(bw["dX"]), g["dX"], "dX")
    assert_attn_parity(_np(bw["dWqkv"]).reshape(N, h, -1), g["dWqkv"].reshape(N, h, -1), "dWqkv")
    for k in ("dWo", "dW1s", "dW2s"):
        assert_attn_parity(_np(bw[k]), g[k], k)
    for k in ("dln1_g", "dln1_b", "dln2_g", "dln2_b"):
        assert_attn_parity(_np(bw[k])[None, :], g[k][None, :], k)


def test_prenorm_layer_zero_projections_is_identity():
    """With Wo = 0 and W2 = 0 both blocks add exactly zero: Z = X bit for bit (the
    residual epilogues add a zero accumulator to a bf16 value), and dX = dZ.  The
    residual gradient dH1 passes through fp16 storage between the two LayerNorm
    backwards, which holds every bf16 value of magnitude 2^-14 .. 65504 exactly:
    there dX = dZ bit for bit; below 2^-14 fp16 is subnormal and the value moves
    by at most half its spacing, 2^-25."""
    B, S, h, H, d, f, N = 1, 200, 512, 4, 64, 1024, 4
    inp, r, fw, bw = _layer(B, S, h, H, d, f, N, seed=6, zero_out=True)
    assert torch.equal(fw["Z"].cpu(), inp["X"])
    dx, dz = bw["dX"].cpu().double(), inp["dZ"].double()
    normal = dz.abs() >= 2.0 ** -14
    assert torch.equal(dx[normal], dz[normal])
    assert float((dx - dz).abs().max()) <= 2.0 ** -25


@pytest.mark.parametrize("mode", [1, 2])
def test_prenorm_layer_each_tiling(mode):
    tp.tp_set_gemm_tiling(mode)
    try:
        B, S, h, H, d, f, N = 1, 130, 256, 4, 64, 512, 2
        inp, r, fw, bw = _layer(B, S, h, H, d, f, N, seed=mode)
        ref = O.prenorm_layer_forward(*_args(r), B, S)
        assert_attn_parity(_np(fw["Z"]), ref["Z"], "Z")
        g = O.prenorm_layer_backward(*_args(r), r["dZ"], B, S)
        assert_attn_parity(_np(bw["dX"]), g["dX"], "dX")
        assert_attn_parity(_np(bw["dW1s"]), g["dW1s"], "dW1s")
    finally:
        tp.tp_set_gemm_tiling(0)


def test_prenorm_layer_full_size():
    """The pre-norm layer at the full layer size (S=4096, h=8192, 64 heads, f=28672,
    N=8): Z on sampled token rows (the oracle's forward restricted to them) and every
    gradient in full against the oracle's backward, each within the stated 5e-3
    relative Frobenius error."""
    B, S, h, H, d, f, N = 1, 4096, 8192, 64, 128, 28672, 8
    inp, r, fw, bw = _layer(B, S, h, H, d, f, N)
    z = _np(fw["Z"])
    out = {k: _np(v) for k, v in bw.items()}
    del fw, bw
    torch.cuda.empty_cache()
    rng = np.random.default_rng(2)
    rows = np.sort(np.concatenate([[0, S - 1], rng.choice(S, 30, replace=False)]))
    ref = O.prenorm_layer_forward_rows(*_args(r), B, S, rows)
    assert_attn_parity(z[rows], ref["Z"], "Z rows")
    g = O.prenorm_layer_backward(*_args(r), r["dZ"], B, S)
    assert_attn_parity(out["dX"], g["dX"], "dX")
    assert_attn_parity(out["dWqkv"].reshape(N, h, -1), g["dWqkv"].reshape(N, h, -1), "dWqkv")
    for k in ("dWo", "dW1s", "dW2s"):
        assert_attn_parity(out[k], g[k], k)
    for k in ("dln1_g", "dln1_b", "dln2_g", "dln2_b"):
        assert_attn_parity(out[k][None, :], g[k][None, :], k)
