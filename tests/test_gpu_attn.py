"""Self-attention block (and the attention+MLP layer) on the GPU against the fp64 oracle."""
import numpy as np
import pytest
import torch

import tensor_transformer_block_gb300 as tp
from oracle import tp_oracle as O
from parity import assert_attn_parity, assert_bf16_rounded
from tensor_transformer_block_gb300 import block, inputs

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _attn(B, S, h, H, d, N, causal=True, backward=True, seed=0):
    inp = inputs.attn_inputs(B, S, h, H, d, N, seed=seed, backward=backward)
    dev = {k: v.cuda() for k, v in inp.items()}
    f = block.attn_forward(dev["X"], dev["Wqkv"], dev["Wo"], B, S, causal)
    g = None
    if backward:
        g = block.attn_backward(dev["X"], dev["Wqkv"], dev["Wo"], f["QKV"], f["O"], f["LSE"], dev["dZ"], B, S, causal)
    torch.cuda.synchronize()
    assert tp.tp_sync_status() == 0
    return inp, {k: _np(v) for k, v in inp.items()}, f, g


def _check_qkv(qkv_gpu, qkv_ref, N, T, hN, d):
    """Q, K and V are stored in fp16: each a single rounding of the fp32 projection
    (at most 2^-11 of the value, held to 2^-10)."""
    g = qkv_gpu.detach().reshape(N, T, 3, hN, d)
    qkv = g.contiguous().view(torch.float16).to("cpu", torch.float64).numpy()
    r = qkv_ref.reshape(N, T, 3, hN, d)
    assert_bf16_rounded(qkv, r, "Q, K, V (fp16)", rel=2.0 ** -10)


def _check(B, S, h, H, d, N, causal=True, backward=True, seed=0):
    inp, r, f, g = _attn(B, S, h, H, d, N, causal, backward, seed)
    ref = O.attention_forward(r["X"], r["Wqkv"], r["Wo"], B, S, causal)
    _check_qkv(f["QKV"], ref["QKV"], N, B * S, H // N, d)
    assert_attn_parity(_np(f["O"]), ref["O"], "O")
    assert_attn_parity(_np(f["LSE"]).reshape(B * H, S), ref["LSE"].reshape(B * H, S), "LSE")
    assert_attn_parity(_np(f["Z"]), ref["Z"], "Z")
    if backward:
        gr = O.attention_backward(r["X"], r["Wqkv"], r["Wo"], r["dZ"], B, S, causal)
        assert_attn_parity(_np(g["dX"]), gr["dX"], "dX")
        assert_attn_parity(_np(g["dWqkv"]).reshape(N, h, -1), gr["dWqkv"].reshape(N, h, -1), "dWqkv")
        assert_attn_parity(_np(g["dWo"]), gr["dWo"], "dWo")


@pytest.mark.parametrize("B,S,h,H,d,N,causal", [
    (2, 256, 256, 4, 64, 2, True),      # two full 128 blocks, d = 64
    (1, 384, 512, 4, 128, 4, True),     # three blocks, d = 128, one head per shard
    (2, 200, 256, 4, 64, 4, True),      # ragged sequence (200 = 128 + 72)
    (1, 130, 512, 8, 64, 2, True),      # a 2-token tail block
    (2, 256, 512, 4, 128, 2, False),    # no mask
    (1, 1, 128, 2, 64, 1, True),        # one token
    (1, 77, 384, 6, 64, 3, False),      # single ragged block, no mask, N = 3
])
def test_attention_block_fwd_bwd(B, S, h, H, d, N, causal):
    _check(B, S, h, H, d, N, causal, True, seed=S + H)


def test_attention_block_full_config_forward():
    """The attention workload at full size: B=2, S=2048, h=4096, 32 heads of 128, N=8."""
    _check(2, 2048, 4096, 32, 128, 8, True, backward=False)


def test_attention_block_h4096_backward_reduced_seq():
    """Backward at the attention workload's widths (h=4096, 32 heads, N=8) with S=512."""
    _check(1, 512, 4096, 32, 128, 8, True, backward=True, seed=5)


def test_attention_head_sharding_invariant():
    """Head-sharded output does not depend on N (the pages' column split by head)."""
    B, S, H, d, h = 1, 256, 8, 64, 512
    base = inputs.attn_inputs(B, S, h, H, d, 1, backward=False)
    Wq = base["Wqkv"][0].reshape(h, 3 * H * d)
    Wo = base["Wo"].reshape(H * d, h)
    zs = []
    for n in (1, 2, 4, 8):
        Wqkv = inputs.split_qkv_heads(Wq, n, H, d).cuda()
        Wos = inputs.split_rows(Wo, n).cuda()
        zs.append(_np(block.attn_forward(base["X"].cuda(), Wqkv, Wos, B, S, True)["Z"]))
    for z in zs[1:]:
        assert_attn_parity(z, zs[0], "Z across N")


def test_attention_rejects_nondividing_shards():
    """32 heads on 5 shards is an error (io.zouht.com 张量并行 §2.2.1)."""
    with pytest.raises(tp.TPError) as e:
        tp.tp_attn_fwd(tp.TP_BF16, 1, 128, 4096, 32, 128, 5, 1, 0, 0, 0, None, None, None, 0, None)
    assert e.value.status == 2


def _layer(B, S, h, H, d, f, N, seed=0):
    inp = inputs.layer_inputs(B, S, h, H, d, f, N, seed=seed)
    dev = {k: v.cuda() for k, v in inp.items()}
    a = block.attn_forward(dev["X"], dev["Wqkv"], dev["Wo"], B, S, True)
    m = block.mlp_forward(a["Z"], dev["W1s"], dev["W2s"])
    gm = block.mlp_backward(a["Z"], dev["W1s"], dev["W2s"], m["Y"], m["A"], dev["dZ"])
    ga = block.attn_backward(dev["X"], dev["Wqkv"], dev["Wo"], a["QKV"], a["O"], a["LSE"], gm["dX"], B, S, True)
    torch.cuda.synchronize()
    assert tp.tp_sync_status() == 0
    return inp, {k: _np(v) for k, v in inp.items()}, a, m, gm, ga


def test_layer_fwd_bwd_reduced():
    """Attention block then MLP block, forward and backward, every output, at
    reduced size (B=1, S=512, h=1024, 8 heads of 128, f=4096, N=8)."""
    B, S, h, H, d, f, N = 1, 512, 1024, 8, 128, 4096, 8
    inp, r, a, m, gm, ga = _layer(B, S, h, H, d, f, N, seed=2)
    ref = O.layer_forward(r["X"], r["Wqkv"], r["Wo"], r["W1s"], r["W2s"], B, S, True)
    assert_attn_parity(_np(m["Z"]), ref["Z"], "Z")
    g = O.layer_backward(r["X"], r["Wqkv"], r["Wo"], r["W1s"], r["W2s"], r["dZ"], B, S, True)
    assert_attn_parity(_np(ga["dX"]), g["dX"], "dX")
    assert_attn_parity(_np(ga["dWqkv"]).reshape(N, h, -1), g["dWqkv"].reshape(N, h, -1), "dWqkv")
    assert_attn_parity(_np(ga["dWo"]), g["dWo"], "dWo")
    assert_attn_parity(_np(gm["dW1s"]), g["dW1s"], "dW1s")
    assert_attn_parity(_np(gm["dW2s"]), g["dW2s"], "dW2s")


def _attn_mlp(B, S, h, H, d, f, N, seed=0, causal=True):
    """The layer through the fused entry points (attention output kept in fp16)."""
    inp = inputs.layer_inputs(B, S, h, H, d, f, N, seed=seed)
    dev = {k: v.cuda() for k, v in inp.items()}
    p = {k: dev[k] for k in ("Wqkv", "Wo", "W1s", "W2s")}
    fw = block.attn_mlp_forward(dev["X"], p, B, S, causal)
    g = block.attn_mlp_backward(dev["X"], p, fw["save"], dev["dZ"], B, S, causal)
    torch.cuda.synchronize()
    assert tp.tp_sync_status() == 0
    out = {"Z": _np(fw["Z"]), **{k: _np(v) for k, v in g.items()}}
    del fw, g, dev, p
    torch.cuda.empty_cache()
    return {k: v.double().numpy() for k, v in inp.items()}, out


def _check_attn_mlp_grads(r, out, g, N, h):
    assert_attn_parity(out["dX"], g["dX"], "dX")
    assert_attn_parity(out["dWqkv"].reshape(N, h, -1), g["dWqkv"].reshape(N, h, -1), "dWqkv")
    assert_attn_parity(out["dWo"], g["dWo"], "dWo")
    assert_attn_parity(out["dW1s"], g["dW1s"], "dW1s")
    assert_attn_parity(out["dW2s"], g["dW2s"], "dW2s")


@pytest.mark.parametrize("B,S,h,H,d,f,N", [
    (1, 512, 1024, 8, 128, 4096, 8),     # the layer's widths scaled down, full 128 blocks
    (2, 200, 256, 4, 64, 528, 2),        # ragged sequence and FFN tails (f/N = 264)
    (1, 130, 384, 6, 64, 768, 3),        # odd shard count, a 2-token tail block
])
def test_attn_mlp_layer_fwd_bwd(B, S, h, H, d, f, N):
    """The fused layer (tp_attn_mlp_fwd / tp_attn_mlp_bwd), every output in full."""
    r, out = _attn_mlp(B, S, h, H, d, f, N, seed=S + f)
    ref = O.layer_forward(r["X"], r["Wqkv"], r["Wo"], r["W1s"], r["W2s"], B, S, True)
    assert_attn_parity(out["Z"], ref["Z"], "Z")
    g = O.layer_backward(r["X"], r["Wqkv"], r["Wo"], r["W1s"], r["W2s"], r["dZ"], B, S, True)
    _check_attn_mlp_grads(r, out, g, N, h)


def test_attn_mlp_layer_full_config():
    """The layer workload at full size (S=4096, h=8192, 64 heads of 128, f=28672,
    N=8) through the fused entry points: the forward output on sampled token rows
    (the oracle's forward restricted to those rows) and every gradient, dX, dWqkv,
    dWo, dW1s and dW2s, in full against the oracle's backward, each within the
    stated 5e-3 relative Frobenius error."""
    B, S, h, H, d, f, N = 1, 4096, 8192, 64, 128, 28672, 8
    r, out = _attn_mlp(B, S, h, H, d, f, N)
    rng = np.random.default_rng(1)
    rows = np.sort(np.concatenate([[0, S - 1], rng.choice(S, 30, replace=False)]))
    att = O.attention_forward_rows(r["X"], r["Wqkv"], r["Wo"], B, S, rows, True)
    assert_attn_parity(out["Z"][rows], O.mlp_forward(att["Z"], r["W1s"], r["W2s"])["Z"], "Z rows")
    g = O.layer_backward(r["X"], r["Wqkv"], r["Wo"], r["W1s"], r["W2s"], r["dZ"], B, S, True)
    _check_attn_mlp_grads(r, out, g, N, h)


@pytest.mark.parametrize("mode", [1, 2])
def test_attention_block_each_tiling(mode):
    """The attention projections (split-residual epilogue, shard-sum output GEMM,
    backward GEMMs) under both GEMM tilings."""
    tp.tp_set_gemm_tiling(mode)
    try:
        _check(2, 256, 512, 8, 64, 4, True, backward=True, seed=mode)
    finally:
        tp.tp_set_gemm_tiling(0)
