"""Grouped-query attention block on the GPU against the fp64 oracle."""
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


def _run(B, S, h, H, Hkv, d, N, causal=True, backward=True, seed=0):
    inp = inputs.gqa_inputs(B, S, h, H, Hkv, d, N, seed=seed, backward=backward)
    dev = {k: v.cuda() for k, v in inp.items()}
    f = block.gqa_forward(dev["X"], dev["Wqkv"], dev["Wo"], H, Hkv, d, B, S, causal)
    g = None
    if backward:
        g = block.gqa_backward(dev["X"], dev["Wqkv"], dev["Wo"], f["QKV"], f["O"], f["LSE"], dev["dZ"], H, Hkv, d, B,
                               S, causal)
    torch.cuda.synchronize()
    assert tp.tp_sync_status() == 0
    return inp, {k: _np(v) for k, v in inp.items()}, f, g


def _check(B, S, h, H, Hkv, d, N, causal=True, backward=True, seed=0):
    inp, r, f, g = _run(B, S, h, H, Hkv, d, N, causal, backward, seed)
    ref = O.gqa_attention_forward(r["X"], r["Wqkv"], r["Wo"], B, S, H, Hkv, causal)
    # Q, K and V planes (fp16): single roundings of the projection
    T, hn, kvn = B * S, H // N, Hkv // N
    qkv = f["QKV"].detach().reshape(N, T, -1)
    for i in range(N):
        q = ref["Q"][:, i * hn * d:(i + 1) * hn * d]
        k = ref["K"][:, i * kvn * d:(i + 1) * kvn * d]
        v = ref["V"][:, i * kvn * d:(i + 1) * kvn * d]
        row = qkv[i]
        as16 = lambda t: t.contiguous().view(torch.float16).to("cpu", torch.float64).numpy()
        assert_bf16_rounded(as16(row[:, :hn * d]), q, "Q (fp16)", rel=2.0 ** -10)
        assert_bf16_rounded(as16(row[:, hn * d:(hn + kvn) * d]), k, "K (fp16)", rel=2.0 ** -10)
        assert_bf16_rounded(as16(row[:, (hn + kvn) * d:]), v, "V (fp16)", rel=2.0 ** -10)
    assert_attn_parity(_np(f["O"]), ref["O"], "O")
    assert_attn_parity(_np(f["LSE"]).reshape(B * H, S), ref["LSE"].reshape(B * H, S), "LSE")
    assert_attn_parity(_np(f["Z"]), ref["Z"], "Z")
    if backward:
        gr = O.gqa_attention_backward(r["X"], r["Wqkv"], r["Wo"], r["dZ"], B, S, H, Hkv, causal)
        assert_attn_parity(_np(g["dX"]), gr["dX"], "dX")
        assert_attn_parity(_np(g["dWqkv"]), gr["dWqkv"], "dWqkv")
        assert_attn_parity(_np(g["dWo"]), gr["dWo"], "dWo")


@pytest.mark.parametrize("B,S,h,H,Hkv,d,N,causal", [
    (2, 256, 256, 8, 2, 64, 2, True),      # groups of 4, one key/value head per shard
    (1, 384, 512, 8, 4, 128, 4, True),     # groups of 2, d = 128
    (2, 200, 256, 8, 2, 64, 2, True),      # ragged sequence
    (1, 130, 512, 16, 2, 64, 2, False),    # groups of 8, no mask, 2-token tail
    (1, 77, 384, 6, 3, 64, 3, True),       # N = 3, groups of 2
    (1, 1, 128, 4, 1, 64, 1, True),        # one token; one key/value head for all (multi-query)
])
def test_gqa_block_fwd_bwd(B, S, h, H, Hkv, d, N, causal):
    _check(B, S, h, H, Hkv, d, N, causal, True, seed=S + H + Hkv)


def test_gqa_with_hkv_equal_h_is_the_mha_block():
    """Hkv = H runs the multi-head block: the same bytes in, bit-identical results out."""
    B, S, h, H, d, N = 1, 256, 512, 4, 128, 2
    inp = inputs.attn_inputs(B, S, h, H, d, N, seed=9)
    dev = {k: v.cuda() for k, v in inp.items()}
    Wg = dev["Wqkv"].reshape(N, h, 3 * (H // N) * d)
    a = block.attn_forward(dev["X"], dev["Wqkv"], dev["Wo"], B, S, True)
    g = block.gqa_forward(dev["X"], Wg, dev["Wo"], H, H, d, B, S, True)
    ga = block.attn_backward(dev["X"], dev["Wqkv"], dev["Wo"], a["QKV"], a["O"], a["LSE"], dev["dZ"], B, S, True)
    gg = block.gqa_backward(dev["X"], Wg, dev["Wo"], g["QKV"], g["O"], g["LSE"], dev["dZ"], H, H, d, B, S, True)
    torch.cuda.synchronize()
    for k in ("Z", "QKV", "O", "LSE"):
        assert torch.equal(a[k].reshape(-1), g[k].reshape(-1)), k
    for k in ("dX", "dWo"):
        assert torch.equal(ga[k], gg[k]), k
    assert torch.equal(ga["dWqkv"].reshape(-1), gg["dWqkv"].reshape(-1))


def test_gqa_full_size_forward():
    """The grouped workload at full size: B=2, S=2048, h=4096, 32 query heads over
    8 key/value heads of 128, N=8."""
    _check(2, 2048, 4096, 32, 8, 128, 8, True, backward=False)


def test_gqa_h4096_backward_reduced_seq():
    _check(1, 512, 4096, 32, 8, 128, 8, True, backward=True, seed=5)
