"""The pre-norm layer in the tensor + sequence parallel form on the GPU."""
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


def _both(B, S, h, H, d, f, N, seed=0):
    inp = inputs.prenorm_inputs(B, S, h, H, d, f, N, seed=seed)
    dev = {k: v.cuda() for k, v in inp.items()}
    tpf = block.prenorm_layer_forward(dev["X"], dev, B, S)
    tpb_ = block.prenorm_layer_backward(dev["X"], dev, tpf["save"], dev["dZ"], B, S)
    Xs = inputs.to_seq_shards(dev["X"], B, S, N)
    dZs = inputs.to_seq_shards(dev["dZ"], B, S, N)
    spf = block.prenorm_layer_forward(Xs, dev, B, S, seq_sharded=True)
    spb = block.prenorm_layer_backward(Xs, dev, spf["save"], dZs, B, S, seq_sharded=True)
    torch.cuda.synchronize()
    assert tp.tp_sync_status() == 0
    return inp, tpf, tpb_, spf, spb


@pytest.mark.parametrize("B,S,h,H,d,f,N", [
    (2, 256, 512, 4, 128, 1024, 2),    # two sequences, 2 shards of 128 positions
    (3, 512, 256, 8, 64, 512, 4),      # three sequences, 4 shards
    (1, 1024, 512, 8, 64, 1024, 8),    # one sequence: the shard layout is the token order
])
def test_sp_layer_matches_tp_layer_bit_for_bit(B, S, h, H, d, f, N):
    """Every GEMM of the sequence-parallel form reads the same values in the same
    order as the plain form (the all-gather and reduce-scatter are addressing), and
    LayerNorm works row by row: Z, dX and the weight gradients are bit-identical
    once the layouts are matched.  dgamma / dbeta sum their rows in storage order,
    so they agree to fp32 rounding before the bf16 rounding."""
    inp, tpf, tpb_, spf, spb = _both(B, S, h, H, d, f, N, seed=S + N)
    assert torch.equal(inputs.from_seq_shards(spf["Z"]), tpf["Z"])
    assert torch.equal(inputs.from_seq_shards(spb["dX"]), tpb_["dX"])
    for k in ("dWqkv", "dWo", "dW1s", "dW2s"):
        assert torch.equal(spb[k], tpb_[k]), k
    for k in ("dln1_g", "dln1_b", "dln2_g", "dln2_b"):
        assert_bf16_rounded(_np(spb[k]), _np(tpb_[k]), k, rel=2.0 ** -7, abs_rms=1e-3)


def test_sp_layer_against_oracle():
    """The sequence-parallel form against the oracle's step-by-step restatement."""
    B, S, h, H, d, f, N = 2, 256, 1024, 8, 128, 4096, 2
    inp, tpf, tpb_, spf, spb = _both(B, S, h, H, d, f, N, seed=3)
    r = {k: _np(v) for k, v in inp.items()}
    args = (r["ln1_g"], r["ln1_b"], r["Wqkv"], r["Wo"], r["ln2_g"], r["ln2_b"], r["W1s"], r["W2s"])
    Xs = O.to_seq_shards(r["X"], B, S, N)
    ref = O.sp_prenorm_layer_forward(Xs, *args, B, S)
    assert_attn_parity(_np(spf["Z"]).reshape(N * B * (S // N), h), ref["Z"].reshape(-1, h), "Z (sequence shards)")
    g = O.sp_prenorm_layer_backward(Xs, *args, O.to_seq_shards(r["dZ"], B, S, N), B, S)
    assert_attn_parity(_np(spb["dX"]).reshape(-1, h), g["dX"].reshape(-1, h), "dX (sequence shards)")
    for k in ("dW1s", "dW2s", "dWo"):
        assert_attn_parity(_np(spb[k]), g[k], k)
    assert_attn_parity(_np(spb["dWqkv"]).reshape(N, h, -1), g["dWqkv"].reshape(N, h, -1), "dWqkv")
