"""Gated (SwiGLU) MLP block on the GPU against the fp64 oracle (same seeded inputs)."""
import numpy as np
import pytest
import torch

import tensor_transformer_block_gb300 as tp
from oracle import tp_oracle as O
from parity import assert_bf16_parity, assert_bf16_rounded, bf16_round, storage_col_tol
from tensor_transformer_block_gb300 import block, inputs

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _run(T, h, f, N, backward=True, seed=0, save=True):
    inp = inputs.gmlp_inputs(T, h, f, N, seed=seed, backward=backward)
    dev = {k: v.cuda() for k, v in inp.items()}
    fwd = block.gmlp_forward(dev["X"], dev["Wgus"], dev["Wds"], save=save)
    bwd = None
    if backward:
        bwd = block.gmlp_backward(dev["X"], dev["Wgus"], dev["Wds"], fwd["GU"], fwd["A"], dev["dZ"])
    torch.cuda.synchronize()
    assert tp.tp_sync_status() == 0
    return inp, {k: _np(v) for k, v in inp.items()}, fwd, bwd


def _check(T, h, f, N, backward=True, seed=0):
    inp, r, fwd, bwd = _run(T, h, f, N, backward=backward, seed=seed)
    ref = O.gated_mlp_forward(r["X"], r["Wgus"], r["Wds"])
    # GU and A are fp32-accumulated values rounded once to bf16
    assert_bf16_rounded(_np(fwd["GU"]), ref["GU"], "GU")
    assert_bf16_rounded(_np(fwd["A"]), ref["A"], "A")
    assert_bf16_parity(_np(fwd["Z"]), ref["Z"], "Z")
    if backward:
        # The backward reads the bf16 gate/up it saved and keeps dG, dU in bf16
        # between its products, so its outputs carry those roundings on top of their
        # own.  The column bound is twice what the oracle reaches with the same
        # intermediates rounded to bf16 (at least 2e-2); rel Frobenius stays 5e-3.
        g = O.gated_mlp_backward(r["X"], r["Wgus"], r["Wds"], r["dZ"])
        gs = O.gated_mlp_backward(r["X"], r["Wgus"], r["Wds"], r["dZ"], store=bf16_round)
        as_cols = lambda a: np.transpose(a, (0, 2, 1, 3))  # [N][2][h][f/N]: rows h per column
        assert_bf16_parity(_np(bwd["dX"]), g["dX"], "dX", col_tol=storage_col_tol(gs["dX"], g["dX"]))
        assert_bf16_parity(as_cols(_np(bwd["dWgus"])), as_cols(g["dWgus"]), "dWgus",
                           col_tol=storage_col_tol(as_cols(gs["dWgus"]), as_cols(g["dWgus"])))
        assert_bf16_parity(_np(bwd["dWds"]), g["dWds"], "dWds", col_tol=storage_col_tol(gs["dWds"], g["dWds"]))


def test_gmlp_bf16_small_config():
    """T=2048, h=1024, f=4096 (gate and up each), N=4, forward + backward, every output."""
    _check(2048, 1024, 4096, 4)


@pytest.mark.parametrize("T,h,f,N", [
    (333, 200, 264, 3),     # f/N = 88: the 128-wide gated tile is ragged inside each part
    (128, 256, 512, 1),     # N = 1
    (384, 128, 2048, 8),    # f/N = 256
    (1, 64, 64, 8),         # one token, f/N = 8
    (200, 520, 1040, 5),    # odd shard count, f/N = 208
    (520, 64, 192, 2),      # K = 64 single block, several M tiles with a tail
])
def test_gmlp_bf16_ragged(T, h, f, N):
    _check(T, h, f, N, seed=T + h)


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("T,h,f,N", [(333, 200, 264, 3), (2048, 1024, 4096, 4), (1, 64, 64, 8)])
def test_gmlp_bf16_each_tiling(mode, T, h, f, N):
    """Both GEMM tilings: in the CTA pair the even CTA stages the gate columns and the
    odd CTA the up columns of the same tile."""
    tp.tp_set_gemm_tiling(mode)
    try:
        _check(T, h, f, N, seed=T + mode)
    finally:
        tp.tp_set_gemm_tiling(0)


def test_gmlp_no_saves_uses_workspace():
    inp = inputs.gmlp_inputs(256, 128, 512, 4, backward=False)
    dev = {k: v.cuda() for k, v in inp.items()}
    a = block.gmlp_forward(dev["X"], dev["Wgus"], dev["Wds"], save=False)["Z"]
    b = block.gmlp_forward(dev["X"], dev["Wgus"], dev["Wds"], save=True)["Z"]
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_gmlp_deterministic():
    inp = inputs.gmlp_inputs(512, 256, 1024, 4)
    dev = {k: v.cuda() for k, v in inp.items()}
    outs = []
    for _ in range(2):
        f = block.gmlp_forward(dev["X"], dev["Wgus"], dev["Wds"])
        g = block.gmlp_backward(dev["X"], dev["Wgus"], dev["Wds"], f["GU"], f["A"], dev["dZ"])
        outs.append([f["Z"].clone(), f["GU"].clone(), g["dX"].clone(), g["dWgus"].clone(), g["dWds"].clone()])
    torch.cuda.synchronize()
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_gmlp_shard_sum_matches_unsharded_gpu():
    """The same gate/up/down weights cut into N = 1, 2, 4, 8 shards give the same Z."""
    T, h, f = 256, 256, 2048
    base = inputs.gmlp_inputs(T, h, f, 1, backward=False)
    Wg = base["Wgus"][0, :, 0, :]
    Wu = base["Wgus"][0, :, 1, :]
    Wd = base["Wds"].reshape(f, h)
    zs = []
    for n in (1, 2, 4, 8):
        Wgus = torch.stack([inputs.split_columns(Wg, n), inputs.split_columns(Wu, n)], dim=2).contiguous().cuda()
        zs.append(_np(block.gmlp_forward(base["X"].cuda(), Wgus, inputs.split_rows(Wd, n).cuda())["Z"]))
    for z in zs[1:]:
        assert_bf16_parity(z, zs[0], "Z across N")


def test_gmlp_full_size_sampled():
    """The gated workload at full size (T=8192, h=4096, f=12288, N=8): Z and dX on
    sampled token rows, the weight gradients on sampled FFN columns."""
    T, h, f, N = 8192, 4096, 12288, 8
    inp, r, fwd, bwd = _run(T, h, f, N)
    rng = np.random.default_rng(0)
    rows = np.sort(np.concatenate([[0, T - 1], rng.choice(T, 30, replace=False)]))
    ref = O.gated_mlp_forward(r["X"][rows], r["Wgus"], r["Wds"])
    assert_bf16_parity(_np(fwd["Z"])[rows], ref["Z"], "Z rows")
    g = O.gated_mlp_backward(r["X"][rows], r["Wgus"], r["Wds"], r["dZ"][rows])
    gs = O.gated_mlp_backward(r["X"][rows], r["Wgus"], r["Wds"], r["dZ"][rows], store=bf16_round)
    assert_bf16_parity(_np(bwd["dX"])[rows], g["dX"], "dX rows", col_tol=storage_col_tol(gs["dX"], g["dX"]))
    cols = np.sort(np.concatenate([[0, f - 1], rng.choice(f, 30, replace=False)]))
    gc = O.gated_mlp_backward_weight_columns(r["X"], r["Wgus"], r["Wds"], r["dZ"], cols)
    gcs = O.gated_mlp_backward_weight_columns(r["X"], r["Wgus"], r["Wds"], r["dZ"], cols, store=bf16_round)
    fN = f // N
    dWgu = _np(bwd["dWgus"])
    dWd = _np(bwd["dWds"])
    got = {"dWg_cols": np.stack([dWgu[c // fN, :, 0, c % fN] for c in cols], axis=1),
           "dWu_cols": np.stack([dWgu[c // fN, :, 1, c % fN] for c in cols], axis=1),
           "dWd_rows": np.stack([dWd[c // fN, c % fN, :] for c in cols], axis=0)}
    for k, v in got.items():
        assert_bf16_parity(v, gc[k], k, col_tol=storage_col_tol(gcs[k], gc[k]))

