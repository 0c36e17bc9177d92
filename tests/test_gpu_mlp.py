"""MLP block on the GPU against the fp64 oracle (same seeded inputs)."""
import numpy as np
import pytest
import torch

from oracle import tp_oracle as O
from parity import assert_bf16_parity, assert_bf16_rounded, assert_f32_parity
from tensor_transformer_block_gb300 import block, inputs

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _run(T, h, f, N, dtype="bf16", backward=True, seed=0, save=True):
    inp = inputs.mlp_inputs(T, h, f, N, dtype=dtype, seed=seed, backward=backward)
    dev = {k: v.cuda() for k, v in inp.items()}
    fwd = block.mlp_forward(dev["X"], dev["W1s"], dev["W2s"], save=save)
    bwd = None
    if backward:
        bwd = block.mlp_backward(dev["X"], dev["W1s"], dev["W2s"], fwd["Y"], fwd["A"], dev["dZ"])
    torch.cuda.synchronize()
    import tensor_transformer_block_gb300 as tp
    assert tp.tp_sync_status() == 0
    ref_in = {k: _np(v) for k, v in inp.items()}
    return inp, ref_in, fwd, bwd


def _check_mlp(T, h, f, N, backward=True, seed=0):
    inp, r, fwd, bwd = _run(T, h, f, N, backward=backward, seed=seed)
    ref = O.mlp_forward(r["X"], r["W1s"], r["W2s"])
    out = {"Y": assert_bf16_rounded(_np(fwd["Y"]), ref["Y"], "Y"),
           "A": assert_bf16_rounded(_np(fwd["A"]), ref["A"], "A"),
           "Z": assert_bf16_parity(_np(fwd["Z"]), ref["Z"], "Z")}
    if backward:
        g = O.mlp_backward(r["X"], r["W1s"], r["W2s"], r["dZ"])
        for k in ("dX", "dW1s", "dW2s"):
            out[k] = assert_bf16_parity(_np(bwd[k]), g[k], k)
    return out


def test_mlp_f32_forward_full_config():
    """fp32 workload: T=64, h=256, f=1024, N=2, forward only, rel Frobenius <= 1e-5."""
    inp, r, fwd, _ = _run(64, 256, 1024, 2, dtype="f32", backward=False)
    ref = O.mlp_forward(r["X"], r["W1s"], r["W2s"])
    assert_f32_parity(_np(fwd["Z"]), ref["Z"], "Z")
    assert_f32_parity(_np(fwd["Y"]), ref["Y"], "Y")
    assert_f32_parity(_np(fwd["A"]), ref["A"], "A")


@pytest.mark.parametrize("T,h,f,N", [
    (77, 40, 96, 3),      # K split over 2 (fc1) and 4 (fc2, one CTA of the cluster idle) CTAs
    (130, 264, 520, 5),   # ragged tiles, K split over 8
    (1, 8, 16, 2),        # one K slice: no split
    (1024, 512, 4096, 2), # fc1 enough tiles for every SM: no split; fc2 split over 2
])
def test_mlp_f32_forward_ragged(T, h, f, N):
    inp, r, fwd, _ = _run(T, h, f, N, dtype="f32", backward=False, seed=3)
    ref = O.mlp_forward(r["X"], r["W1s"], r["W2s"])
    assert_f32_parity(_np(fwd["Z"]), ref["Z"], "Z")


def test_mlp_bf16_full_config_small():
    """bf16 workload T=2048, h=1024, f=4096, N=4, forward + backward, every output."""
    _check_mlp(2048, 1024, 4096, 4)


@pytest.mark.parametrize("T,h,f,N", [
    (333, 200, 264, 3),     # ragged in every GEMM dimension, several tiles
    (128, 256, 512, 1),     # N = 1: no split at all
    (384, 128, 2048, 8),    # N = 8, f/N = 256
    (1, 64, 64, 8),         # one token, f/N = 8
    (200, 520, 1040, 5),    # odd shard count, f/N = 208
    (520, 64, 192, 2),      # K = 64 single block, several M tiles with a tail
])
def test_mlp_bf16_ragged(T, h, f, N):
    _check_mlp(T, h, f, N, seed=T + h)


def test_mlp_bf16_no_saves_uses_workspace():
    inp = inputs.mlp_inputs(256, 128, 512, 4, backward=False)
    dev = {k: v.cuda() for k, v in inp.items()}
    a = block.mlp_forward(dev["X"], dev["W1s"], dev["W2s"], save=False)["Z"]
    b = block.mlp_forward(dev["X"], dev["W1s"], dev["W2s"], save=True)["Z"]
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_mlp_bf16_deterministic():
    inp = inputs.mlp_inputs(512, 256, 1024, 4)
    dev = {k: v.cuda() for k, v in inp.items()}
    outs = []
    for _ in range(2):
        f = block.mlp_forward(dev["X"], dev["W1s"], dev["W2s"])
        g = block.mlp_backward(dev["X"], dev["W1s"], dev["W2s"], f["Y"], f["A"], dev["dZ"])
        outs.append([f["Z"].clone(), g["dX"].clone(), g["dW1s"].clone(), g["dW2s"].clone()])
    torch.cuda.synchronize()
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_mlp_shard_sum_matches_unsharded_gpu():
    """The row-parallel shard sum is the pages' all-reduce: the same inputs cut into
    N = 1, 2, 4, 8 shards give the same Z up to rounding."""
    base = inputs.mlp_inputs(256, 256, 2048, 1, backward=False)
    W1 = base["W1s"][0]
    W2 = base["W2s"].reshape(2048, 256)
    zs = []
    for n in (1, 2, 4, 8):
        W1s = inputs.split_columns(W1, n).cuda()
        W2s = inputs.split_rows(W2, n).cuda()
        zs.append(_np(block.mlp_forward(base["X"].cuda(), W1s, W2s)["Z"]))
    for z in zs[1:]:
        assert_bf16_parity(z, zs[0], "Z across N")


def test_mlp_bf16_h4096_sampled():
    """The h=4096 workload (T=8192, f=16384, N=8) at full size, checked on sampled
    token rows (Z, dX) and sampled FFN columns (dW1, dW2)."""
    T, h, f, N = 8192, 4096, 16384, 8
    inp, r, fwd, bwd = _run(T, h, f, N)
    rng = np.random.default_rng(0)
    rows = np.sort(np.concatenate([[0, T - 1], rng.choice(T, 30, replace=False)]))
    ref = O.mlp_forward(r["X"][rows], r["W1s"], r["W2s"])
    assert_bf16_parity(_np(fwd["Z"])[rows], ref["Z"], "Z rows")
    g = O.mlp_backward(r["X"][rows], r["W1s"], r["W2s"], r["dZ"][rows])
    assert_bf16_parity(_np(bwd["dX"])[rows], g["dX"], "dX rows")
    cols = np.sort(np.concatenate([[0, f - 1], rng.choice(f, 30, replace=False)]))
    gc = O.mlp_backward_weight_columns(r["X"], r["W1s"], r["W2s"], r["dZ"], cols)
    fN = f // N
    dW1 = _np(bwd["dW1s"])
    dW2 = _np(bwd["dW2s"])
    got1 = np.stack([dW1[c // fN, :, c % fN] for c in cols], axis=1)
    got2 = np.stack([dW2[c // fN, c % fN, :] for c in cols], axis=0)
    assert_bf16_parity(got1, gc["dW1_cols"], "dW1 cols")
    assert_bf16_parity(got2, gc["dW2_rows"], "dW2 rows")


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("T,h,f,N", [(333, 200, 264, 3), (2048, 1024, 4096, 4), (600, 520, 1040, 5), (1, 64, 64, 8)])
def test_mlp_bf16_each_tiling(mode, T, h, f, N):
    """Both GEMM tilings (one CTA per 128x256 tile; a CTA pair per 256x256 tile,
    cta_group::2) against the oracle, including tails in M, N and K."""
    import tensor_transformer_block_gb300 as tp
    tp.tp_set_gemm_tiling(mode)
    try:
        _check_mlp(T, h, f, N, seed=T + mode)
    finally:
        tp.tp_set_gemm_tiling(0)


@pytest.mark.parametrize("T,h,f,N", [(2048, 1024, 4096, 4), (1000, 520, 2048, 2)])
def test_mlp_split_k_row_parallel(T, h, f, N):
    """Row-parallel GEMMs (Z, dX) too small to fill the GPU split their K loop in two
    halves whose fp32 partials a second kernel adds in fixed order: the launch
    counters show the split ran, results match the oracle, and a rerun is
    bit-identical (no order depends on scheduling).  The second shape has a ragged
    last column block (h = 520)."""
    import tensor_transformer_block_gb300 as tp
    inp = inputs.mlp_inputs(T, h, f, N, seed=T + f)
    d = {k: v.cuda() for k, v in inp.items()}
    tp.tp_timing_enable(True)
    try:
        runs = []
        for _ in range(2):
            fw = block.mlp_forward(d["X"], d["W1s"], d["W2s"])
            g = block.mlp_backward(d["X"], d["W1s"], d["W2s"], fw["Y"], fw["A"], d["dZ"])
            runs.append((fw["Z"], g["dX"], g["dW1s"], g["dW2s"]))
        torch.cuda.synchronize()
        rep = tp.timing_report()
    finally:
        tp.tp_timing_enable(False)
    assert tp.tp_sync_status() == 0
    assert rep.get("gemm.splitk_reduce", (0, 0))[0] == 4, rep  # Z and dX, twice
    for a, b in zip(*runs):
        assert torch.equal(a, b)
    r = {k: _np(v) for k, v in inp.items()}
    ref = O.mlp_forward(r["X"], r["W1s"], r["W2s"])
    gr = O.mlp_backward(r["X"], r["W1s"], r["W2s"], r["dZ"])
    Z, dX, dW1, dW2 = runs[0]
    assert_bf16_parity(_np(Z), ref["Z"], "Z (split-K)")
    assert_bf16_parity(_np(dX), gr["dX"], "dX (split-K)")
    assert_bf16_parity(_np(dW1), gr["dW1s"], "dW1s")
    assert_bf16_parity(_np(dW2), gr["dW2s"], "dW2s")
