"""Pins for the fp64 oracle: each checks it against something other than itself.

* brute-force pure-Python loops on tiny inputs (no numpy, no BLAS);
* the pages' block-matrix identities, on small-integer matrices where float64
  arithmetic is exact, so that "equal" means bit-equal;
* independent library routines (torch fp64 GeLU, SDPA, autograd);
* closed forms and invariants (softmax rows sum to 1, causal row 0, uniform
  attention when Wq = 0, the odd part of the tanh-GeLU);
* central finite differences of L = <dZ, Z> for every gradient.
"""
import itertools
import math

import numpy as np
import pytest
import torch

from oracle import tp_oracle as O

RNG = np.random.default_rng(1234)


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


# ---------------------------------------------------------------- GEMM core
def brute_matmul(a, b):
    M, K = len(a), len(a[0])
    N = len(b[0])
    out = [[0.0] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s = 0.0
            for k in range(K):
                s += float(a[i][k]) * float(b[k][j])
            out[i][j] = s
    return out


@pytest.mark.parametrize("M,K,N", [(1, 1, 1), (5, 8, 12), (7, 3, 9), (4, 16, 2)])
def test_matmul_vs_triple_loop(M, K, N):
    a = RNG.standard_normal((M, K))
    b = RNG.standard_normal((K, N))
    ref = np.array(brute_matmul(a.tolist(), b.tolist()))
    assert rel(O.matmul(a, b), ref) < 1e-14


def test_matmul_integer_exact():
    a = RNG.integers(-9, 10, (6, 10)).astype(np.float64)
    b = RNG.integers(-9, 10, (10, 7)).astype(np.float64)
    ref = np.array(brute_matmul(a.tolist(), b.tolist()))
    assert np.array_equal(O.matmul(a, b), ref)


# ---------------------------------------------------------------- GeLU
def test_gelu_special_values():
    assert O.gelu_tanh(np.array([0.0]))[0] == 0.0
    big = np.array([10.0, 30.0, 100.0])
    assert np.allclose(O.gelu_tanh(big), big, rtol=0, atol=1e-12)
    assert np.allclose(O.gelu_tanh(-big), 0.0, atol=1e-12)


def test_gelu_odd_part_identity():
    # 0.5x(1+tanh u) - (-0.5x)(1+tanh(-u)) = x for the tanh form, any constants
    x = RNG.standard_normal(1000) * 4
    assert np.allclose(O.gelu_tanh(x) - O.gelu_tanh(-x), x, rtol=0, atol=1e-13)


def test_gelu_scalar_by_hand():
    # written out with math.tanh, one scalar at a time
    for x in [-3.0, -1.0, -0.25, 0.5, 1.0, 2.5]:
        u = math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)
        ref = 0.5 * x * (1.0 + math.tanh(u))
        assert abs(O.gelu_tanh(np.array([x]))[0] - ref) < 1e-15


def test_gelu_vs_torch():
    x = RNG.standard_normal(4096) * 5
    ref = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    assert np.max(np.abs(O.gelu_tanh(x) - ref)) < 1e-14


def test_gelu_is_not_erf_gelu():
    # the tanh form differs from the exact (erf) GeLU by ~1e-4 somewhere
    x = np.linspace(-4, 4, 801)
    erf = torch.nn.functional.gelu(torch.from_numpy(x)).numpy()
    assert np.max(np.abs(O.gelu_tanh(x) - erf)) > 1e-5


def test_gelu_grad_finite_difference_and_autograd():
    x = RNG.standard_normal(512) * 3
    eps = 1e-6
    fd = (O.gelu_tanh(x + eps) - O.gelu_tanh(x - eps)) / (2 * eps)
    assert np.max(np.abs(O.gelu_tanh_grad(x) - fd)) < 1e-8
    t = torch.from_numpy(x.copy()).requires_grad_(True)
    torch.nn.functional.gelu(t, approximate="tanh").sum().backward()
    assert np.max(np.abs(O.gelu_tanh_grad(x) - t.grad.numpy())) < 1e-13


# ---------------------------------------------------------------- split identities
def divisors(n):
    return [k for k in range(1, n + 1) if n % k == 0]


@pytest.mark.parametrize("f", [12, 8])
def test_column_split_concat_exact(f):
    """X [W_0, W_1, ...] = [X W_0, X W_1, ...], bit-exact on integer data, every N | f."""
    T, h = 5, 8
    X = RNG.integers(-5, 6, (T, h)).astype(np.float64)
    W = RNG.integers(-5, 6, (h, f)).astype(np.float64)
    full = np.array(brute_matmul(X.tolist(), W.tolist()))
    for n in divisors(f):
        Ws = np.stack([W[:, i * (f // n):(i + 1) * (f // n)] for i in range(n)])
        assert np.array_equal(O.concat_columns(Ws), W)
        parts = [O.matmul(X, Ws[i]) for i in range(n)]
        assert np.array_equal(np.concatenate(parts, axis=1), full)


@pytest.mark.parametrize("f", [12, 8])
def test_row_split_sum_exact(f):
    """[X_0, X_1, ...][W_0; W_1; ...] = sum_i X_i W_i, bit-exact on integer data."""
    T, h = 5, 7
    A = RNG.integers(-5, 6, (T, f)).astype(np.float64)
    W = RNG.integers(-5, 6, (f, h)).astype(np.float64)
    full = np.array(brute_matmul(A.tolist(), W.tolist()))
    for n in divisors(f):
        c = f // n
        Ws = np.stack([W[i * c:(i + 1) * c, :] for i in range(n)])
        assert np.array_equal(O.stack_rows(Ws), W)
        s = np.zeros((T, h))
        for i in range(n):
            s += O.matmul(A[:, i * c:(i + 1) * c], Ws[i])
        assert np.array_equal(s, full)


def _mlp_inputs(T, h, f, n, seed=0):
    r = np.random.default_rng(seed)
    X = r.standard_normal((T, h))
    W1 = r.standard_normal((h, f)) * 0.3
    W2 = r.standard_normal((f, h)) * 0.3
    dZ = r.standard_normal((T, h))
    W1s = np.stack([W1[:, i * (f // n):(i + 1) * (f // n)] for i in range(n)])
    W2s = np.stack([W2[i * (f // n):(i + 1) * (f // n), :] for i in range(n)])
    return X, W1, W2, W1s, W2s, dZ


def brute_mlp(X, W1, W2):
    T, h = len(X), len(X[0])
    f = len(W1[0])
    Z = [[0.0] * h for _ in range(T)]
    for t in range(T):
        a = []
        for j in range(f):
            y = sum(X[t][k] * W1[k][j] for k in range(h))
            u = math.sqrt(2.0 / math.pi) * (y + 0.044715 * y * y * y)
            a.append(0.5 * y * (1.0 + math.tanh(u)))
        for c in range(h):
            Z[t][c] = sum(a[j] * W2[j][c] for j in range(f))
    return Z


def test_mlp_forward_vs_brute_force():
    X, W1, W2, W1s, W2s, _ = _mlp_inputs(4, 6, 10, 2)
    ref = np.array(brute_mlp(X.tolist(), W1.tolist(), W2.tolist()))
    assert rel(O.mlp_forward(X, W1s, W2s)["Z"], ref) < 1e-13


@pytest.mark.parametrize("n", divisors(12))
def test_mlp_sharded_equals_unsharded_every_n(n):
    X, W1, W2, W1s, W2s, dZ = _mlp_inputs(5, 8, 12, n)
    a = O.mlp_forward(X, W1s, W2s)
    b = O.mlp_forward_sharded(X, W1s, W2s)
    assert rel(b["Z"], a["Z"]) < 1e-13
    assert np.array_equal(b["Y"], a["Y"]) or rel(b["Y"], a["Y"]) < 1e-14
    # Act commutes with the column split: A_i = GeLU(Y_i) is GeLU(Y)'s block i
    assert rel(b["A"], a["A"]) < 1e-14
    # the naive two-all-gather formulation gives the same numbers
    if 8 % n == 0:
        assert rel(O.mlp_forward_two_allgather(X, W1s, W2s), a["Z"]) < 1e-13
    gb = O.mlp_backward_sharded(X, W1s, W2s, dZ)
    ga = O.mlp_backward(X, W1s, W2s, dZ)
    for k in ("dX", "dW1s", "dW2s"):
        assert rel(gb[k], ga[k]) < 1e-13, k


def _loss_mlp(X, W1s, W2s, dZ):
    return float(np.sum(dZ * O.mlp_forward(X, W1s, W2s)["Z"]))


def test_mlp_backward_finite_differences():
    X, _, _, W1s, W2s, dZ = _mlp_inputs(3, 4, 6, 2, seed=7)
    g = O.mlp_backward(X, W1s, W2s, dZ)
    eps = 1e-6
    for name, arr, grad in (("X", X, g["dX"]), ("W1s", W1s, g["dW1s"]), ("W2s", W2s, g["dW2s"])):
        fd = np.zeros_like(arr)
        for idx in itertools.product(*[range(s) for s in arr.shape]):
            old = arr[idx]
            arr[idx] = old + eps
            lp = _loss_mlp(X, W1s, W2s, dZ)
            arr[idx] = old - eps
            lm = _loss_mlp(X, W1s, W2s, dZ)
            arr[idx] = old
            fd[idx] = (lp - lm) / (2 * eps)
        assert rel(grad, fd) < 1e-6, name


def test_mlp_backward_vs_torch_autograd():
    X, W1, W2, W1s, W2s, dZ = _mlp_inputs(6, 8, 16, 4, seed=3)
    tX, tW1, tW2 = (torch.from_numpy(a.copy()).requires_grad_(True) for a in (X, W1, W2))
    Z = torch.nn.functional.gelu(tX @ tW1, approximate="tanh") @ tW2
    (Z * torch.from_numpy(dZ)).sum().backward()
    g = O.mlp_backward(X, W1s, W2s, dZ)
    assert rel(g["dX"], tX.grad.numpy()) < 1e-13
    assert rel(O.concat_columns(g["dW1s"]), tW1.grad.numpy()) < 1e-13
    assert rel(O.stack_rows(g["dW2s"]), tW2.grad.numpy()) < 1e-13


def test_mlp_weight_column_restriction():
    X, _, _, W1s, W2s, dZ = _mlp_inputs(9, 8, 12, 3, seed=5)
    g = O.mlp_backward(X, W1s, W2s, dZ)
    cols = np.array([0, 3, 4, 11])
    r = O.mlp_backward_weight_columns(X, W1s, W2s, dZ, cols)
    assert rel(r["dW1_cols"], O.concat_columns(g["dW1s"])[:, cols]) < 1e-13
    assert rel(r["dW2_rows"], O.stack_rows(g["dW2s"])[cols, :]) < 1e-13


# ---------------------------------------------------------------- attention
def _attn_inputs(B, S, H, d, n, h=None, seed=0, wstd=0.3):
    r = np.random.default_rng(seed)
    h = h or H * d
    X = r.standard_normal((B * S, h))
    Wq, Wk, Wv = (r.standard_normal((h, H * d)) * wstd for _ in range(3))
    Wo = r.standard_normal((H * d, h)) * wstd
    dZ = r.standard_normal((B * S, h))
    Wqkv = O.pack_qkv(Wq, Wk, Wv, n, d)
    Wos = np.stack([Wo[i * (H // n) * d:(i + 1) * (H // n) * d] for i in range(n)])
    return X, Wq, Wk, Wv, Wo, Wqkv, Wos, dZ


def test_qkv_pack_layout():
    B, S, H, d, n = 1, 3, 4, 2, 2
    X, Wq, Wk, Wv, Wo, Wqkv, Wos, _ = _attn_inputs(B, S, H, d, n)
    # shard i, part p, local head jj is global head i*H/n+jj's column block
    for i in range(n):
        for jj in range(H // n):
            j = i * (H // n) + jj
            assert np.array_equal(Wqkv[i, :, 0, jj, :], Wq[:, j * d:(j + 1) * d])
            assert np.array_equal(Wqkv[i, :, 1, jj, :], Wk[:, j * d:(j + 1) * d])
            assert np.array_equal(Wqkv[i, :, 2, jj, :], Wv[:, j * d:(j + 1) * d])
    q, k, v = O.unpack_qkv(Wqkv)
    assert np.array_equal(q, Wq) and np.array_equal(k, Wk) and np.array_equal(v, Wv)


def brute_attention(X, Wq, Wk, Wv, Wo, B, S, H, d, causal):
    T, h = X.shape
    Q, K, V = X @ Wq, X @ Wk, X @ Wv
    Ocat = np.zeros((T, H * d))
    for b in range(B):
        for j in range(H):
            for s in range(S):
                t = b * S + s
                keys = range(s + 1) if causal else range(S)
                sc = []
                for s2 in keys:
                    t2 = b * S + s2
                    sc.append(sum(Q[t, j * d + e] * K[t2, j * d + e] for e in range(d)) / math.sqrt(d))
                m = max(sc)
                w = [math.exp(x - m) for x in sc]
                z = sum(w)
                for e in range(d):
                    Ocat[t, j * d + e] = sum(w[i] / z * V[b * S + s2, j * d + e]
                                             for i, s2 in enumerate(keys))
    return Ocat @ Wo


@pytest.mark.parametrize("causal", [True, False])
def test_attention_vs_brute_force(causal):
    B, S, H, d, n = 2, 5, 4, 3, 2
    X, Wq, Wk, Wv, Wo, Wqkv, Wos, _ = _attn_inputs(B, S, H, d, n)
    ref = brute_attention(X, Wq, Wk, Wv, Wo, B, S, H, d, causal)
    assert rel(O.attention_forward(X, Wqkv, Wos, B, S, causal)["Z"], ref) < 1e-13


@pytest.mark.parametrize("causal", [True, False])
def test_attention_vs_torch_sdpa(causal):
    B, S, H, d, n = 2, 9, 4, 8, 4
    X, Wq, Wk, Wv, Wo, Wqkv, Wos, _ = _attn_inputs(B, S, H, d, n, seed=2)
    t = lambda a: torch.from_numpy(a)
    q = (t(X) @ t(Wq)).reshape(B, S, H, d).transpose(1, 2)
    k = (t(X) @ t(Wk)).reshape(B, S, H, d).transpose(1, 2)
    v = (t(X) @ t(Wv)).reshape(B, S, H, d).transpose(1, 2)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal)
    Z = (o.transpose(1, 2).reshape(B * S, H * d) @ t(Wo)).numpy()
    out = O.attention_forward(X, Wqkv, Wos, B, S, causal)
    assert rel(out["Z"], Z) < 1e-13
    # LSE against torch.logsumexp of the masked scaled scores
    sc = (q @ k.transpose(-1, -2)) / math.sqrt(d)
    if causal:
        sc = sc.masked_fill(~torch.tril(torch.ones(S, S, dtype=torch.bool)), float("-inf"))
    assert np.max(np.abs(out["LSE"] - torch.logsumexp(sc, dim=-1).numpy())) < 1e-12


def test_attention_causal_row0_and_uniform_closed_forms():
    B, S, H, d, n = 2, 6, 4, 4, 2
    X, Wq, Wk, Wv, Wo, Wqkv, Wos, _ = _attn_inputs(B, S, H, d, n, seed=9)
    out = O.attention_forward(X, Wqkv, Wos, B, S, True)
    V = X @ Wv
    Ocat = np.concatenate([out["O"][i] for i in range(n)], axis=1)
    for b in range(B):
        # query 0 sees only key 0: its output is V[0] for every head
        assert np.allclose(Ocat[b * S], V[b * S], atol=1e-13)
    # Wq = 0: every visible key gets the same weight, O[s] = mean(V[0..s])
    Wqkv0 = O.pack_qkv(np.zeros_like(Wq), Wk, Wv, n, d)
    out0 = O.attention_forward(X, Wqkv0, Wos, B, S, True)
    O0 = np.concatenate([out0["O"][i] for i in range(n)], axis=1)
    for b in range(B):
        for s in range(S):
            assert np.allclose(O0[b * S + s], V[b * S:b * S + s + 1].mean(axis=0), atol=1e-13)
        # and LSE = log(number of visible keys)
        assert np.allclose(out0["LSE"][b], np.log(np.arange(1, S + 1))[None, :], atol=1e-13)


def test_attention_softmax_rows_sum_to_one():
    s = RNG.standard_normal((7, 7)) * 3
    s = np.where(np.tril(np.ones((7, 7), bool)), s, -np.inf)
    P, _ = O._softmax_rows(s)
    assert np.allclose(P.sum(axis=1), 1.0, atol=1e-15)
    assert np.all(P[np.triu_indices(7, 1)] == 0.0)


@pytest.mark.parametrize("n", [1, 2, 4])
def test_attention_head_sharded_equals_unsharded(n):
    B, S, H, d = 2, 5, 4, 3
    X, Wq, Wk, Wv, Wo, Wqkv, Wos, _ = _attn_inputs(B, S, H, d, n, seed=4)
    a = O.attention_forward(X, Wqkv, Wos, B, S, True)["Z"]
    b = O.attention_forward_sharded(X, Wqkv, Wos, B, S, True)
    assert rel(b, a) < 1e-13


def test_attention_rows_restriction():
    B, S, H, d, n = 2, 7, 4, 3, 2
    X, Wq, Wk, Wv, Wo, Wqkv, Wos, _ = _attn_inputs(B, S, H, d, n, seed=8)
    full = O.attention_forward(X, Wqkv, Wos, B, S, True)
    rows = np.array([0, 3, 6, 7, 13])
    r = O.attention_forward_rows(X, Wqkv, Wos, B, S, rows, True)
    assert rel(r["Z"], full["Z"][rows]) < 1e-13
    Ocat = np.concatenate([full["O"][i] for i in range(n)], axis=1)
    assert rel(r["O"], Ocat[rows]) < 1e-13
    lse = full["LSE"].transpose(0, 2, 1).reshape(B * S, -1)
    assert np.max(np.abs(r["LSE"] - lse[rows])) < 1e-12


def test_attention_backward_finite_differences():
    B, S, H, d, n = 1, 4, 2, 2, 2
    X, Wq, Wk, Wv, Wo, Wqkv, Wos, dZ = _attn_inputs(B, S, H, d, n, seed=11)
    g = O.attention_backward(X, Wqkv, Wos, dZ, B, S, True)
    loss = lambda: float(np.sum(dZ * O.attention_forward(X, Wqkv, Wos, B, S, True)["Z"]))
    eps = 1e-6
    for name, arr, grad in (("X", X, g["dX"]), ("Wqkv", Wqkv, g["dWqkv"]), ("Wo", Wos, g["dWo"])):
        fd = np.zeros_like(arr)
        for idx in itertools.product(*[range(s) for s in arr.shape]):
            old = arr[idx]
            arr[idx] = old + eps
            lp = loss()
            arr[idx] = old - eps
            lm = loss()
            arr[idx] = old
            fd[idx] = (lp - lm) / (2 * eps)
        assert rel(grad, fd) < 1e-6, name


@pytest.mark.parametrize("causal", [True, False])
def test_attention_backward_vs_torch_autograd(causal):
    B, S, H, d, n = 2, 6, 4, 4, 2
    X, Wq, Wk, Wv, Wo, Wqkv, Wos, dZ = _attn_inputs(B, S, H, d, n, seed=12)
    tX, tq, tk, tv, to = (torch.from_numpy(a.copy()).requires_grad_(True) for a in (X, Wq, Wk, Wv, Wo))
    shp = lambda a: a.reshape(B, S, H, d).transpose(1, 2)
    o = torch.nn.functional.scaled_dot_product_attention(shp(tX @ tq), shp(tX @ tk), shp(tX @ tv),
                                                         is_causal=causal)
    Z = o.transpose(1, 2).reshape(B * S, H * d) @ to
    (Z * torch.from_numpy(dZ)).sum().backward()
    g = O.attention_backward(X, Wqkv, Wos, dZ, B, S, causal)
    assert rel(g["dX"], tX.grad.numpy()) < 1e-12
    q, k, v = O.unpack_qkv(g["dWqkv"])
    assert rel(q, tq.grad.numpy()) < 1e-12
    assert rel(k, tk.grad.numpy()) < 1e-12
    assert rel(v, tv.grad.numpy()) < 1e-12
    assert rel(O.stack_rows(g["dWo"]), to.grad.numpy()) < 1e-12


# ---------------------------------------------------------------- layer
def test_layer_backward_finite_differences():
    B, S, H, d, n, f = 1, 3, 2, 2, 2, 6
    X, Wq, Wk, Wv, Wo, Wqkv, Wos, dZ = _attn_inputs(B, S, H, d, n, seed=13)
    h = X.shape[1]
    r = np.random.default_rng(14)
    W1s = np.stack(np.split(r.standard_normal((h, f)) * 0.3, n, axis=1))
    W2s = np.stack(np.split(r.standard_normal((f, h)) * 0.3, n, axis=0))
    g = O.layer_backward(X, Wqkv, Wos, W1s, W2s, dZ, B, S, True)
    loss = lambda: float(np.sum(dZ * O.layer_forward(X, Wqkv, Wos, W1s, W2s, B, S, True)["Z"]))
    eps = 1e-6
    for name, arr in (("dX", X), ("dWqkv", Wqkv), ("dWo", Wos), ("dW1s", W1s), ("dW2s", W2s)):
        fd = np.zeros_like(arr)
        for idx in itertools.product(*[range(s) for s in arr.shape]):
            old = arr[idx]
            arr[idx] = old + eps
            lp = loss()
            arr[idx] = old - eps
            lm = loss()
            arr[idx] = old
            fd[idx] = (lp - lm) / (2 * eps)
        assert rel(g[name], fd) < 1e-6, name


# ---------------------------------------------------------------- planted mistakes
def test_planted_mistakes_are_caught(monkeypatch):
    """A plausible slip in the oracle must fail a pin: drop the cubic GeLU term,
    or use the wrong attention scale, and the library cross-checks disagree."""
    x = RNG.standard_normal(256) * 3
    ref = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    monkeypatch.setattr(O, "GELU_CUBIC", 0.0)
    assert np.max(np.abs(O.gelu_tanh(x) - ref)) > 1e-4
    monkeypatch.setattr(O, "GELU_CUBIC", 0.044715)
    B, S, H, d, n = 1, 5, 2, 4, 2
    X, Wq, Wk, Wv, Wo, Wqkv, Wos, _ = _attn_inputs(B, S, H, d, n, seed=21)
    good = O.attention_forward(X, Wqkv, Wos, B, S, True)["Z"]
    bad_scores = lambda q, k, dd, causal: O.matmul(q, k.T) / dd + np.where(
        np.tril(np.ones((q.shape[0], k.shape[0]), bool)), 0.0, -np.inf)
    monkeypatch.setattr(O, "_causal_scores", bad_scores)
    assert rel(O.attention_forward(X, Wqkv, Wos, B, S, True)["Z"], good) > 1e-3


# ---------------------------------------------------------------- gated MLP
def _gmlp_inputs(T, h, f, n, seed=0):
    r = np.random.default_rng(seed)
    X = r.standard_normal((T, h))
    Wg, Wu = r.standard_normal((h, f)) * 0.3, r.standard_normal((h, f)) * 0.3
    Wd = r.standard_normal((f, h)) * 0.3
    dZ = r.standard_normal((T, h))
    c = f // n
    Wgus = np.stack([np.stack([Wg[:, i * c:(i + 1) * c], Wu[:, i * c:(i + 1) * c]], axis=1) for i in range(n)])
    Wds = np.stack([Wd[i * c:(i + 1) * c] for i in range(n)])
    return X, Wg, Wu, Wd, Wgus, Wds, dZ


def test_silu_vs_torch_and_closed_forms():
    x = RNG.standard_normal(2048) * 6
    ref = torch.nn.functional.silu(torch.from_numpy(x)).numpy()
    assert np.max(np.abs(O.silu(x) - ref)) < 1e-13
    assert O.silu(np.array([0.0]))[0] == 0.0
    assert np.allclose(O.silu(np.array([40.0])), 40.0)
    t = torch.from_numpy(x.copy()).requires_grad_(True)
    torch.nn.functional.silu(t).sum().backward()
    assert np.max(np.abs(O.silu_grad(x) - t.grad.numpy())) < 1e-13


def test_gated_mlp_vs_brute_force_and_sharded():
    X, Wg, Wu, Wd, Wgus, Wds, _ = _gmlp_inputs(4, 6, 8, 2)
    T, h = X.shape
    f = Wg.shape[1]
    ref = np.zeros((T, h))
    for t in range(T):
        xs = []
        for c in range(f):
            g = sum(X[t, k] * Wg[k, c] for k in range(h))
            u = sum(X[t, k] * Wu[k, c] for k in range(h))
            xs.append(g / (1.0 + math.exp(-g)) * u)
        for o in range(h):
            ref[t, o] = sum(xs[c] * Wd[c, o] for c in range(f))
    assert rel(O.gated_mlp_forward(X, Wgus, Wds)["Z"], ref) < 1e-13
    for n in divisors(8):
        X, Wg, Wu, Wd, Wgus, Wds, _ = _gmlp_inputs(5, 6, 8, n, seed=n)
        assert rel(O.gated_mlp_forward_sharded(X, Wgus, Wds), O.gated_mlp_forward(X, Wgus, Wds)["Z"]) < 1e-13


def test_gated_mlp_backward_vs_autograd_and_fd():
    X, Wg, Wu, Wd, Wgus, Wds, dZ = _gmlp_inputs(5, 6, 8, 2, seed=4)
    tX, tg, tu, td = (torch.from_numpy(a.copy()).requires_grad_(True) for a in (X, Wg, Wu, Wd))
    Z = (torch.nn.functional.silu(tX @ tg) * (tX @ tu)) @ td
    (Z * torch.from_numpy(dZ)).sum().backward()
    g = O.gated_mlp_backward(X, Wgus, Wds, dZ)
    assert rel(g["dX"], tX.grad.numpy()) < 1e-13
    assert rel(np.concatenate([g["dWgus"][i, :, 0] for i in range(2)], axis=1), tg.grad.numpy()) < 1e-13
    assert rel(np.concatenate([g["dWgus"][i, :, 1] for i in range(2)], axis=1), tu.grad.numpy()) < 1e-13
    assert rel(O.stack_rows(g["dWds"]), td.grad.numpy()) < 1e-13
    # finite differences on a few entries of every input
    loss = lambda: float(np.sum(dZ * O.gated_mlp_forward(X, Wgus, Wds)["Z"]))
    eps = 1e-6
    for arr, grad in ((X, g["dX"]), (Wgus, g["dWgus"]), (Wds, g["dWds"])):
        for idx in [tuple(RNG.integers(0, s) for s in arr.shape) for _ in range(6)]:
            old = arr[idx]
            arr[idx] = old + eps
            lp = loss()
            arr[idx] = old - eps
            lm = loss()
            arr[idx] = old
            assert abs((lp - lm) / (2 * eps) - grad[idx]) < 1e-6 * max(1.0, abs(grad[idx]))


def test_gated_mlp_weight_column_restriction():
    X, Wg, Wu, Wd, Wgus, Wds, dZ = _gmlp_inputs(9, 8, 12, 3, seed=5)
    g = O.gated_mlp_backward(X, Wgus, Wds, dZ)
    cols = np.array([0, 3, 4, 11])
    r = O.gated_mlp_backward_weight_columns(X, Wgus, Wds, dZ, cols)
    dWg = np.concatenate([g["dWgus"][i, :, 0, :] for i in range(3)], axis=1)
    dWu = np.concatenate([g["dWgus"][i, :, 1, :] for i in range(3)], axis=1)
    assert rel(r["dWg_cols"], dWg[:, cols]) < 1e-13
    assert rel(r["dWu_cols"], dWu[:, cols]) < 1e-13
    assert rel(r["dWd_rows"], O.stack_rows(g["dWds"])[cols, :]) < 1e-13


def test_gated_mlp_store_hook():
    """The storage hook: the identity reproduces the exact gradients bit for bit, and
    a rounding hook touches exactly the five stored intermediates (gate, up, A, dG,
    dU), whose rounding moves the gradients by about the rounding's own size."""
    X, Wg, Wu, Wd, Wgus, Wds, dZ = _gmlp_inputs(16, 8, 12, 3, seed=9)
    exact = O.gated_mlp_backward(X, Wgus, Wds, dZ)
    same = O.gated_mlp_backward(X, Wgus, Wds, dZ, store=lambda x: x)
    for k in exact:
        assert np.array_equal(exact[k], same[k]), k
    seen = []
    O.gated_mlp_backward(X, Wgus, Wds, dZ, store=lambda x: seen.append(x.shape) or x)
    assert sorted(seen) == sorted([(16, 12)] * 5)
    q = lambda x: np.round(x * 2.0 ** 10) / 2.0 ** 10     # a coarse fixed-point storage
    rounded = O.gated_mlp_backward(X, Wgus, Wds, dZ, store=q)
    for k in exact:
        d = rel(rounded[k], exact[k])
        assert 0 < d < 1e-2, (k, d)
    cols = np.array([1, 5, 11])
    rc = O.gated_mlp_backward_weight_columns(X, Wgus, Wds, dZ, cols, store=q)
    dWg = np.concatenate([rounded["dWgus"][i, :, 0, :] for i in range(3)], axis=1)
    assert rel(rc["dWg_cols"], dWg[:, cols]) < 1e-13
    assert rel(rc["dWd_rows"], O.stack_rows(rounded["dWds"])[cols, :]) < 1e-13


# ---------------------------------------------------------------- LayerNorm + residual
def test_layer_norm_brute_force_and_torch():
    """The page's three formulas written as loops on a tiny case, and
    torch.nn.functional.layer_norm (fp64, eps = 1e-5)."""
    x = RNG.standard_normal((5, 7)) * 3 + 1.5
    g, b = RNG.standard_normal(7), RNG.standard_normal(7)
    y = O.layer_norm(x, g, b)["y"]
    ref = np.zeros_like(x)
    for t in range(5):
        mu = sum(x[t]) / 7
        var = sum((v - mu) ** 2 for v in x[t]) / 7
        for i in range(7):
            ref[t, i] = g[i] * (x[t, i] - mu) / math.sqrt(var + 1e-5) + b[i]
    assert rel(y, ref) < 1e-14
    tl = torch.nn.functional.layer_norm(torch.from_numpy(x), (7,), torch.from_numpy(g), torch.from_numpy(b), 1e-5)
    assert rel(y, tl.numpy()) < 1e-14


def test_layer_norm_invariants():
    """With gamma = 1, beta = 0 each output row has mean 0 and variance
    var / (var + eps); the output ignores a constant added to a row; scaling a row
    by c changes it only through eps."""
    x = RNG.standard_normal((6, 64)) * 2
    one, zero = np.ones(64), np.zeros(64)
    f = O.layer_norm(x, one, zero)
    var = x.var(axis=1)
    assert np.abs(f["y"].mean(axis=1)).max() < 1e-14
    assert np.allclose(f["y"].var(axis=1), var / (var + 1e-5), rtol=0, atol=1e-13)
    assert rel(O.layer_norm(x + 7.25, one, zero)["y"], f["y"]) < 1e-13
    assert rel(O.layer_norm(x * 3.0, one, zero, eps=0.0)["y"], O.layer_norm(x, one, zero, eps=0.0)["y"]) < 1e-13


def test_layer_norm_backward_vs_autograd_and_fd():
    x = RNG.standard_normal((4, 9)) * 2 + 0.5
    g, b, dy = RNG.standard_normal(9), RNG.standard_normal(9), RNG.standard_normal((4, 9))
    tx, tg, tb = (torch.from_numpy(a.copy()).requires_grad_(True) for a in (x, g, b))
    (torch.nn.functional.layer_norm(tx, (9,), tg, tb, 1e-5) * torch.from_numpy(dy)).sum().backward()
    r = O.layer_norm_backward(x, g, dy)
    assert rel(r["dx"], tx.grad.numpy()) < 1e-12
    assert rel(r["dgamma"], tg.grad.numpy()) < 1e-12
    assert rel(r["dbeta"], tb.grad.numpy()) < 1e-12
    loss = lambda xx: float((O.layer_norm(xx, g, b)["y"] * dy).sum())
    fd = np.zeros_like(x)
    for idx in itertools.product(range(4), range(9)):
        xp, xm = x.copy(), x.copy()
        xp[idx] += 1e-6
        xm[idx] -= 1e-6
        fd[idx] = (loss(xp) - loss(xm)) / 2e-6
    assert rel(r["dx"], fd) < 1e-7


def _prenorm_inputs(seed=21):
    B, S, H, d, n, f = 2, 4, 2, 4, 2, 12
    X, Wq, Wk, Wv, Wo, Wqkv, Wos, dZ = _attn_inputs(B, S, H, d, n, seed=seed)
    h = X.shape[1]
    r = np.random.default_rng(seed + 1)
    W1, W2 = r.standard_normal((h, f)) * 0.3, r.standard_normal((f, h)) * 0.3
    ln = [r.standard_normal(h) * 0.5 + 1.0, r.standard_normal(h) * 0.1, r.standard_normal(h) * 0.5 + 1.0,
          r.standard_normal(h) * 0.1]
    return (B, S, H, d, n, X, Wq, Wk, Wv, Wo, Wqkv, Wos, W1, W2,
            np.stack(np.split(W1, n, axis=1)), np.stack(np.split(W2, n, axis=0)), ln, dZ)


def test_prenorm_layer_vs_torch_autograd():
    """The pre-norm layer written with torch's own LayerNorm, SDPA and tanh-GeLU
    (fp64): forward and every gradient."""
    B, S, H, d, n, X, Wq, Wk, Wv, Wo, Wqkv, Wos, W1, W2, W1s, W2s, ln, dZ = _prenorm_inputs()
    h = X.shape[1]
    F = torch.nn.functional
    t = [torch.from_numpy(a.copy()).requires_grad_(True) for a in (X, Wq, Wk, Wv, Wo, W1, W2, *ln)]
    tX, tq, tk, tv, to, t1, t2, g1, b1, g2, b2 = t
    shp = lambda a: a.reshape(B, S, H, d).transpose(1, 2)
    l1 = F.layer_norm(tX, (h,), g1, b1, 1e-5)
    o = F.scaled_dot_product_attention(shp(l1 @ tq), shp(l1 @ tk), shp(l1 @ tv), is_causal=True)
    H1 = tX + o.transpose(1, 2).reshape(B * S, H * d) @ to
    Z = H1 + F.gelu(F.layer_norm(H1, (h,), g2, b2, 1e-5) @ t1, approximate="tanh") @ t2
    (Z * torch.from_numpy(dZ)).sum().backward()
    fw = O.prenorm_layer_forward(X, ln[0], ln[1], Wqkv, Wos, ln[2], ln[3], W1s, W2s, B, S)
    assert rel(fw["Z"], Z.detach().numpy()) < 1e-13
    assert rel(fw["H1"], H1.detach().numpy()) < 1e-13
    g = O.prenorm_layer_backward(X, ln[0], ln[1], Wqkv, Wos, ln[2], ln[3], W1s, W2s, dZ, B, S)
    assert rel(g["dX"], tX.grad.numpy()) < 1e-12
    q, k, v = O.unpack_qkv(g["dWqkv"])
    for a, b in ((q, tq), (k, tk), (v, tv)):
        assert rel(a, b.grad.numpy()) < 1e-12
    assert rel(O.stack_rows(g["dWo"]), to.grad.numpy()) < 1e-12
    assert rel(O.concat_columns(g["dW1s"]), t1.grad.numpy()) < 1e-12
    assert rel(O.stack_rows(g["dW2s"]), t2.grad.numpy()) < 1e-12
    for name, tt in (("dln1_g", g1), ("dln1_b", b1), ("dln2_g", g2), ("dln2_b", b2)):
        assert rel(g[name], tt.grad.numpy()) < 1e-12, name


def test_prenorm_layer_residual_structure():
    """Zero output projections make both blocks vanish: Z = H1 = X exactly, and the
    input gradient is dZ itself (the residual path alone)."""
    B, S, H, d, n, X, Wq, Wk, Wv, Wo, Wqkv, Wos, W1, W2, W1s, W2s, ln, dZ = _prenorm_inputs(seed=5)
    fw = O.prenorm_layer_forward(X, ln[0], ln[1], Wqkv, np.zeros_like(Wos), ln[2], ln[3], W1s,
                                 np.zeros_like(W2s), B, S)
    assert np.array_equal(fw["Z"], X) and np.array_equal(fw["H1"], X)
    g = O.prenorm_layer_backward(X, ln[0], ln[1], Wqkv, np.zeros_like(Wos), ln[2], ln[3], W1s,
                                 np.zeros_like(W2s), dZ, B, S)
    assert np.array_equal(g["dX"], dZ)


def test_prenorm_layer_row_restriction():
    B, S, H, d, n, X, Wq, Wk, Wv, Wo, Wqkv, Wos, W1, W2, W1s, W2s, ln, dZ = _prenorm_inputs(seed=8)
    full = O.prenorm_layer_forward(X, ln[0], ln[1], Wqkv, Wos, ln[2], ln[3], W1s, W2s, B, S)
    rows = np.array([0, 3, 4, 7])
    r = O.prenorm_layer_forward_rows(X, ln[0], ln[1], Wqkv, Wos, ln[2], ln[3], W1s, W2s, B, S, rows)
    assert rel(r["H1"], full["H1"][rows]) < 1e-13
    assert rel(r["Z"], full["Z"][rows]) < 1e-13
    same = O.prenorm_layer_forward_rows(X, ln[0], ln[1], Wqkv, Wos, ln[2], ln[3], W1s, W2s, B, S, rows,
                                        store=lambda x: x)
    assert rel(same["Z"], full["Z"][rows]) < 1e-13
    q = lambda x: np.round(x * 2.0 ** 10) / 2.0 ** 10
    coarse = O.prenorm_layer_forward_rows(X, ln[0], ln[1], Wqkv, Wos, ln[2], ln[3], W1s, W2s, B, S, rows, store=q)
    assert 0 < rel(coarse["Z"], full["Z"][rows]) < 1e-2
    assert np.array_equal(coarse["H1"], q(coarse["H1"]))


# ---------------------------------------------------------------- grouped-query attention
def _gqa_inputs(B, S, H, Hkv, d, n, h=32, seed=0, wstd=0.3):
    r = np.random.default_rng(seed)
    X = r.standard_normal((B * S, h))
    Wq = r.standard_normal((h, H * d)) * wstd
    Wk, Wv = r.standard_normal((h, Hkv * d)) * wstd, r.standard_normal((h, Hkv * d)) * wstd
    Wo = r.standard_normal((H * d, h)) * wstd
    dZ = r.standard_normal((B * S, h))
    return X, Wq, Wk, Wv, Wo, O.pack_qkv_gqa(Wq, Wk, Wv, n, d), O.split_rows_like(Wo, n), dZ


def test_gqa_with_one_head_per_group_is_mha():
    """Hkv = H: the GQA layout [N][h][(H/N + 2H/N) d] is the MHA layout
    [N][h][3][H/N][d] byte for byte, and the results coincide."""
    B, S, H, d, n = 2, 5, 4, 4, 2
    X, Wq, Wk, Wv, Wo, Wg, Wos, dZ = _gqa_inputs(B, S, H, H, d, n, seed=3)
    Wm = O.pack_qkv(Wq, Wk, Wv, n, d)
    assert np.array_equal(Wm.reshape(Wg.shape), Wg)
    a = O.gqa_attention_forward(X, Wg, Wos, B, S, H, H)
    m = O.attention_forward(X, Wm, Wos, B, S)
    assert rel(a["Z"], m["Z"]) < 1e-14 and rel(a["LSE"], m["LSE"]) < 1e-14
    ga = O.gqa_attention_backward(X, Wg, Wos, dZ, B, S, H, H)
    gm = O.attention_backward(X, Wm, Wos, dZ, B, S)
    assert rel(ga["dX"], gm["dX"]) < 1e-13
    assert rel(ga["dWqkv"], gm["dWqkv"].reshape(ga["dWqkv"].shape)) < 1e-13


def test_gqa_equals_mha_with_repeated_kv_heads():
    """A group shares one K/V head: MHA whose K/V weights repeat each shared head
    for every query head of its group gives the same Z, dX, dWq and dWo, and the
    shared head's gradient is the sum of its copies' gradients."""
    B, S, H, Hkv, d, n = 2, 6, 8, 2, 4, 2
    g = H // Hkv
    X, Wq, Wk, Wv, Wo, Wg, Wos, dZ = _gqa_inputs(B, S, H, Hkv, d, n, seed=4)
    rep = lambda W: np.concatenate([W[:, (j // g) * d:(j // g + 1) * d] for j in range(H)], axis=1)
    Wm = O.pack_qkv(Wq, rep(Wk), rep(Wv), n, d)
    for causal in (True, False):
        a = O.gqa_attention_forward(X, Wg, Wos, B, S, H, Hkv, causal)
        m = O.attention_forward(X, Wm, Wos, B, S, causal)
        assert rel(a["Z"], m["Z"]) < 1e-13
        ga = O.gqa_attention_backward(X, Wg, Wos, dZ, B, S, H, Hkv, causal)
        gm = O.attention_backward(X, Wm, Wos, dZ, B, S, causal)
        assert rel(ga["dX"], gm["dX"]) < 1e-13 and rel(ga["dWo"], gm["dWo"]) < 1e-13
        aq, ak, av = O.unpack_qkv_gqa(ga["dWqkv"], Hkv, d)
        mq, mk, mv = O.unpack_qkv(gm["dWqkv"])
        fold = lambda W: sum(W[:, [c * g * d + gi * d + e for c in range(Hkv) for e in range(d)]]
                             for gi in range(g))
        assert rel(aq, mq) < 1e-13
        assert rel(ak, fold(mk)) < 1e-13 and rel(av, fold(mv)) < 1e-13


def test_gqa_vs_torch_sdpa_autograd():
    """torch's SDPA on K/V heads repeated per group (fp64), forward and autograd."""
    B, S, H, Hkv, d, n = 2, 7, 6, 2, 4, 2
    X, Wq, Wk, Wv, Wo, Wg, Wos, dZ = _gqa_inputs(B, S, H, Hkv, d, n, seed=5)
    t = [torch.from_numpy(a.copy()).requires_grad_(True) for a in (X, Wq, Wk, Wv, Wo)]
    tX, tq, tk, tv, to = t
    shp = lambda a, hh: a.reshape(B, S, hh, d).transpose(1, 2)
    k = shp(tX @ tk, Hkv).repeat_interleave(H // Hkv, dim=1)
    v = shp(tX @ tv, Hkv).repeat_interleave(H // Hkv, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(shp(tX @ tq, H), k, v, is_causal=True)
    Z = o.transpose(1, 2).reshape(B * S, H * d) @ to
    (Z * torch.from_numpy(dZ)).sum().backward()
    assert rel(O.gqa_attention_forward(X, Wg, Wos, B, S, H, Hkv)["Z"], Z.detach().numpy()) < 1e-13
    g = O.gqa_attention_backward(X, Wg, Wos, dZ, B, S, H, Hkv)
    assert rel(g["dX"], tX.grad.numpy()) < 1e-12
    q_, k_, v_ = O.unpack_qkv_gqa(g["dWqkv"], Hkv, d)
    for a, b in ((q_, tq), (k_, tk), (v_, tv)):
        assert rel(a, b.grad.numpy()) < 1e-12
    assert rel(O.stack_rows(g["dWo"]), to.grad.numpy()) < 1e-12


def test_gqa_sharded_equals_unsharded():
    """Every shard count N dividing Hkv (each shard holds whole groups)."""
    B, S, H, Hkv, d = 1, 5, 8, 4, 4
    for n in divisors(Hkv):
        X, Wq, Wk, Wv, Wo, Wg, Wos, dZ = _gqa_inputs(B, S, H, Hkv, d, n, seed=6)
        assert rel(O.gqa_attention_forward_sharded(X, Wg, Wos, B, S, H, Hkv),
                   O.gqa_attention_forward(X, Wg, Wos, B, S, H, Hkv)["Z"]) < 1e-13, n


# ---------------------------------------------------------------- sequence parallelism
def test_seq_shard_layout_roundtrip_and_split_direction():
    """The page's split: TP cuts (batch, seq, hidden) along hidden, SP along seq:
    shard c of the SP layout holds positions c*S/N .. of every sequence, whole
    hidden vectors."""
    B, S, n, h = 3, 8, 4, 5
    X = np.arange(B * S * h, dtype=np.float64).reshape(B * S, h)
    Xs = O.to_seq_shards(X, B, S, n)
    assert Xs.shape == (n, B, S // n, h)
    for c in range(n):
        for b in range(B):
            for sl in range(S // n):
                assert np.array_equal(Xs[c, b, sl], X[b * S + c * (S // n) + sl])
    assert np.array_equal(O.from_seq_shards(Xs), X)


def test_sp_layer_equals_tp_layer():
    """TP + SP computes the same layer: all-gather before each block and
    reduce-scatter after it give the all-reduce's sums, row by row."""
    B, S, H, d, n, X, Wq, Wk, Wv, Wo, Wqkv, Wos, W1, W2, W1s, W2s, ln, dZ = _prenorm_inputs(seed=11)
    ref = O.prenorm_layer_forward(X, ln[0], ln[1], Wqkv, Wos, ln[2], ln[3], W1s, W2s, B, S)
    sp = O.sp_prenorm_layer_forward(O.to_seq_shards(X, B, S, n), ln[0], ln[1], Wqkv, Wos, ln[2], ln[3], W1s, W2s, B, S)
    assert rel(O.from_seq_shards(sp["Z"]), ref["Z"]) < 1e-13
    assert rel(O.from_seq_shards(sp["H1"]), ref["H1"]) < 1e-13
    g = O.sp_prenorm_layer_backward(O.to_seq_shards(X, B, S, n), ln[0], ln[1], Wqkv, Wos, ln[2], ln[3], W1s, W2s,
                                    O.to_seq_shards(dZ, B, S, n), B, S)
    gr = O.prenorm_layer_backward(X, ln[0], ln[1], Wqkv, Wos, ln[2], ln[3], W1s, W2s, dZ, B, S)
    assert rel(O.from_seq_shards(g["dX"]), gr["dX"]) < 1e-13
    assert rel(g["dW1s"], gr["dW1s"]) < 1e-13 and rel(g["dln2_g"], gr["dln2_g"]) < 1e-13


def test_sp_reduce_scatter_then_all_gather_is_all_reduce():
    """The page's cost argument rests on all-reduce = reduce-scatter + all-gather:
    the composition gives every shard the full sum."""
    B, S, n, h = 2, 8, 4, 3
    parts = [RNG.standard_normal((B * S, h)) for _ in range(n)]
    rs = O._reduce_scatter_seq(parts, B, S, n)
    assert rel(O._all_gather_seq(rs), sum(parts)) < 1e-15
