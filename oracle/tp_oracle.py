"""fp64 CPU oracle for the Megatron tensor-parallel transformer block.

TEST INFRASTRUCTURE ONLY.  This module is the yardstick the CUDA path is measured
against; it is imported by ``tests/``, by ``__graft_entry__.smoke()`` and by the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` and by nothing else.
The product path (``tensor_transformer_block_gb300``) never imports it, and it
never imports the product path: the two share no code.  Inputs reach it as plain
numpy arrays (the seeded generators live in a module of their own).

Everything is computed in float64 from the *unsharded* definitions, because the
tensor-parallel method reaches exactly the same numbers (up to rounding order)
as the plain product: the pages' block-matrix identities

    column split:  X [W_0, W_1] = [X W_0, X W_1]          (io.zouht.com 张量并行 §2.1, first identity)
    row split:     [X_0, X_1] [W_0; W_1] = X_0 W_0 + X_1 W_1  (same §2.1, second identity)

say so.  The sharded re-statements at the bottom follow the split step by step;
the tests use them to pin the identities themselves.

Page short names used in the citations (the pages are Chinese web articles):
  * "damodev 3D并行"      damodev.csdn.net/6a43867610ee7a33f284fb9e.html
  * "zouht 张量并行"      io.zouht.com/197.html
  * "wangyu 张量并行"     wangyu.me/posts/llm/tensor-parallelism/ (大语言模型并行策略（三）：张量并行)
  * "guijiagi 张量并行"   guijiagi.com/tags/张量并行/
  * "sunjinbo 并行方式"   sunjinbo.space/document/parallelism.html (大模型分布式并行方式详解)

Conventions (readings where the pages are silent):
  * Y = X W with W stored [in x out] (wangyu 张量并行 §两种切分方式: X is B x M,
    W is M x N; guijiagi 张量并行 §线性层的切分: W in R^{d x h}).
  * No biases: none of the pages' split identities carries one.
  * Act = GeLU, tanh form 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))
    (zouht 张量并行 §2.2.1 names "Gelu(X W_1)"; the tanh form is the named workload's).
  * Attention: per head softmax(Q K^T / sqrt(d)) V with a causal mask
    (key position <= query position), no dropout.
  * Shard layouts are the pages' splits: W1s[i] = W1[:, i*f/N:(i+1)*f/N]
    (column split), W2s[i] = W2[i*f/N:(i+1)*f/N, :] (row split); shard i owns
    heads i*H/N .. (i+1)*H/N-1 (zouht 张量并行 §2.2.1, 32 heads on 4 GPUs = 8 each).
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "matmul", "gelu_tanh", "gelu_tanh_grad",
    "concat_columns", "stack_rows", "split_columns_like", "split_rows_like",
    "mlp_forward", "mlp_backward",
    "mlp_forward_sharded", "mlp_forward_two_allgather", "mlp_backward_sharded",
    "unpack_qkv", "pack_qkv",
    "attention_forward", "attention_backward", "attention_forward_sharded",
    "layer_forward", "layer_backward",
    "mlp_backward_weight_columns", "attention_forward_rows",
    "silu", "silu_grad", "gated_mlp_forward", "gated_mlp_backward", "gated_mlp_forward_sharded",
    "gated_mlp_backward_weight_columns",
    "LN_EPS", "layer_norm", "layer_norm_backward", "prenorm_layer_forward", "prenorm_layer_backward",
    "prenorm_layer_forward_rows",
    "unpack_qkv_gqa", "pack_qkv_gqa", "gqa_attention_forward", "gqa_attention_backward",
    "gqa_attention_forward_sharded",
    "to_seq_shards", "from_seq_shards", "sp_prenorm_layer_forward", "sp_prenorm_layer_backward",
]

SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)
GELU_CUBIC = 0.044715


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def matmul(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Plain fp64 matrix product (library primitive; pinned by a brute-force
    triple loop in the tests)."""
    return _f64(a) @ _f64(b)


# --------------------------------------------------------------------------
# Activation
# --------------------------------------------------------------------------
def gelu_tanh(x: np.ndarray) -> np.ndarray:
    """GeLU, tanh form: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).

    The MLP's Act (damodev 3D并行 §1.2.1: "ReLU or GeLU"; zouht 张量并行 §2.2.1:
    first layer Gelu(X W_1)).  Element-wise, which is what lets it run per shard.
    """
    x = _f64(x)
    u = SQRT_2_OVER_PI * (x + GELU_CUBIC * x * x * x)
    return 0.5 * x * (1.0 + np.tanh(u))


def gelu_tanh_grad(x: np.ndarray) -> np.ndarray:
    """d/dx of :func:`gelu_tanh`, differentiated by hand:
    0.5 (1 + tanh u) + 0.5 x (1 - tanh^2 u) sqrt(2/pi) (1 + 3*0.044715 x^2)."""
    x = _f64(x)
    u = SQRT_2_OVER_PI * (x + GELU_CUBIC * x * x * x)
    t = np.tanh(u)
    du = SQRT_2_OVER_PI * (1.0 + 3.0 * GELU_CUBIC * x * x)
    return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * du


# --------------------------------------------------------------------------
# Shard layouts <-> unsharded matrices (the pages' splits)
# --------------------------------------------------------------------------
def concat_columns(ws: np.ndarray) -> np.ndarray:
    """[N][rows][cols/N] column blocks -> the unsharded [rows][cols] matrix.

    Column split (damodev 3D并行 §1.1 "列切分"; wangyu 张量并行 §按列切分: each
    W_i is M x (N/n)): W = [W_0, W_1, ..., W_{N-1}].
    """
    ws = _f64(ws)
    n, rows, cols = ws.shape
    return np.concatenate([ws[i] for i in range(n)], axis=1).reshape(rows, n * cols)


def stack_rows(ws: np.ndarray) -> np.ndarray:
    """[N][rows/N][cols] row blocks -> the unsharded [rows][cols] matrix.

    Row split (damodev 3D并行 §1.1 "外积和切分"; wangyu 张量并行 §按行切分: each
    W_i is (M/m) x N): W = [W_0; W_1; ...; W_{N-1}].
    """
    ws = _f64(ws)
    n, rows, cols = ws.shape
    return np.concatenate([ws[i] for i in range(n)], axis=0).reshape(n * rows, cols)


def split_columns_like(w: np.ndarray, n: int) -> np.ndarray:
    """Inverse of :func:`concat_columns` (used to return gradients in shard layout)."""
    w = _f64(w)
    rows, cols = w.shape
    c = cols // n
    return np.stack([w[:, i * c:(i + 1) * c] for i in range(n)])


def split_rows_like(w: np.ndarray, n: int) -> np.ndarray:
    """Inverse of :func:`stack_rows`."""
    w = _f64(w)
    rows, cols = w.shape
    r = rows // n
    return np.stack([w[i * r:(i + 1) * r, :] for i in range(n)])


# --------------------------------------------------------------------------
# MLP block
# --------------------------------------------------------------------------
def mlp_forward(X, W1s, W2s) -> dict:
    """Unsharded MLP block Z = Act(X W1) W2 (damodev 3D并行 §1.2.1, eq. 1.2-1.3;
    zouht 张量并行 §2.2.1 前馈网络).

    W1 is the column concatenation of the shards W1s[i] and W2 the row stack of
    W2s[i]; by the §2.1 identities the sharded block computes the same Z.
    Returns Y = X W1 (pre-activation, in shard layout [N][T][f/N]),
    A = GeLU(Y) (shard layout) and Z [T][h].
    """
    X = _f64(X)
    n = W1s.shape[0]
    W1 = concat_columns(W1s)
    W2 = stack_rows(W2s)
    Y = matmul(X, W1)
    A = gelu_tanh(Y)
    Z = matmul(A, W2)
    return {"Y": split_columns_like(Y, n), "A": split_columns_like(A, n), "Z": Z}


def mlp_backward(X, W1s, W2s, dZ) -> dict:
    """Gradients of L = <dZ, Z> for the unsharded block, by the chain rule.

    dA = dZ W2^T, dY = dA * GeLU'(Y), dW2 = A^T dZ, dW1 = X^T dY, dX = dY W1^T.
    The pages give the sharded forms (wangyu 张量并行 §通信模式: for the column
    split dW_i = X^T dY_i and dX = sum_i dY_i W_i^T, the all-reduce; for the row
    split dL/dY_i = dL/dY, dW_i = X_i^T dY); the unsharded product is the same
    numbers.  Weight gradients come back in shard layout.
    """
    X, dZ = _f64(X), _f64(dZ)
    n = W1s.shape[0]
    W1 = concat_columns(W1s)
    W2 = stack_rows(W2s)
    Y = matmul(X, W1)
    A = gelu_tanh(Y)
    dA = matmul(dZ, W2.T)
    dY = dA * gelu_tanh_grad(Y)
    dW2 = matmul(A.T, dZ)
    dW1 = matmul(X.T, dY)
    dX = matmul(dY, W1.T)
    return {"dX": dX, "dW1s": split_columns_like(dW1, n), "dW2s": split_rows_like(dW2, n),
            "dY": split_columns_like(dY, n)}


def mlp_forward_sharded(X, W1s, W2s) -> dict:
    """The pages' tensor-parallel MLP, shard by shard (damodev 3D并行 §1.2.1;
    wangyu 张量并行 §多层感知机（MLP）中的张量并行):

      shard i:  Y_i = X W1_i  (column split, X replicated),
                A_i = Act(Y_i)  (element-wise, so no communication),
                P_i = A_i W2_i  (row split; A_i is already X's column block i),
      all-reduce: Z = sum_i P_i.
    """
    X = _f64(X)
    n = W1s.shape[0]
    Ys, As, Ps = [], [], []
    for i in range(n):
        Yi = matmul(X, W1s[i])
        Ai = gelu_tanh(Yi)
        Ys.append(Yi)
        As.append(Ai)
        Ps.append(matmul(Ai, W2s[i]))
    Z = Ps[0].copy()
    for i in range(1, n):
        Z = Z + Ps[i]
    return {"Y": np.stack(Ys), "A": np.stack(As), "Z": Z, "partials": np.stack(Ps)}


def mlp_forward_two_allgather(X, W1s, W2s) -> np.ndarray:
    """The naive variant the damodev page rejects (§1.2.1, eq. 1.4-1.5): column
    split of both GEMMs with an all-gather after each.  Same Z, two gathers."""
    X = _f64(X)
    n = W1s.shape[0]
    A = np.concatenate([gelu_tanh(matmul(X, W1s[i])) for i in range(n)], axis=1)  # all-gather 1
    W2 = stack_rows(W2s)
    h = W2.shape[1]
    c = h // n if h % n == 0 else None
    if c is None:  # the column split of W2 needs n | h; fall back to one block
        return matmul(A, W2)
    return np.concatenate([matmul(A, W2[:, i * c:(i + 1) * c]) for i in range(n)], axis=1)  # all-gather 2


def mlp_backward_sharded(X, W1s, W2s, dZ) -> dict:
    """Sharded backward as the pages state it (wangyu 张量并行 §通信模式):
    row-split layer: dL/dP_i = dL/dZ (broadcast), dW2_i = A_i^T dZ, dA_i = dZ W2_i^T;
    column-split layer: dW1_i = X^T dY_i, dX = sum_i dY_i W1_i^T (the all-reduce)."""
    X, dZ = _f64(X), _f64(dZ)
    n = W1s.shape[0]
    dW1s, dW2s, parts = [], [], []
    for i in range(n):
        Yi = matmul(X, W1s[i])
        Ai = gelu_tanh(Yi)
        dW2s.append(matmul(Ai.T, dZ))
        dYi = matmul(dZ, _f64(W2s[i]).T) * gelu_tanh_grad(Yi)
        dW1s.append(matmul(X.T, dYi))
        parts.append(matmul(dYi, _f64(W1s[i]).T))
    dX = parts[0].copy()
    for i in range(1, n):
        dX = dX + parts[i]
    return {"dX": dX, "dW1s": np.stack(dW1s), "dW2s": np.stack(dW2s)}


# --------------------------------------------------------------------------
# Self-attention block
# --------------------------------------------------------------------------
def unpack_qkv(Wqkv) -> tuple:
    """Shard-major [N][h][3][H/N][d] -> unsharded Wq, Wk, Wv, each [h][H*d].

    Q/K/V are split by columns, head by head (zouht 张量并行 §2.2.1 多头注意力机制;
    wangyu 张量并行 §注意力机制中的张量并行: split by the head dimension, which is
    a column split); shard i holds heads i*H/N .. (i+1)*H/N-1, Q then K then V.
    """
    W = _f64(Wqkv)
    n, h, three, hn, d = W.shape
    assert three == 3
    full = np.transpose(W, (1, 2, 0, 3, 4)).reshape(h, 3, n * hn * d)
    return full[:, 0, :].copy(), full[:, 1, :].copy(), full[:, 2, :].copy()


def pack_qkv(Wq, Wk, Wv, n: int, d: int) -> np.ndarray:
    """Inverse of :func:`unpack_qkv`."""
    h, hd = Wq.shape
    H = hd // d
    full = np.stack([_f64(Wq), _f64(Wk), _f64(Wv)], axis=1).reshape(h, 3, n, H // n, d)
    return np.ascontiguousarray(np.transpose(full, (2, 0, 1, 3, 4)))


def _causal_scores(q, k, d, causal):
    s = matmul(q, k.T) / math.sqrt(d)
    if causal:
        S = s.shape[0]
        s = np.where(np.tril(np.ones((S, S), dtype=bool)), s, -np.inf)
    return s


def _softmax_rows(s):
    m = np.max(s, axis=1, keepdims=True)
    e = np.exp(s - m)
    z = np.sum(e, axis=1, keepdims=True)
    return e / z, (m + np.log(z))[:, 0]


def attention_forward(X, Wqkv, Wo, B: int, S: int, causal: bool = True) -> dict:
    """Unsharded multi-head self-attention block.

    Per batch b and head j (damodev 3D并行 §1.2.2, eq. 1.12 stripped from the
    page; wangyu 张量并行 §注意力机制中的张量并行):
        Q = X_b Wq_j, K = X_b Wk_j, V = X_b Wv_j,
        head_j = softmax(mask(Q K^T / sqrt(d))) V,
    then Z = concat_j(head_j) Wo (damodev §1.2.2, eq. 1.13).  Returns Z [T][h],
    QKV in shard layout [N][T][3][H/N][d], O in shard layout [N][T][H/N*d] and
    LSE [B][H][S] = log sum_k exp(scores) (natural log of the scaled scores).
    """
    X = _f64(X)
    n, h, _, hn, d = Wqkv.shape
    H = n * hn
    T = B * S
    Wq, Wk, Wv = unpack_qkv(Wqkv)
    Wo_full = stack_rows(Wo)
    Q, K, V = matmul(X, Wq), matmul(X, Wk), matmul(X, Wv)
    O = np.zeros((T, H * d))
    LSE = np.zeros((B, H, S))
    for b in range(B):
        r = slice(b * S, (b + 1) * S)
        for j in range(H):
            c = slice(j * d, (j + 1) * d)
            P, lse = _softmax_rows(_causal_scores(Q[r, c], K[r, c], d, causal))
            O[r, c] = matmul(P, V[r, c])
            LSE[b, j] = lse
    Z = matmul(O, Wo_full)
    QKV = np.stack([Q, K, V], axis=1).reshape(T, 3, n, hn, d).transpose(2, 0, 1, 3, 4)
    Osh = O.reshape(T, n, hn * d).transpose(1, 0, 2)
    return {"Z": Z, "QKV": np.ascontiguousarray(QKV).reshape(n, T, 3 * hn * d),
            "O": np.ascontiguousarray(Osh), "LSE": LSE}


def attention_backward(X, Wqkv, Wo, dZ, B: int, S: int, causal: bool = True) -> dict:
    """Gradients of L = <dZ, Z> for :func:`attention_forward`.

    The pages give no attention backward; this is the chain rule through the
    definition, with the textbook softmax Jacobian dS = P * (dP - rowsum(dP * P)).
    """
    X, dZ = _f64(X), _f64(dZ)
    n, h, _, hn, d = Wqkv.shape
    H = n * hn
    T = B * S
    Wq, Wk, Wv = unpack_qkv(Wqkv)
    Wo_full = stack_rows(Wo)
    Q, K, V = matmul(X, Wq), matmul(X, Wk), matmul(X, Wv)
    O = np.zeros((T, H * d))
    for b in range(B):
        r = slice(b * S, (b + 1) * S)
        for j in range(H):
            c = slice(j * d, (j + 1) * d)
            P, _ = _softmax_rows(_causal_scores(Q[r, c], K[r, c], d, causal))
            O[r, c] = matmul(P, V[r, c])
    dWo = matmul(O.T, dZ)
    dO = matmul(dZ, Wo_full.T)
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    for b in range(B):
        r = slice(b * S, (b + 1) * S)
        for j in range(H):
            c = slice(j * d, (j + 1) * d)
            # P is recomputed from its definition rather than kept per head
            P, _ = _softmax_rows(_causal_scores(Q[r, c], K[r, c], d, causal))
            dV[r, c] = matmul(P.T, dO[r, c])
            dP = matmul(dO[r, c], V[r, c].T)
            dS = P * (dP - np.sum(dP * P, axis=1, keepdims=True))
            dQ[r, c] = matmul(dS, K[r, c]) / math.sqrt(d)
            dK[r, c] = matmul(dS.T, Q[r, c]) / math.sqrt(d)
    dWq, dWk, dWv = matmul(X.T, dQ), matmul(X.T, dK), matmul(X.T, dV)
    dX = matmul(dQ, Wq.T) + matmul(dK, Wk.T) + matmul(dV, Wv.T)
    return {"dX": dX, "dWqkv": pack_qkv(dWq, dWk, dWv, n, d), "dWo": split_rows_like(dWo, n)}


def attention_forward_sharded(X, Wqkv, Wo, B: int, S: int, causal: bool = True) -> np.ndarray:
    """Head-sharded attention as the pages split it (zouht 张量并行 §2.2.1; wangyu
    张量并行 §注意力机制中的张量并行): shard i computes its own heads' Q/K/V with
    its column block of Wqkv, runs attention on those heads, multiplies its O_i by
    its row block Wo_i; an all-reduce sums the N partial outputs."""
    X = _f64(X)
    n, h, _, hn, d = Wqkv.shape
    T = B * S
    Z = None
    for i in range(n):
        Wi = _f64(Wqkv[i]).reshape(h, 3 * hn * d)
        qkv = matmul(X, Wi).reshape(T, 3, hn, d)
        Oi = np.zeros((T, hn * d))
        for b in range(B):
            r = slice(b * S, (b + 1) * S)
            for jj in range(hn):
                q, k, v = qkv[r, 0, jj], qkv[r, 1, jj], qkv[r, 2, jj]
                P, _ = _softmax_rows(_causal_scores(q, k, d, causal))
                Oi[r, jj * d:(jj + 1) * d] = matmul(P, v)
        part = matmul(Oi, Wo[i])
        Z = part if Z is None else Z + part
    return Z


# --------------------------------------------------------------------------
# Full layer: attention block then MLP block
# --------------------------------------------------------------------------
def layer_forward(X, Wqkv, Wo, W1s, W2s, B: int, S: int, causal: bool = True) -> dict:
    """Z = MLP(Attn(X)).  The pages place LayerNorm, dropout and residuals outside
    the tensor-parallel regions (zouht 张量并行 §2.2.2) and give no layer formula;
    the layer here is the two TP blocks in sequence, attention first."""
    a = attention_forward(X, Wqkv, Wo, B, S, causal)
    m = mlp_forward(a["Z"], W1s, W2s)
    return {"Z": m["Z"], "H": a["Z"], "attn": a, "mlp": m}


def layer_backward(X, Wqkv, Wo, W1s, W2s, dZ, B: int, S: int, causal: bool = True) -> dict:
    """Gradients of L = <dZ, layer_forward(X)["Z"]>: MLP backward, then the
    attention backward fed with the MLP's input gradient."""
    a = attention_forward(X, Wqkv, Wo, B, S, causal)
    gm = mlp_backward(a["Z"], W1s, W2s, dZ)
    ga = attention_backward(X, Wqkv, Wo, gm["dX"], B, S, causal)
    return {"dX": ga["dX"], "dWqkv": ga["dWqkv"], "dWo": ga["dWo"],
            "dW1s": gm["dW1s"], "dW2s": gm["dW2s"], "dH": gm["dX"]}


# --------------------------------------------------------------------------
# Restrictions of the same definitions to a subset of outputs (for sampled
# checks at full size, where the whole product would take the CPU too long)
# --------------------------------------------------------------------------
def mlp_backward_weight_columns(X, W1s, W2s, dZ, cols) -> dict:
    """dW1[:, cols] and dW2[cols, :] of :func:`mlp_backward`, for global FFN
    column indices ``cols``.  Column c of dY only needs column c of Y and of dA:
    dY[:, c] = (dZ W2[c, :]^T) * GeLU'(X W1[:, c]); dW1[:, c] = X^T dY[:, c];
    dW2[c, :] = A[:, c]^T dZ with A[:, c] = GeLU(X W1[:, c])."""
    X, dZ = _f64(X), _f64(dZ)
    cols = np.asarray(cols, dtype=np.int64)
    W1 = concat_columns(W1s)[:, cols]
    W2 = stack_rows(W2s)[cols, :]
    Y = matmul(X, W1)
    dY = matmul(dZ, W2.T) * gelu_tanh_grad(Y)
    return {"dW1_cols": matmul(X.T, dY), "dW2_rows": matmul(gelu_tanh(Y).T, dZ)}


def attention_forward_rows(X, Wqkv, Wo, B: int, S: int, rows, causal: bool = True) -> dict:
    """Z[rows] and O[rows] of :func:`attention_forward` for global token indices
    ``rows``: each query row needs its own Q row and the K/V rows of its batch."""
    X = _f64(X)
    n, h, _, hn, d = Wqkv.shape
    H = n * hn
    rows = np.asarray(rows, dtype=np.int64)
    Wq, Wk, Wv = unpack_qkv(Wqkv)
    Wo_full = stack_rows(Wo)
    K, V = matmul(X, Wk), matmul(X, Wv)
    Q = matmul(X[rows], Wq)
    O = np.zeros((len(rows), H * d))
    LSE = np.zeros((len(rows), H))
    for ri, t in enumerate(rows):
        b, s = divmod(int(t), S)
        last = s + 1 if causal else S
        kr = slice(b * S, b * S + last)
        for j in range(H):
            c = slice(j * d, (j + 1) * d)
            sc = matmul(Q[ri:ri + 1, c], K[kr, c].T) / math.sqrt(d)
            P, lse = _softmax_rows(sc)
            O[ri, c] = matmul(P, V[kr, c])[0]
            LSE[ri, j] = lse[0]
    return {"Z": matmul(O, Wo_full), "O": O, "LSE": LSE}


# --------------------------------------------------------------------------
# Gated MLP (the Qwen3-style MLP of wangyu 张量并行 §多层感知机（MLP）中的张量并行)
# --------------------------------------------------------------------------
def silu(x: np.ndarray) -> np.ndarray:
    """silu(x) = x * sigmoid(x) = x / (1 + e^-x)."""
    x = _f64(x)
    return x / (1.0 + np.exp(-x))


def silu_grad(x: np.ndarray) -> np.ndarray:
    """d/dx silu(x) = s (1 + x (1 - s)) with s = sigmoid(x)."""
    x = _f64(x)
    s = 1.0 / (1.0 + np.exp(-x))
    return s * (1.0 + x * (1.0 - s))


def _split_gate_up(Wgus):
    """Shard-major [N][h][2][f/N] (shard i = [W_gate_i | W_up_i], the page's fused
    column concatenation) -> unsharded W_gate, W_up, each [h][f]."""
    W = _f64(Wgus)
    n, h, two, fn = W.shape
    assert two == 2
    Wg = np.concatenate([W[i, :, 0, :] for i in range(n)], axis=1)
    Wu = np.concatenate([W[i, :, 1, :] for i in range(n)], axis=1)
    return Wg, Wu


def gated_mlp_forward(X, Wgus, Wds) -> dict:
    """gate = X W_gate, up = X W_up, x = silu(gate) * up, down = x W_down (wangyu
    张量并行 §多层感知机: the Qwen3 MLP; W_gate and W_up concatenated by columns so
    gate and up come from one GEMM).  Unsharded; returns GU in shard layout
    [N][T][2][f/N] (gate block then up block per shard), A = x [N][T][f/N], Z."""
    X = _f64(X)
    n = Wgus.shape[0]
    Wg, Wu = _split_gate_up(Wgus)
    Wd = stack_rows(Wds)
    G = matmul(X, Wg)
    U = matmul(X, Wu)
    A = silu(G) * U
    Z = matmul(A, Wd)
    GU = np.stack([split_columns_like(G, n), split_columns_like(U, n)], axis=2)  # [N][T][2][f/N]
    return {"GU": GU, "A": split_columns_like(A, n), "Z": Z}


def _keep(x):
    return x


def gated_mlp_backward(X, Wgus, Wds, dZ, store=None) -> dict:
    """Gradients of <dZ, Z>: dA = dZ W_down^T, dG = dA * up * silu'(gate),
    dU = dA * silu(gate), dW_down = A^T dZ, dW_gate = X^T dG, dW_up = X^T dU,
    dX = dG W_gate^T + dU W_up^T.  Weight gradients in shard layout.

    ``store`` (default: none) is applied to each intermediate a tensor-parallel
    implementation keeps in memory between its products (gate, up, A, dG, dU);
    the tests pass a rounding to the storage type to measure the error that
    storage alone causes.  Without it this is the exact definition."""
    st = store or _keep
    X, dZ = _f64(X), _f64(dZ)
    n = Wgus.shape[0]
    Wg, Wu = _split_gate_up(Wgus)
    Wd = stack_rows(Wds)
    G0 = matmul(X, Wg)
    U0 = matmul(X, Wu)
    A = st(silu(G0) * U0)
    G, U = st(G0), st(U0)
    dA = matmul(dZ, Wd.T)
    dG = st(dA * U * silu_grad(G))
    dU = st(dA * silu(G))
    dWd = matmul(A.T, dZ)
    dWg = matmul(X.T, dG)
    dWu = matmul(X.T, dU)
    dX = matmul(dG, Wg.T) + matmul(dU, Wu.T)
    dWgus = np.stack([split_columns_like(dWg, n), split_columns_like(dWu, n)], axis=2)  # [N][h][2][f/N]
    return {"dX": dX, "dWgus": dWgus, "dWds": split_rows_like(dWd, n)}


def gated_mlp_forward_sharded(X, Wgus, Wds) -> np.ndarray:
    """Shard by shard: shard i computes [gate_i | up_i] = X [W_gate_i | W_up_i] in one
    product, x_i = silu(gate_i) * up_i locally, then x_i W_down_i; the all-reduce
    sums the partial products."""
    X = _f64(X)
    n = Wgus.shape[0]
    Z = None
    for i in range(n):
        Wi = _f64(Wgus[i])
        h, _, fn = Wi.shape
        GUi = matmul(X, Wi.reshape(h, 2 * fn))
        xi = silu(GUi[:, :fn]) * GUi[:, fn:]
        part = matmul(xi, Wds[i])
        Z = part if Z is None else Z + part
    return Z


def gated_mlp_backward_weight_columns(X, Wgus, Wds, dZ, cols, store=None) -> dict:
    """dW_gate[:, cols], dW_up[:, cols] and dW_down[cols, :] of
    :func:`gated_mlp_backward` for global FFN column indices ``cols``.  Column c of
    dG and dU needs only column c of gate, up and dA: dA[:, c] = dZ W_down[c, :]^T,
    dG[:, c] = dA[:, c] up[:, c] silu'(gate[:, c]), dU[:, c] = dA[:, c] silu(gate[:, c]).
    ``store`` as in :func:`gated_mlp_backward`."""
    st = store or _keep
    X, dZ = _f64(X), _f64(dZ)
    cols = np.asarray(cols, dtype=np.int64)
    Wg, Wu = _split_gate_up(Wgus)
    Wd = stack_rows(Wds)[cols, :]
    G0 = matmul(X, Wg[:, cols])
    U0 = matmul(X, Wu[:, cols])
    A = st(silu(G0) * U0)
    G, U = st(G0), st(U0)
    dA = matmul(dZ, Wd.T)
    return {"dWg_cols": matmul(X.T, st(dA * U * silu_grad(G))), "dWu_cols": matmul(X.T, st(dA * silu(G))),
            "dWd_rows": matmul(A.T, dZ)}


# --------------------------------------------------------------------------
# LayerNorm and residuals around the two blocks
# --------------------------------------------------------------------------
LN_EPS = 1e-5  # the pages leave epsilon open ("a very small value"); 1e-5 is the reading taken


def layer_norm(x, gamma, beta, eps: float = LN_EPS) -> dict:
    """Per row (one hidden state of d_model = h values): mu = mean(h_i),
    sigma^2 = mean((h_i - mu)^2), h_hat = (h - mu) / sqrt(sigma^2 + eps),
    h' = gamma * h_hat + beta (zouht 张量并行 §2.2.2, LayerNorm).  Returns y = h'
    and the per-row mean and 1 / sqrt(sigma^2 + eps) a backward needs."""
    x = _f64(x)
    mu = x.mean(axis=1)
    var = ((x - mu[:, None]) ** 2).mean(axis=1)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (x - mu[:, None]) * rstd[:, None]
    return {"y": xhat * _f64(gamma)[None, :] + _f64(beta)[None, :], "mean": mu, "rstd": rstd}


def layer_norm_backward(x, gamma, dy, eps: float = LN_EPS) -> dict:
    """Gradients of <dy, layer_norm(x)["y"]>.  The pages give no backward; by the
    chain rule through the definition above, with g = dy * gamma and h the row
    length: dx = rstd (g - mean(g) - h_hat mean(g h_hat)) per row,
    dgamma = sum over rows of dy * h_hat, dbeta = sum over rows of dy."""
    x, dy = _f64(x), _f64(dy)
    f = layer_norm(x, np.ones(x.shape[1]), np.zeros(x.shape[1]), eps)
    xhat, rstd = f["y"], f["rstd"]
    g = dy * _f64(gamma)[None, :]
    dx = rstd[:, None] * (g - g.mean(axis=1, keepdims=True) - xhat * (g * xhat).mean(axis=1, keepdims=True))
    return {"dx": dx, "dgamma": (dy * xhat).sum(axis=0), "dbeta": dy.sum(axis=0)}


def prenorm_layer_forward(X, ln1_g, ln1_b, Wqkv, Wo, ln2_g, ln2_b, W1s, W2s, B: int, S: int,
                          causal: bool = True, eps: float = LN_EPS) -> dict:
    """The layer with LayerNorm and residuals in the replicated (non-TP) region
    (zouht 张量并行 §2.2.2; sunjinbo 并行方式 §SP: LayerNorm, dropout and the
    residual sit outside the tensor-parallel blocks).  The pages give no placement;
    the reading taken is the pre-norm layer, dropout off:
        H1 = X + Attn(LN1(X)),   Z = H1 + MLP(LN2(H1))."""
    X = _f64(X)
    l1 = layer_norm(X, ln1_g, ln1_b, eps)
    a = attention_forward(l1["y"], Wqkv, Wo, B, S, causal)
    H1 = X + a["Z"]
    l2 = layer_norm(H1, ln2_g, ln2_b, eps)
    m = mlp_forward(l2["y"], W1s, W2s)
    return {"Z": H1 + m["Z"], "H1": H1, "LN1": l1, "LN2": l2, "attn": a, "mlp": m}


def prenorm_layer_backward(X, ln1_g, ln1_b, Wqkv, Wo, ln2_g, ln2_b, W1s, W2s, dZ, B: int, S: int,
                           causal: bool = True, eps: float = LN_EPS) -> dict:
    """Gradients of <dZ, prenorm_layer_forward(...)["Z"]>: each residual passes its
    gradient through unchanged and adds the gradient through its block."""
    dZ = _f64(dZ)
    f = prenorm_layer_forward(X, ln1_g, ln1_b, Wqkv, Wo, ln2_g, ln2_b, W1s, W2s, B, S, causal, eps)
    gm = mlp_backward(f["LN2"]["y"], W1s, W2s, dZ)
    g2 = layer_norm_backward(f["H1"], ln2_g, gm["dX"], eps)
    dH1 = dZ + g2["dx"]
    ga = attention_backward(f["LN1"]["y"], Wqkv, Wo, dH1, B, S, causal)
    g1 = layer_norm_backward(_f64(X), ln1_g, ga["dX"], eps)
    return {"dX": dH1 + g1["dx"], "dln1_g": g1["dgamma"], "dln1_b": g1["dbeta"], "dWqkv": ga["dWqkv"],
            "dWo": ga["dWo"], "dln2_g": g2["dgamma"], "dln2_b": g2["dbeta"], "dW1s": gm["dW1s"],
            "dW2s": gm["dW2s"], "dH1": dH1}


def prenorm_layer_forward_rows(X, ln1_g, ln1_b, Wqkv, Wo, ln2_g, ln2_b, W1s, W2s, B: int, S: int, rows,
                               causal: bool = True, eps: float = LN_EPS, store=None) -> dict:
    """H1[rows] and Z[rows] of :func:`prenorm_layer_forward`: LayerNorm, the MLP and
    the residuals act row by row; only the attention needs the other rows (its
    keys and values), which :func:`attention_forward_rows` provides.

    ``store`` (default: none) is applied to the tensors a layer implementation keeps
    in memory between its kernels outside the attention core (LN1(X), H1, LN2(H1),
    the MLP activation); the tests pass a rounding to the storage type to measure
    the error that storage alone causes.  Without it this is the exact definition."""
    st = store or _keep
    X = _f64(X)
    rows = np.asarray(rows, dtype=np.int64)
    l1 = st(layer_norm(X, ln1_g, ln1_b, eps)["y"])
    H1 = st(X[rows] + attention_forward_rows(l1, Wqkv, Wo, B, S, rows, causal)["Z"])
    m = mlp_forward(st(layer_norm(H1, ln2_g, ln2_b, eps)["y"]), W1s, W2s)
    Z = H1 + (matmul(st(concat_columns(m["A"])), stack_rows(W2s)) if store else m["Z"])
    return {"H1": H1, "Z": Z}


# --------------------------------------------------------------------------
# Grouped-query attention (named on wangyu 张量并行 §注意力机制中的张量并行 next to
# MHA; the page gives no formula).  Reading: H query heads share Hkv key/value
# heads, query head j using key/value head j // (H / Hkv) (consecutive query
# heads form a group); the head split of the same section puts query heads
# i*H/N .. (i+1)*H/N-1 and key/value heads i*Hkv/N .. (i+1)*Hkv/N-1 on shard i,
# which keeps every group on one shard when N divides Hkv.
# --------------------------------------------------------------------------
def unpack_qkv_gqa(Wqkv, Hkv: int, d: int) -> tuple:
    """Shard-major [N][h][(H/N + 2 Hkv/N) d] (shard i: its query heads, then its
    key heads, then its value heads, each head d columns) -> unsharded Wq [h][H d],
    Wk [h][Hkv d], Wv [h][Hkv d]."""
    W = _f64(Wqkv)
    n, h, cols = W.shape
    kvn = Hkv // n
    hn = cols // d - 2 * kvn
    Wq = np.concatenate([W[i, :, :hn * d] for i in range(n)], axis=1)
    Wk = np.concatenate([W[i, :, hn * d:(hn + kvn) * d] for i in range(n)], axis=1)
    Wv = np.concatenate([W[i, :, (hn + kvn) * d:] for i in range(n)], axis=1)
    return Wq, Wk, Wv


def pack_qkv_gqa(Wq, Wk, Wv, n: int, d: int) -> np.ndarray:
    """Inverse of :func:`unpack_qkv_gqa`."""
    qn, kn = Wq.shape[1] // n, Wk.shape[1] // n
    return np.stack([np.concatenate([_f64(Wq)[:, i * qn:(i + 1) * qn], _f64(Wk)[:, i * kn:(i + 1) * kn],
                                     _f64(Wv)[:, i * kn:(i + 1) * kn]], axis=1) for i in range(n)])


def gqa_attention_forward(X, Wqkv, Wo, B: int, S: int, H: int, Hkv: int, causal: bool = True) -> dict:
    """Per batch b and query head j, with c = j // (H / Hkv):
        head_j = softmax(mask(Q_j K_c^T / sqrt(d))) V_c,  Z = concat_j(head_j) Wo.
    Returns Z, O (shard layout [N][T][H/N d]), LSE [B][H][S] and Q, K, V unsharded."""
    X = _f64(X)
    n = Wqkv.shape[0]
    d = Wo.shape[1] * n // H
    g = H // Hkv
    T = B * S
    Wq, Wk, Wv = unpack_qkv_gqa(Wqkv, Hkv, d)
    Q, K, V = matmul(X, Wq), matmul(X, Wk), matmul(X, Wv)
    O = np.zeros((T, H * d))
    LSE = np.zeros((B, H, S))
    for b in range(B):
        r = slice(b * S, (b + 1) * S)
        for j in range(H):
            c, kc = slice(j * d, (j + 1) * d), slice((j // g) * d, (j // g + 1) * d)
            P, lse = _softmax_rows(_causal_scores(Q[r, c], K[r, kc], d, causal))
            O[r, c] = matmul(P, V[r, kc])
            LSE[b, j] = lse
    Z = matmul(O, stack_rows(Wo))
    return {"Z": Z, "O": np.ascontiguousarray(O.reshape(T, n, -1).transpose(1, 0, 2)), "LSE": LSE,
            "Q": Q, "K": K, "V": V}


def gqa_attention_backward(X, Wqkv, Wo, dZ, B: int, S: int, H: int, Hkv: int, causal: bool = True) -> dict:
    """Gradients of <dZ, Z> for :func:`gqa_attention_forward`: each query head's
    softmax Jacobian as in :func:`attention_backward`; a key/value head's gradient
    is the sum over the query heads of its group."""
    X, dZ = _f64(X), _f64(dZ)
    n = Wqkv.shape[0]
    d = Wo.shape[1] * n // H
    g = H // Hkv
    T = B * S
    Wq, Wk, Wv = unpack_qkv_gqa(Wqkv, Hkv, d)
    Wo_full = stack_rows(Wo)
    Q, K, V = matmul(X, Wq), matmul(X, Wk), matmul(X, Wv)
    O = np.zeros((T, H * d))
    dO = matmul(dZ, Wo_full.T)
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    for b in range(B):
        r = slice(b * S, (b + 1) * S)
        for j in range(H):
            c, kc = slice(j * d, (j + 1) * d), slice((j // g) * d, (j // g + 1) * d)
            P, _ = _softmax_rows(_causal_scores(Q[r, c], K[r, kc], d, causal))
            O[r, c] = matmul(P, V[r, kc])
            dV[r, kc] += matmul(P.T, dO[r, c])
            dP = matmul(dO[r, c], V[r, kc].T)
            dS = P * (dP - np.sum(dP * P, axis=1, keepdims=True))
            dQ[r, c] = matmul(dS, K[r, kc]) / math.sqrt(d)
            dK[r, kc] += matmul(dS.T, Q[r, c]) / math.sqrt(d)
    dWo = matmul(O.T, dZ)
    dX = matmul(dQ, Wq.T) + matmul(dK, Wk.T) + matmul(dV, Wv.T)
    return {"dX": dX, "dWqkv": pack_qkv_gqa(matmul(X.T, dQ), matmul(X.T, dK), matmul(X.T, dV), n, d),
            "dWo": split_rows_like(dWo, n)}


def gqa_attention_forward_sharded(X, Wqkv, Wo, B: int, S: int, H: int, Hkv: int, causal: bool = True) -> np.ndarray:
    """Shard by shard: shard i projects its own query and key/value heads with its
    column block of Wqkv, attends within its groups, multiplies by its row block of
    Wo; the all-reduce sums the partial outputs."""
    X = _f64(X)
    n = Wqkv.shape[0]
    d = Wo.shape[1] * n // H
    hn, kvn = H // n, Hkv // n
    g = H // Hkv
    T = B * S
    Z = None
    for i in range(n):
        qkv = matmul(X, _f64(Wqkv[i]))
        q, k, v = qkv[:, :hn * d], qkv[:, hn * d:(hn + kvn) * d], qkv[:, (hn + kvn) * d:]
        Oi = np.zeros((T, hn * d))
        for b in range(B):
            r = slice(b * S, (b + 1) * S)
            for jj in range(hn):
                c, kc = slice(jj * d, (jj + 1) * d), slice((jj // g) * d, (jj // g + 1) * d)
                P, _ = _softmax_rows(_causal_scores(q[r, c], k[r, kc], d, causal))
                Oi[r, c] = matmul(P, v[r, kc])
        part = matmul(Oi, Wo[i])
        Z = part if Z is None else Z + part
    return Z


# --------------------------------------------------------------------------
# Tensor + sequence parallelism (zouht 张量并行 §2.2.2 与序列并行结合, §2.3): outside
# the TP blocks the activations are split along the sequence, (batch, seq, hidden)
# -> N x (batch, seq/N, hidden); entering a block an all-gather (g) rebuilds the
# full sequence, leaving it a reduce-scatter (g*) sums the shards' partial outputs
# and hands each sequence shard its rows.
# --------------------------------------------------------------------------
def to_seq_shards(X, B: int, S: int, n: int) -> np.ndarray:
    """[B*S][h] (token t = b*S + s) -> [n][B][S/n][h]: shard c holds positions
    c*S/n .. (c+1)*S/n - 1 of every sequence."""
    X = _f64(X)
    return np.ascontiguousarray(X.reshape(B, n, S // n, -1).transpose(1, 0, 2, 3))


def from_seq_shards(Xs) -> np.ndarray:
    """Inverse of :func:`to_seq_shards`."""
    Xs = _f64(Xs)
    n, B, L, h = Xs.shape
    return np.ascontiguousarray(Xs.transpose(1, 0, 2, 3).reshape(B * n * L, h))


def _all_gather_seq(shards):
    """g: every shard's rows, concatenated along the sequence."""
    return from_seq_shards(np.stack(shards))


def _reduce_scatter_seq(partials, B: int, S: int, n: int):
    """g*: the sum of the tensor shards' partial outputs, each sequence shard
    receiving its own rows."""
    total = partials[0]
    for p in partials[1:]:
        total = total + p
    return list(to_seq_shards(total, B, S, n))


def sp_prenorm_layer_forward(Xs, ln1_g, ln1_b, Wqkv, Wo, ln2_g, ln2_b, W1s, W2s, B: int, S: int,
                             causal: bool = True, eps: float = LN_EPS) -> dict:
    """:func:`prenorm_layer_forward` in the sequence-parallel form, step by step:
    LayerNorm and the residual on each sequence shard, g before each block, the
    block's per-tensor-shard partial outputs, g* after it.  Xs is [N][B][S/N][h];
    returns Z and H1 in the same layout."""
    n = Wqkv.shape[0]
    xs = [_f64(x) for x in Xs]
    ln1 = [layer_norm(x.reshape(-1, x.shape[-1]), ln1_g, ln1_b, eps)["y"].reshape(x.shape) for x in xs]
    full = _all_gather_seq(ln1)
    # attention block: tensor shard i holds heads i*H/N .. and Wo's rows for them
    a = attention_forward(full, Wqkv, Wo, B, S, causal)
    Wo_rows = np.asarray(Wo)
    parts = [matmul(a["O"][i], Wo_rows[i]) for i in range(n)]
    h1 = [x + r for x, r in zip(xs, _reduce_scatter_seq(parts, B, S, n))]
    ln2 = [layer_norm(x.reshape(-1, x.shape[-1]), ln2_g, ln2_b, eps)["y"].reshape(x.shape) for x in h1]
    full2 = _all_gather_seq(ln2)
    m = mlp_forward(full2, W1s, W2s)
    parts2 = [matmul(m["A"][i], _f64(W2s[i])) for i in range(n)]
    z = [x + r for x, r in zip(h1, _reduce_scatter_seq(parts2, B, S, n))]
    return {"Z": np.stack(z), "H1": np.stack(h1)}


def sp_prenorm_layer_backward(Xs, ln1_g, ln1_b, Wqkv, Wo, ln2_g, ln2_b, W1s, W2s, dZs, B: int, S: int,
                              causal: bool = True, eps: float = LN_EPS) -> dict:
    """Gradients of <dZs, Z> for the sequence-parallel form.  The form computes the
    same function of the same parameters, only with the activations laid out by
    sequence shard, so the weight and LayerNorm gradients are those of the plain
    layer and dX comes back in the shard layout (in the backward, g becomes a
    reduce-scatter and g* an all-gather, the transposes of the forward's)."""
    X = from_seq_shards(Xs)
    g = prenorm_layer_backward(X, ln1_g, ln1_b, Wqkv, Wo, ln2_g, ln2_b, W1s, W2s, from_seq_shards(dZs), B, S,
                               causal, eps)
    n = Wqkv.shape[0]
    out = {k: v for k, v in g.items() if k not in ("dX", "dH1")}
    out["dX"] = to_seq_shards(g["dX"], B, S, n)
    return out
