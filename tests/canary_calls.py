"""Every C-ABI call on ragged shapes with each output, save buffer and workspace
placed between guard bands of a known byte pattern; after the calls the bands are
checked, so a write past either end of any buffer is caught.  Used by
test_gpu_canary.py, in-process (release library) and in a fresh process with
TPBLOCK_LIB pointing at the bounds-checked debug build."""
from __future__ import annotations

import torch

import tensor_transformer_block_gb300 as tp
from tensor_transformer_block_gb300 import inputs

GUARD = 4096      # bytes on each side (keeps 256-byte alignment of the buffer)
PATTERN = 0xA5


class Guarded:
    """A device buffer of ``shape`` and ``dtype`` inside two guard bands."""

    def __init__(self, shape, dtype, dev="cuda"):
        numel = 1
        for s in shape:
            numel *= int(s)
        self.nbytes = numel * torch.empty((), dtype=dtype).element_size()
        self.full = torch.full((2 * GUARD + (self.nbytes + 15) // 16 * 16,), PATTERN, dtype=torch.uint8, device=dev)
        self.t = self.full[GUARD:GUARD + self.nbytes].view(dtype).view(*shape)

    def intact(self) -> bool:
        return bool((self.full[:GUARD] == PATTERN).all()) and bool((self.full[GUARD + self.nbytes:] == PATTERN).all())


def _ws(nbytes):
    return Guarded((max(int(nbytes), 16),), torch.uint8)


def run_calls() -> list:
    """Runs every call once; returns the names of buffers whose guards were hit."""
    torch.manual_seed(0)
    bf = torch.bfloat16
    bufs = {}

    def g(name, shape, dtype=bf):
        bufs[name] = Guarded(shape, dtype)
        return bufs[name].t

    # MLP block (ragged T, h, f/N; N = 3), bf16 and fp32
    T, h, f, N = 333, 200, 264, 3
    m = {k: v.cuda() for k, v in inputs.mlp_inputs(T, h, f, N, seed=1).items()}
    ws = _ws(tp.tp_mlp_workspace_bytes(tp.TP_BF16, T, h, f, N))
    bufs["mlp.ws"] = ws
    Y, A, Z = g("mlp.Y", (N, T, f // N)), g("mlp.A", (N, T, f // N)), g("mlp.Z", (T, h))
    tp.tp_mlp_fwd(tp.TP_BF16, T, h, f, N, m["X"], m["W1s"], m["W2s"], Y, A, Z, ws.t)
    tp.tp_mlp_bwd(tp.TP_BF16, T, h, f, N, m["X"], m["W1s"], m["W2s"], Y, A, m["dZ"], g("mlp.dX", (T, h)),
                  g("mlp.dW1s", (N, h, f // N)), g("mlp.dW2s", (N, f // N, h)), ws.t)
    tp.tp_mlp_fwd_noalloc(tp.TP_BF16, T, h, f, N, m["X"], m["W1s"], m["W2s"], g("mlp.Z_noalloc", (T, h)))
    # a shape whose row-parallel GEMMs split K (fp32 partials in the workspace)
    Ts, hs, fs, Ns = 1000, 520, 2048, 2
    ms = {k: v.cuda() for k, v in inputs.mlp_inputs(Ts, hs, fs, Ns, seed=9).items()}
    wss = _ws(tp.tp_mlp_workspace_bytes(tp.TP_BF16, Ts, hs, fs, Ns))
    bufs["mlp_split.ws"] = wss
    Ys, As = g("mlp_split.Y", (Ns, Ts, fs // Ns)), g("mlp_split.A", (Ns, Ts, fs // Ns))
    tp.tp_mlp_fwd(tp.TP_BF16, Ts, hs, fs, Ns, ms["X"], ms["W1s"], ms["W2s"], Ys, As, g("mlp_split.Z", (Ts, hs)), wss.t)
    tp.tp_mlp_bwd(tp.TP_BF16, Ts, hs, fs, Ns, ms["X"], ms["W1s"], ms["W2s"], Ys, As, ms["dZ"],
                  g("mlp_split.dX", (Ts, hs)), g("mlp_split.dW1s", (Ns, hs, fs // Ns)),
                  g("mlp_split.dW2s", (Ns, fs // Ns, hs)), wss.t)
    m32 = {k: v.cuda() for k, v in inputs.mlp_inputs(64, 256, 1024, 2, dtype="f32", seed=2, backward=False).items()}
    ws32 = _ws(tp.tp_mlp_workspace_bytes(tp.TP_F32, 64, 256, 1024, 2))
    bufs["mlp32.ws"] = ws32
    tp.tp_mlp_fwd(tp.TP_F32, 64, 256, 1024, 2, m32["X"], m32["W1s"], m32["W2s"], None, None,
                  g("mlp32.Z", (64, 256), torch.float32), ws32.t)

    # gated MLP
    gi = {k: v.cuda() for k, v in inputs.gmlp_inputs(T, h, f, N, seed=3).items()}
    gws = _ws(tp.tp_gmlp_workspace_bytes(tp.TP_BF16, T, h, f, N))
    bufs["gmlp.ws"] = gws
    GU, GA = g("gmlp.GU", (N, T, 2, f // N)), g("gmlp.A", (N, T, f // N))
    tp.tp_gmlp_fwd(tp.TP_BF16, T, h, f, N, gi["X"], gi["Wgus"], gi["Wds"], GU, GA, g("gmlp.Z", (T, h)), gws.t)
    tp.tp_gmlp_bwd(tp.TP_BF16, T, h, f, N, gi["X"], gi["Wgus"], gi["Wds"], GU, GA, gi["dZ"], g("gmlp.dX", (T, h)),
                   g("gmlp.dWgus", tuple(gi["Wgus"].shape)), g("gmlp.dWds", tuple(gi["Wds"].shape)), gws.t)

    # attention block and GQA (ragged S = 200; d = 64)
    B, S, ha, H, Hkv, d, Na = 2, 200, 256, 4, 2, 64, 2
    Ta = B * S
    a = {k: v.cuda() for k, v in inputs.attn_inputs(B, S, ha, H, d, Na, seed=4).items()}
    aws = _ws(tp.tp_attn_workspace_bytes(tp.TP_BF16, B, S, ha, H, d, Na))
    bufs["attn.ws"] = aws
    QKV, O_ = g("attn.QKV", (Na, Ta, 3 * H // Na * d)), g("attn.O", (Na, Ta, H // Na * d))
    LSE = g("attn.LSE", (B, H, S), torch.float32)
    tp.tp_attn_fwd(tp.TP_BF16, B, S, ha, H, d, Na, True, a["X"], a["Wqkv"], a["Wo"], QKV, O_, LSE, g("attn.Z", (Ta, ha)),
                   aws.t)
    tp.tp_attn_bwd(tp.TP_BF16, B, S, ha, H, d, Na, True, a["X"], a["Wqkv"], a["Wo"], QKV, O_, LSE, a["dZ"],
                   g("attn.dX", (Ta, ha)), g("attn.dWqkv", tuple(a["Wqkv"].shape)), g("attn.dWo", tuple(a["Wo"].shape)),
                   aws.t)
    q = {k: v.cuda() for k, v in inputs.gqa_inputs(B, S, ha, H, Hkv, d, Na, seed=5).items()}
    qws = _ws(tp.tp_gqa_workspace_bytes(tp.TP_BF16, B, S, ha, H, Hkv, d, Na))
    bufs["gqa.ws"] = qws
    W = (H + 2 * Hkv) * d // Na
    QKVg, Og = g("gqa.QKV", (Na, Ta, W)), g("gqa.O", (Na, Ta, H // Na * d))
    LSEg = g("gqa.LSE", (B, H, S), torch.float32)
    tp.tp_gqa_fwd(tp.TP_BF16, B, S, ha, H, Hkv, d, Na, True, q["X"], q["Wqkv"], q["Wo"], QKVg, Og, LSEg,
                  g("gqa.Z", (Ta, ha)), qws.t)
    tp.tp_gqa_bwd(tp.TP_BF16, B, S, ha, H, Hkv, d, Na, True, q["X"], q["Wqkv"], q["Wo"], QKVg, Og, LSEg, q["dZ"],
                  g("gqa.dX", (Ta, ha)), g("gqa.dWqkv", tuple(q["Wqkv"].shape)), g("gqa.dWo", tuple(q["Wo"].shape)),
                  qws.t)

    # the attention + MLP layer, the pre-norm layer and its sequence-parallel form
    fl = 528
    li = {k: v.cuda() for k, v in inputs.layer_inputs(B, S, ha, H, d, fl, Na, seed=6).items()}
    sv = _ws(tp.tp_attn_mlp_save_bytes(tp.TP_BF16, B, S, ha, H, d, fl, Na))
    lw = _ws(tp.tp_attn_mlp_workspace_bytes(tp.TP_BF16, B, S, ha, H, d, fl, Na))
    bufs["attn_mlp.save"], bufs["attn_mlp.ws"] = sv, lw
    tp.tp_attn_mlp_fwd(tp.TP_BF16, B, S, ha, H, d, fl, Na, True, li["X"], li["Wqkv"], li["Wo"], li["W1s"], li["W2s"],
                       sv.t, g("attn_mlp.Z", (Ta, ha)))
    tp.tp_attn_mlp_bwd(tp.TP_BF16, B, S, ha, H, d, fl, Na, True, li["X"], li["Wqkv"], li["Wo"], li["W1s"], li["W2s"],
                       sv.t, li["dZ"], g("attn_mlp.dX", (Ta, ha)), g("attn_mlp.dWqkv", tuple(li["Wqkv"].shape)),
                       g("attn_mlp.dWo", tuple(li["Wo"].shape)), g("attn_mlp.dW1s", tuple(li["W1s"].shape)),
                       g("attn_mlp.dW2s", tuple(li["W2s"].shape)), lw.t)
    for name, Sl, fn in (("layer", S, (tp.tp_layer_fwd, tp.tp_layer_bwd)),
                         ("sp_layer", 256, (tp.tp_sp_layer_fwd, tp.tp_sp_layer_bwd))):
        p = {k: v.cuda() for k, v in inputs.prenorm_inputs(B, Sl, ha, H, d, fl, Na, seed=7).items()}
        Tl = B * Sl
        sv = _ws(tp.tp_layer_save_bytes(tp.TP_BF16, B, Sl, ha, H, d, fl, Na))
        lw = _ws(tp.tp_layer_workspace_bytes(tp.TP_BF16, B, Sl, ha, H, d, fl, Na))
        bufs[name + ".save"], bufs[name + ".ws"] = sv, lw
        X, dZ = p["X"], p["dZ"]
        if name == "sp_layer":
            X, dZ = inputs.to_seq_shards(X, B, Sl, Na), inputs.to_seq_shards(dZ, B, Sl, Na)
        fn[0](tp.TP_BF16, B, Sl, ha, H, d, fl, Na, True, 1e-5, X, p["ln1_g"], p["ln1_b"], p["Wqkv"], p["Wo"],
              p["ln2_g"], p["ln2_b"], p["W1s"], p["W2s"], sv.t, g(name + ".Z", tuple(X.shape)))
        grads = {k: g(name + ".d" + k, tuple(p[k].shape)) for k in
                 ("ln1_g", "ln1_b", "Wqkv", "Wo", "ln2_g", "ln2_b", "W1s", "W2s")}
        fn[1](tp.TP_BF16, B, Sl, ha, H, d, fl, Na, True, X, p["ln1_g"], p["Wqkv"], p["Wo"], p["ln2_g"], p["W1s"],
              p["W2s"], sv.t, dZ, g(name + ".dX", tuple(X.shape)), grads["ln1_g"], grads["ln1_b"], grads["Wqkv"],
              grads["Wo"], grads["ln2_g"], grads["ln2_b"], grads["W1s"], grads["W2s"], lw.t)

    # LayerNorm on its own (ragged h)
    ln = {k: v.cuda() for k, v in inputs.ln_inputs(77, 8200, seed=8).items()}
    mean, rstd = g("ln.mean", (77,), torch.float32), g("ln.rstd", (77,), torch.float32)
    tp.tp_layernorm_fwd(tp.TP_BF16, 77, 8200, 1e-5, ln["X"], ln["gamma"], ln["beta"], g("ln.Y", (77, 8200)), mean, rstd)
    lnws = _ws(tp.tp_layernorm_workspace_bytes(tp.TP_BF16, 77, 8200))
    bufs["ln.ws"] = lnws
    tp.tp_layernorm_bwd(tp.TP_BF16, 77, 8200, ln["X"], ln["gamma"], mean, rstd, ln["dY"], ln["dR"],
                        g("ln.dX", (77, 8200)), g("ln.dgamma", (8200,)), g("ln.dbeta", (8200,)), lnws.t)
    torch.cuda.synchronize()
    return [k for k, v in bufs.items() if not v.intact()]


if __name__ == "__main__":
    # child process: the library chosen by TPBLOCK_LIB; prints the result
    torch.cuda.set_device(0)
    hit = run_calls()
    st = tp.tp_sync_status()
    print(f"guards hit: {hit}; sync status: {st}; library: {tp.LIB_PATH}")
    raise SystemExit(0 if not hit and st == 0 else 1)
