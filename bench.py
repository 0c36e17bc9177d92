#!/usr/bin/env python3
"""Throughput of the tensor-parallel block on GB300 through libtpblock.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step is one pass of the block over one batch of synthetic input: for the
default workload (MLP block, T=8192 tokens, h=4096, f=16384, N=8 logical shards)
the forward and the backward call.  The metric is algorithmic TFLOP/s (2 flop per
multiply-add; the causal half of attention only; softmax/GeLU not counted).
Prints one JSON line on rank 0.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the shards are logical; there is no data-path collective): value = all ranks'
flops / the slowest rank's time ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "TFLOP/s (fwd+bwd) of TP-sharded MLP/attention block, 1 GB300; % BF16 peak"
# Timed regions at least this long run at the power-capped clock: their roofline
# fraction is taken against the sustained GEMM peak, shorter ones against the burst.
SUSTAINED_REGION_MS = 1000.0
# NVIDIA's dense bf16 tensor rate per GB300 GPU: the HGX B300 specification table
# (www.nvidia.com/en-us/data-center/hgx/) gives 36 PFLOPS FP16/BF16 for eight GPUs
# with 2:4 sparsity, i.e. 4.5 sparse and 2.25 dense PFLOP/s per GPU.
NOMINAL_DENSE_BF16_TFLOPS = 2250.0
NOMINAL_SOURCE = ("NVIDIA HGX B300 specifications (www.nvidia.com/en-us/data-center/hgx/): 36 PFLOPS FP16/BF16 "
                  "per 8 GPUs with 2:4 sparsity = 2.25 PFLOP/s dense per GPU")
DEFAULT_WORKLOAD = "mlp_bf16_T8192_h4096_f16384_N8"

# DRAM bytes (read + write) per launch from one ncu capture of the kernel, with
# the sha256 of the kernel source it was taken on; reported as null once the
# source has changed.
NCU_TRAFFIC: dict = {
    k: {"bytes": v, "sha": "e001161d2256cb7b", "workload": "mlp_bf16_T8192_h4096_f16384_N8"}
    for k, v in {
        "mlp.fc1_col_gemm_gelu": 1034888960,
        "mlp.fc2_row_gemm_shard_sum": 1446203648,
        "mlp.bwd_dA_gemm_dgelu": 1178239488,
        "mlp.bwd_dW2_gemm": 1337640192,
        "mlp.bwd_dW1_gemm": 1341266432,
        "mlp.bwd_dX_row_gemm_shard_sum": 1446592768,
    }.items()
}

def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return {"bf16_tflops": float(d["bf16_tflops"]), "bf16_tflops_sustained": float(d["bf16_tflops_sustained"]),
                "hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


# ------------------------------------------------------------------ flop counts
def kernel_flops(w) -> dict:
    """Algorithmic flops per launch of each kernel kind of the workload."""
    T, h, f = w.T, w.h, w.f
    out = {}
    if w.kind in ("mlp", "layer", "lnlayer", "splayer"):
        g = 2.0 * T * h * f
        out.update({"mlp.fc1_col_gemm_gelu": g, "mlp.fc2_row_gemm_shard_sum": g, "mlp.bwd_dA_gemm_dgelu": g,
                    "mlp.bwd_dW2_gemm": g, "mlp.bwd_dW1_gemm": g, "mlp.bwd_dX_row_gemm_shard_sum": g,
                    "mlp.f32_fc1_col_gemm_gelu": g, "mlp.f32_fc2_row_gemm": g})
    if w.kind == "gmlp":
        g = 2.0 * T * h * f
        out.update({"gmlp.fc1_col_gemm_swiglu": 2 * g, "gmlp.fc2_row_gemm_shard_sum": g,
                    "gmlp.bwd_dA_gemm_dswiglu": g, "gmlp.bwd_dWd_gemm": g, "gmlp.bwd_dWgu_gemm": 2 * g,
                    "gmlp.bwd_dX_row_gemm_shard_sum": 2 * g})
    if w.kind == "gqa":
        Hd, qkv = w.H * w.d, (w.H + 2 * w.Hkv) * w.d
        pairs = w.B * w.H * (w.S * w.S if w.causal else 2 * w.S * w.S) * w.d
        out.update({"attn.qkv_col_gemm": 2.0 * T * h * qkv, "attn.core_fwd": 2.0 * pairs,
                    "attn.out_row_gemm_shard_sum": 2.0 * T * Hd * h, "attn.bwd_dO_gemm": 2.0 * T * h * Hd,
                    "attn.bwd_dWo_gemm": 2.0 * T * Hd * h, "attn.bwd_core_dkdv": 3.0 * pairs,
                    "attn.bwd_core_dq": 1.0 * pairs, "attn.bwd_dWqkv_gemm": 2.0 * T * h * qkv,
                    "attn.bwd_dX_row_gemm_shard_sum": 2.0 * T * qkv * h})
    if w.kind in ("attn", "layer", "lnlayer", "splayer"):
        Hd = w.H * w.d
        pairs = w.B * w.H * (w.S * w.S if w.causal else 2 * w.S * w.S) * w.d  # (causal half) x d
        out.update({"attn.qkv_col_gemm": 2.0 * T * h * 3 * Hd, "attn.core_fwd": 2.0 * pairs,
                    "attn.out_row_gemm_shard_sum": 2.0 * T * Hd * h, "attn.bwd_dO_gemm": 2.0 * T * h * Hd,
                    "attn.bwd_dWo_gemm": 2.0 * T * Hd * h, "attn.bwd_core_dkdv": 3.0 * pairs,
                    "attn.bwd_core_dq": 1.0 * pairs, "attn.bwd_dWqkv_gemm": 2.0 * T * h * 3 * Hd,
                    "attn.bwd_dX_row_gemm_shard_sum": 2.0 * T * 3 * Hd * h})
    return out


# ------------------------------------------------------------ replicas (N > 1)
def dist_env() -> tuple:
    """(world size, rank, local rank) from the launcher's environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of every rank's x (the whole job ends with its slowest rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step: float, steps: int, ms: float, world: int) -> float:
    """Every rank runs the same step on its own GPU (independent replicas, weak
    scaling): the job does world x steps steps in the slowest rank's time."""
    return world * flops_per_step * steps / (ms / 1e3) / 1e12


def step_flops(w) -> float:
    T, h, f = w.T, w.h, w.f
    tot = 0.0
    if w.kind in ("mlp", "layer", "lnlayer", "splayer"):
        tot += (12.0 if w.backward else 4.0) * T * h * f
    if w.kind == "gmlp":
        tot += (18.0 if w.backward else 6.0) * T * h * f
    if w.kind == "gqa":
        Hd, qkv = w.H * w.d, (w.H + 2 * w.Hkv) * w.d
        core = 2.0 * w.B * w.H * (w.S * w.S if w.causal else 2 * w.S * w.S) * w.d
        tot += 2.0 * T * h * qkv + 2.0 * T * Hd * h + core
        if w.backward:
            tot += 4.0 * T * h * Hd + 4.0 * T * h * qkv + 2.0 * core
    if w.kind in ("attn", "layer", "lnlayer", "splayer"):
        Hd = w.H * w.d
        core = 2.0 * w.B * w.H * (w.S * w.S if w.causal else 2 * w.S * w.S) * w.d
        tot += 8.0 * T * h * Hd + core
        if w.backward:
            tot += 16.0 * T * h * Hd + 2.0 * core
    return tot


def describe(w) -> str:
    if w.kind == "mlp":
        return (f"MLP block {'fwd+bwd' if w.backward else 'fwd'}, {w.dtype}, T={w.T} tokens, h={w.h}, f={w.f}, "
                f"N={w.N} logical shards")
    if w.kind == "gmlp":
        return (f"gated (SwiGLU) MLP block {'fwd+bwd' if w.backward else 'fwd'}, {w.dtype}, T={w.T} tokens, "
                f"h={w.h}, f={w.f} (gate and up each), N={w.N} logical shards")
    if w.kind == "gqa":
        return (f"grouped-query attention block {'fwd+bwd' if w.backward else 'fwd'}, {w.dtype}, B={w.B} x S={w.S}, "
                f"h={w.h}, {w.H} query heads over {w.Hkv} key/value heads x d={w.d}, "
                f"{'causal' if w.causal else 'full'}, N={w.N} logical shards")
    if w.kind == "attn":
        return (f"self-attention block fwd, {w.dtype}, B={w.B} x S={w.S}, h={w.h}, {w.H} heads x d={w.d}, "
                f"{'causal' if w.causal else 'full'}, N={w.N} logical shards")
    if w.kind == "splayer":
        return (f"pre-norm layer in the tensor + sequence parallel form (X, Z, dZ, dX in {w.N} sequence shards of "
                f"{w.S // w.N} positions) fwd+bwd, {w.dtype}, B={w.B} x S={w.S}, h={w.h}, {w.H} heads x d={w.d}, "
                f"f={w.f}, causal, N={w.N} logical shards; LayerNorm and residual adds not counted in the flops")
    if w.kind == "lnlayer":
        return (f"pre-norm layer (LN, attention, residual, LN, MLP, residual) fwd+bwd, {w.dtype}, B={w.B} x "
                f"S={w.S}, h={w.h}, {w.H} heads x d={w.d}, f={w.f}, causal, N={w.N} logical shards; LayerNorm and "
                f"residual adds not counted in the flops")
    return (f"attention + MLP layer fwd+bwd (tp_attn_mlp_fwd/bwd: the attention output stays in fp16 between "
            f"the blocks), {w.dtype}, B={w.B} x S={w.S}, h={w.h}, {w.H} heads x d={w.d}, f={w.f}, causal, "
            f"N={w.N} logical shards")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples (every 50 ms) of SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if self.gpu_id is not None:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
            return self
        # nvidia-smi's start-up must not overlap the timed work: wait for its first sample
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5.0 and self.proc.poll() is None:
            time.sleep(0.02)
        self.skip = len(self.lines)
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self) -> dict | None:
        rows = []
        lines = self.lines[getattr(self, "skip", 0):] or self.lines
        for ln in lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]), "power": float(parts[3]),
                             "hw": parts[5], "hwt": parts[6], "swt": parts[7], "swpc": parts[8]})
            except ValueError:
                continue
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                              ("swpc", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "power_w_max": max(r["power"] for r in rows)}


def clocks_rejected(c: dict | None) -> bool:
    if not c:
        return False
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    if bad & set(c["reasons"]):
        return True
    # stuck well below max with no reason at all: a leftover clock lock
    return c["sm_mhz"] < 0.5 * c["sm_max_mhz"] and not c["reasons"]


# ------------------------------------------------------------------ oracle arm
def oracle_step(w, inp_np: dict, rows: int) -> float:
    """Runs the fp64 oracle as it stands on the first ``rows`` tokens of the
    workload (or the first ``rows`` sequence positions of batch 0 for attention);
    returns the algorithmic flops that sample stands for."""
    from oracle import tp_oracle as O
    if w.kind == "mlp":
        X, dZ = inp_np["X"][:rows], inp_np.get("dZ")
        O.mlp_forward(X, inp_np["W1s"], inp_np["W2s"])
        if w.backward:
            O.mlp_backward(X, inp_np["W1s"], inp_np["W2s"], dZ[:rows])
        return (12.0 if w.backward else 4.0) * rows * w.h * w.f
    if w.kind == "gmlp":
        X, dZ = inp_np["X"][:rows], inp_np.get("dZ")
        O.gated_mlp_forward(X, inp_np["Wgus"], inp_np["Wds"])
        if w.backward:
            O.gated_mlp_backward(X, inp_np["Wgus"], inp_np["Wds"], dZ[:rows])
        return (18.0 if w.backward else 6.0) * rows * w.h * w.f
    import dataclasses
    sub = dataclasses.replace(w, B=1, S=rows, T=rows)
    X = inp_np["X"][:rows]
    if w.kind == "attn":
        O.attention_forward(X, inp_np["Wqkv"], inp_np["Wo"], 1, rows, w.causal)
    elif w.kind == "gqa":
        O.gqa_attention_forward(X, inp_np["Wqkv"], inp_np["Wo"], 1, rows, w.H, w.Hkv, w.causal)
        if w.backward:
            O.gqa_attention_backward(X, inp_np["Wqkv"], inp_np["Wo"], inp_np["dZ"][:rows], 1, rows, w.H, w.Hkv,
                                     w.causal)
    elif w.kind in ("lnlayer", "splayer"):
        args = (X, inp_np["ln1_g"], inp_np["ln1_b"], inp_np["Wqkv"], inp_np["Wo"], inp_np["ln2_g"], inp_np["ln2_b"],
                inp_np["W1s"], inp_np["W2s"])
        O.prenorm_layer_forward(*args, 1, rows, True)
        O.prenorm_layer_backward(*args, inp_np["dZ"][:rows], 1, rows, True)
    else:
        O.layer_forward(X, inp_np["Wqkv"], inp_np["Wo"], inp_np["W1s"], inp_np["W2s"], 1, rows, True)
        O.layer_backward(X, inp_np["Wqkv"], inp_np["Wo"], inp_np["W1s"], inp_np["W2s"], inp_np["dZ"][:rows], 1,
                         rows, True)
    return step_flops(sub)


def oracle_inputs(w) -> dict:
    from tensor_transformer_block_gb300 import inputs
    import torch
    inp = inputs.workload_inputs(w)
    return {k: v.to(torch.float64).numpy() for k, v in inp.items()}


def oracle_cores() -> int:
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


def calibrate_rows(w, inp_np, target_s: float) -> int:
    rows = 128 if w.kind not in ("mlp", "gmlp") else 256
    t0 = time.perf_counter()
    oracle_step(w, inp_np, rows)
    dt = max(time.perf_counter() - t0, 1e-3)
    limit = w.T if w.kind in ("mlp", "gmlp") else w.S
    return int(max(64, min(limit, rows * target_s / dt)))


def cpu_baseline(w, inp_np, target_s: float = 15.0) -> dict:
    rows = calibrate_rows(w, inp_np, target_s)
    t0 = time.perf_counter()
    fl = oracle_step(w, inp_np, rows)
    dt = time.perf_counter() - t0
    unit = "tokens" if w.kind in ("mlp", "gmlp") else "sequence positions of batch 0"
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": oracle_cores(), "kind": "oracle",
            "sample": f"fp64 oracle on the first {rows} {unit} of the same workload ({dt:.1f} s)",
            "seconds": dt}


def run_reference(args, w) -> None:
    if dist_env()[1] != 0:  # rank 0 alone times the oracle; the other ranks exit without work
        return
    inp_np = oracle_inputs(w)
    rows = calibrate_rows(w, inp_np, 3.0)
    for _ in range(args.warmup):
        oracle_step(w, inp_np, rows)
    t0 = time.perf_counter()
    fl = 0.0
    for _ in range(args.steps):
        fl += oracle_step(w, inp_np, rows)
    dt = time.perf_counter() - t0
    value = fl / dt / 1e12
    unit = "tokens" if w.kind in ("mlp", "gmlp") else "sequence positions of batch 0"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded normals, same draws as the GPU arm)",
            "config": {"workload": w.name, "description": describe(w), "sample_rows_per_step": rows},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle_cores(), "kind": "oracle",
                             "sample": f"each step: fp64 oracle on the first {rows} {unit}"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ library baseline
def library_composition(w, d: dict):
    """(forward function, unsharded weights) of the workload's step composed from
    torch library calls: matmuls, torch's tanh GeLU, SiLU, LayerNorm and
    scaled-dot-product attention.  The shard-major weights are viewed back as the
    unsharded matrices the pages split."""
    import torch.nn.functional as F

    N, h, f, T = w.N, w.h, w.f, w.T

    def cols(Ws):  # [N][rows][c] -> [rows][N*c]: shard i holds columns i*c..
        return Ws.permute(1, 0, 2).reshape(Ws.shape[1], -1)

    def heads(t, nh):  # [T][nh*d] -> [B][nh][S][d]
        return t.view(w.B, w.S, nh, w.d).transpose(1, 2)

    def attention(x, Wq, Wk, Wv, Wo, H, Hkv):
        q, k, v = heads(x @ Wq, H), heads(x @ Wk, Hkv), heads(x @ Wv, Hkv)
        if H != Hkv:
            o = F.scaled_dot_product_attention(q, k, v, is_causal=bool(w.causal), enable_gqa=True)
        else:
            o = F.scaled_dot_product_attention(q, k, v, is_causal=bool(w.causal))
        return o.transpose(1, 2).reshape(T, H * w.d) @ Wo

    def mlp(x, W1, W2):
        return F.gelu(x @ W1, approximate="tanh") @ W2

    def qkv_mha(Wqkv):  # [N][h][3][H/N][d] (same bytes as [N][h][3 H/N d])
        q = Wqkv.reshape(N, h, 3, -1)
        return cols(q[:, :, 0]), cols(q[:, :, 1]), cols(q[:, :, 2])

    p = {}
    if w.kind == "mlp":
        p = {"W1": cols(d["W1s"]), "W2": d["W2s"].reshape(f, h)}
        fwd = lambda x, q: mlp(x, q["W1"], q["W2"])  # noqa: E731
    elif w.kind == "gmlp":
        p = {"Wg": cols(d["Wgus"][:, :, 0]), "Wu": cols(d["Wgus"][:, :, 1]), "Wd": d["Wds"].reshape(f, h)}
        fwd = lambda x, q: (F.silu(x @ q["Wg"]) * (x @ q["Wu"])) @ q["Wd"]  # noqa: E731
    elif w.kind == "gqa":
        hN, kvN = w.H // N, w.Hkv // N
        Wqkv = d["Wqkv"]
        p = {"Wq": cols(Wqkv[:, :, :hN * w.d]), "Wk": cols(Wqkv[:, :, hN * w.d:(hN + kvN) * w.d]),
             "Wv": cols(Wqkv[:, :, (hN + kvN) * w.d:]), "Wo": d["Wo"].reshape(w.H * w.d, h)}
        fwd = lambda x, q: attention(x, q["Wq"], q["Wk"], q["Wv"], q["Wo"], w.H, w.Hkv)  # noqa: E731
    else:
        Wq, Wk, Wv = qkv_mha(d["Wqkv"])
        p = {"Wq": Wq, "Wk": Wk, "Wv": Wv, "Wo": d["Wo"].reshape(w.H * w.d, h)}
        if w.kind == "attn":
            fwd = lambda x, q: attention(x, q["Wq"], q["Wk"], q["Wv"], q["Wo"], w.H, w.H)  # noqa: E731
        else:
            p.update({"W1": cols(d["W1s"]), "W2": d["W2s"].reshape(f, h)})
            if w.kind == "layer":
                def fwd(x, q):
                    return mlp(attention(x, q["Wq"], q["Wk"], q["Wv"], q["Wo"], w.H, w.H), q["W1"], q["W2"])
            else:
                p.update({k: d[k] for k in ("ln1_g", "ln1_b", "ln2_g", "ln2_b")})

                def fwd(x, q):
                    a = F.layer_norm(x, (h,), q["ln1_g"], q["ln1_b"], 1e-5)
                    h1 = x + attention(a, q["Wq"], q["Wk"], q["Wv"], q["Wo"], w.H, w.H)
                    return h1 + mlp(F.layer_norm(h1, (h,), q["ln2_g"], q["ln2_b"], 1e-5), q["W1"], q["W2"])
    return fwd, p


def library_baseline(w, d: dict, X, dZ, steps: int, warmup: int, dev, gpu_id=None) -> dict:
    """The same step composed from torch library calls on the unsharded weights
    (cuBLAS matmuls, torch's elementwise ops and attention, autograd for the
    backward), timed with CUDA events.  Reported beside the kernels' number as
    context; it is not a product path and shares nothing with it but the inputs."""
    import torch

    fwd, p = library_composition(w, d)
    p = {k: v.contiguous().detach().requires_grad_(w.backward) for k, v in p.items()}
    x = X.detach().requires_grad_(w.backward)

    def step():
        if not w.backward:
            with torch.no_grad():
                return fwd(x, p)
        z = fwd(x, p)
        return torch.autograd.grad(z, [x] + list(p.values()), dZ)

    try:
        for _ in range(warmup):
            step()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(gpu_id) as cs:
            e0.record()
            for _ in range(steps):
                step()
            e1.record()
            torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / steps
    except Exception as e:  # a backend torch lacks on this GPU: report, do not fail the run
        return {"unavailable": f"{type(e).__name__}: {str(e)[:160]}"}
    return {"value": step_flops(w) / (ms / 1e3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms, "steps": steps,
            "clocks": cs.summary(),
            "what": "torch library composition of the same step on the unsharded weights (cuBLAS matmuls, "
                    "torch GeLU/SiLU/LayerNorm/scaled_dot_product_attention, autograd backward); context only"}


# ------------------------------------------------------------------ GPU arm
def source_sha(kind: str) -> str:
    f = "gemm_tc.cu" if "gemm" in kind else ("attn_fwd.cu" if kind == "attn.core_fwd" else "attn_bwd.cu")
    p = os.path.join(ROOT, "tensor_transformer_block_gb300", "csrc", f)
    return hashlib.sha256(open(p, "rb").read()).hexdigest()[:16]


def run_gpu(args, w) -> None:
    import torch
    import torch.distributed as dist

    import tensor_transformer_block_gb300 as tp
    from tensor_transformer_block_gb300 import block, inputs

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    tp.load_library()
    if tp.tp_device_check() != 0:
        raise RuntimeError("not an sm_103 GPU")
    tp.tp_set_gemm_tiling(args.gemm_tiling)
    tp.tp_set_launch_overlap(bool(args.launch_overlap))

    inp = inputs.workload_inputs(w)
    inp_tok = inp  # token-major copies (the oracle's layout)
    d = {k: v.to(dev) for k, v in inp.items()}
    stream = torch.cuda.current_stream(dev)
    dt = tp.TP_BF16 if w.dtype == "bf16" else tp.TP_F32
    T, h, f, N = w.T, w.h, w.f, w.N
    buf = {}
    if w.kind == "mlp":
        fN = f // N
        buf["Y"] = torch.empty(N, T, fN, dtype=d["W1s"].dtype, device=dev)
        buf["A"] = torch.empty_like(buf["Y"])
        buf["Z"] = torch.empty(T, h, dtype=d["W1s"].dtype, device=dev)
        buf["dX"] = torch.empty(T, h, dtype=d["W1s"].dtype, device=dev)
        buf["dW1s"] = torch.empty_like(d["W1s"])
        buf["dW2s"] = torch.empty_like(d["W2s"])
        buf["mws"] = block.workspace(tp.tp_mlp_workspace_bytes(dt, T, h, f, N), dev)
    if w.kind == "gmlp":
        fN = f // N
        buf["GU"] = torch.empty(N, T, 2, fN, dtype=torch.bfloat16, device=dev)
        buf["A"] = torch.empty(N, T, fN, dtype=torch.bfloat16, device=dev)
        buf["Z"] = torch.empty(T, h, dtype=torch.bfloat16, device=dev)
        buf["dX"] = torch.empty(T, h, dtype=torch.bfloat16, device=dev)
        buf["dWgus"] = torch.empty_like(d["Wgus"])
        buf["dWds"] = torch.empty_like(d["Wds"])
        buf["gws"] = block.workspace(tp.tp_gmlp_workspace_bytes(dt, T, h, f, N), dev)
    if w.kind == "gqa":
        hN, kvN = w.H // N, w.Hkv // N
        buf["QKV"] = torch.empty(N, T, (hN + 2 * kvN) * w.d, dtype=torch.bfloat16, device=dev)
        buf["O"] = torch.empty(N, T, hN * w.d, dtype=torch.bfloat16, device=dev)
        buf["LSE"] = torch.empty(w.B, w.H, w.S, dtype=torch.float32, device=dev)
        buf["Z"] = torch.empty(T, h, dtype=torch.bfloat16, device=dev)
        buf["dX"] = torch.empty(T, h, dtype=torch.bfloat16, device=dev)
        buf["dWqkv"] = torch.empty_like(d["Wqkv"])
        buf["dWo"] = torch.empty_like(d["Wo"])
        buf["qws"] = block.workspace(tp.tp_gqa_workspace_bytes(dt, w.B, w.S, h, w.H, w.Hkv, w.d, N), dev)
    if w.kind == "splayer":
        # the sequence-parallel layout of the inputs the step consumes
        d["X"] = inputs.to_seq_shards(d["X"], w.B, w.S, N)
        d["dZ"] = inputs.to_seq_shards(d["dZ"], w.B, w.S, N)
        inp = dict(inp, X=inputs.to_seq_shards(inp["X"], w.B, w.S, N), dZ=inputs.to_seq_shards(inp["dZ"], w.B, w.S, N))
    if w.kind in ("lnlayer", "splayer"):
        p = {k: d[k] for k in ("ln1_g", "ln1_b", "Wqkv", "Wo", "ln2_g", "ln2_b", "W1s", "W2s")}
        buf["save"] = block.workspace(tp.tp_layer_save_bytes(dt, w.B, w.S, h, w.H, w.d, f, N), dev)
        buf["lws"] = block.workspace(tp.tp_layer_workspace_bytes(dt, w.B, w.S, h, w.H, w.d, f, N), dev)
        buf["Z"] = torch.empty(T, h, dtype=torch.bfloat16, device=dev)
        buf["grads"] = {"dX": torch.empty(T, h, dtype=torch.bfloat16, device=dev),
                        **{"d" + k: torch.empty_like(v) for k, v in p.items()}}
    if w.kind == "attn":
        hN = w.H // N
        buf["QKV"] = torch.empty(N, T, tp.QKV_PLANES * hN * w.d, dtype=torch.bfloat16, device=dev)
        buf["O"] = torch.empty(N, T, hN * w.d, dtype=torch.bfloat16, device=dev)
        buf["LSE"] = torch.empty(w.B, w.H, w.S, dtype=torch.float32, device=dev)
        buf["H"] = torch.empty(T, h, dtype=torch.bfloat16, device=dev)
        buf["aws"] = block.workspace(tp.tp_attn_workspace_bytes(dt, w.B, w.S, h, w.H, w.d, N), dev)
    if w.kind == "layer":
        p = {k: d[k] for k in ("Wqkv", "Wo", "W1s", "W2s")}
        buf["save"] = block.workspace(tp.tp_attn_mlp_save_bytes(dt, w.B, w.S, h, w.H, w.d, f, N), dev)
        buf["lws"] = block.workspace(tp.tp_attn_mlp_workspace_bytes(dt, w.B, w.S, h, w.H, w.d, f, N), dev)
        buf["Z"] = torch.empty(T, h, dtype=torch.bfloat16, device=dev)
        buf["grads"] = {"dX": torch.empty(T, h, dtype=torch.bfloat16, device=dev),
                        **{"d" + k: torch.empty_like(v) for k, v in p.items()}}

    def step(X, dZ):
        if w.kind == "mlp":
            tp.tp_mlp_fwd(dt, T, h, f, N, X, d["W1s"], d["W2s"], buf["Y"], buf["A"], buf["Z"], buf["mws"], stream)
            if w.backward:
                tp.tp_mlp_bwd(dt, T, h, f, N, X, d["W1s"], d["W2s"], buf["Y"], buf["A"], dZ, buf["dX"], buf["dW1s"],
                              buf["dW2s"], buf["mws"], stream)
            return buf["Z"], buf["dX"] if w.backward else None
        if w.kind == "gmlp":
            tp.tp_gmlp_fwd(dt, T, h, f, N, X, d["Wgus"], d["Wds"], buf["GU"], buf["A"], buf["Z"], buf["gws"], stream)
            if w.backward:
                tp.tp_gmlp_bwd(dt, T, h, f, N, X, d["Wgus"], d["Wds"], buf["GU"], buf["A"], dZ, buf["dX"],
                               buf["dWgus"], buf["dWds"], buf["gws"], stream)
            return buf["Z"], buf["dX"] if w.backward else None
        if w.kind == "gqa":
            tp.tp_gqa_fwd(dt, w.B, w.S, h, w.H, w.Hkv, w.d, N, w.causal, X, d["Wqkv"], d["Wo"], buf["QKV"], buf["O"],
                          buf["LSE"], buf["Z"], buf["qws"], stream)
            if w.backward:
                tp.tp_gqa_bwd(dt, w.B, w.S, h, w.H, w.Hkv, w.d, N, w.causal, X, d["Wqkv"], d["Wo"], buf["QKV"],
                              buf["O"], buf["LSE"], dZ, buf["dX"], buf["dWqkv"], buf["dWo"], buf["qws"], stream)
            return buf["Z"], buf["dX"] if w.backward else None
        if w.kind in ("lnlayer", "splayer"):
            gr = buf["grads"]
            fwd, bwd = (tp.tp_sp_layer_fwd, tp.tp_sp_layer_bwd) if w.kind == "splayer" else (tp.tp_layer_fwd,
                                                                                            tp.tp_layer_bwd)
            fwd(dt, w.B, w.S, h, w.H, w.d, f, N, True, 1e-5, X, p["ln1_g"], p["ln1_b"], p["Wqkv"], p["Wo"],
                p["ln2_g"], p["ln2_b"], p["W1s"], p["W2s"], buf["save"], buf["Z"], stream)
            bwd(dt, w.B, w.S, h, w.H, w.d, f, N, True, X, p["ln1_g"], p["Wqkv"], p["Wo"], p["ln2_g"], p["W1s"],
                p["W2s"], buf["save"], dZ, gr["dX"], gr["dln1_g"], gr["dln1_b"], gr["dWqkv"], gr["dWo"], gr["dln2_g"],
                gr["dln2_b"], gr["dW1s"], gr["dW2s"], buf["lws"], stream)
            return buf["Z"], gr["dX"]
        if w.kind == "attn":
            tp.tp_attn_fwd(dt, w.B, w.S, h, w.H, w.d, N, w.causal, X, d["Wqkv"], d["Wo"], buf["QKV"], buf["O"],
                           buf["LSE"], buf["H"], buf["aws"], stream)
            return buf["H"], None
        gr = buf["grads"]
        tp.tp_attn_mlp_fwd(dt, w.B, w.S, h, w.H, w.d, f, N, True, X, p["Wqkv"], p["Wo"], p["W1s"], p["W2s"],
                           buf["save"], buf["Z"], stream)
        tp.tp_attn_mlp_bwd(dt, w.B, w.S, h, w.H, w.d, f, N, True, X, p["Wqkv"], p["Wo"], p["W1s"], p["W2s"],
                           buf["save"], dZ, gr["dX"], gr["dWqkv"], gr["dWo"], gr["dW1s"], gr["dW2s"], buf["lws"],
                           stream)
        return buf["Z"], gr["dX"]

    # L2: flush between steps unless one step's working set is far above L2
    work_bytes = sum(t.numel() * t.element_size() for t in list(d.values()) + list(buf.values())
                     if isinstance(t, torch.Tensor))
    want_flush = {"auto": work_bytes < 4 * (129 << 20), "flush": True, "none": False}[args.l2]
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev) if want_flush else None

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step(d["X"], d.get("dZ"))
    torch.cuda.synchronize(dev)
    if tp.tp_sync_status(stream) != 0:
        raise RuntimeError("device error during warm-up")

    gpu_id = None
    try:
        gpu_id = str(torch.cuda.get_device_properties(dev).uuid)
        gpu_id = gpu_id if gpu_id.startswith("GPU-") else "GPU-" + gpu_id
    except Exception:
        gpu_id = None

    def timed_region(kernel_events: bool):
        # kernel_events: an event pair around every library kernel (tp_timing_*), for
        # the per-kernel durations.  Events between the kernels of a step serialise
        # them (no launch overlap), so the step time is taken in a pass without them.
        tp.tp_timing_enable(kernel_events)
        barrier()
        torch.cuda.synchronize(dev)
        with ClockSampler(gpu_id) as cs:
            if flush is None:
                evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
                evs[0].record(stream)
                for i in range(args.steps):
                    step(d["X"], d.get("dZ"))
                    evs[i + 1].record(stream)
                torch.cuda.synchronize(dev)
                ms = evs[0].elapsed_time(evs[-1])
                per = [evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps)]
            else:
                # L2 flushed before every step, outside the step's own events
                evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(args.steps)]
                for a, b in evs:
                    flush.zero_()
                    a.record(stream)
                    step(d["X"], d.get("dZ"))
                    b.record(stream)
                torch.cuda.synchronize(dev)
                per = [a.elapsed_time(b) for a, b in evs]
                ms = sum(per)
        barrier()
        rep = tp.timing_report()
        tp.tp_timing_enable(False)
        return ms, statistics.median(per), rep, cs.summary()

    ms, ms_median, rep_value, clocks = timed_region(False)
    if clocks_rejected(clocks):
        ms, ms_median, rep_value, clocks = timed_region(False)  # re-measured once
    # the same K steps again with per-kernel events: the roofline's launch durations
    ms_ev, _, rep, clocks_ev = timed_region(True)
    if tp.tp_sync_status(stream) != 0:
        raise RuntimeError("device error during the timed region")
    ms = max_over_ranks(ms, world, dev)
    flops = step_flops(w)
    value = whole_job_tflops(flops, args.steps, ms, world)

    # the dominant kernel: largest share of event-measured time in the timed region
    pk = peaks()
    kfl = kernel_flops(w)
    gemm_kinds = {k: v for k, v in rep.items() if k in kfl}
    dom = max(gemm_kinds, key=lambda k: gemm_kinds[k][1]) if gemm_kinds else None
    roof = None
    if dom:
        n, tot = rep[dom]
        avg_ms = tot / n
        achieved = kfl[dom] / (avg_ms / 1e3) / 1e12
        tr = NCU_TRAFFIC.get(dom)
        traffic = tr["bytes"] if tr and tr.get("sha") == source_sha(dom) and tr.get("workload") == w.name else None
        # a timed region of under a second is a burst: the clocks have not settled at
        # the power cap, so the burst GEMM peak is the denominator; a longer region is
        # compared with the sustained one
        sustained = ms >= SUSTAINED_REGION_MS
        peak = pk["bf16_tflops_sustained"] if sustained else pk["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic, "kernel": dom,
                "avg_launch_ms": avg_ms, "flops_per_launch": kfl[dom],
                "peak_source": (f"{'bf16_tflops_sustained' if sustained else 'bf16_tflops'} ({pk['source']}): "
                                f"timed region {ms:.0f} ms, {'at least' if sustained else 'under'} "
                                f"{SUSTAINED_REGION_MS:.0f} ms"),
                "events_pass": {"ms": ms_ev, "sm_mhz": clocks_ev.get("sm_mhz"), "reasons": clocks_ev.get("reasons"),
                                "what": "avg_launch_ms comes from a second pass of the same steps with a CUDA "
                                        "event pair around every library kernel on its launch stream; the value "
                                        "pass runs without them, since events between kernels serialise them"}}
    launches = sum(v[0] for v in rep_value.values())

    # end to end: host buffers, copies inside the timed region.  Two sets of device
    # inputs and outputs: step i+1's inputs are copied in on one stream and step i-1's
    # outputs copied out on another while step i computes, as a user of the C-ABI
    # overlaps them; every step still moves its inputs in and its outputs out.
    e2e = None
    if w.kind in ("mlp", "gmlp", "layer", "lnlayer", "splayer", "attn", "gqa"):
        hX = inp["X"].pin_memory()
        hdZ = inp["dZ"].pin_memory() if "dZ" in inp and w.backward else None
        zkey = "H" if w.kind == "attn" else "Z"

        def dx_get():
            if w.kind in ("lnlayer", "splayer", "layer"):
                return buf["grads"]["dX"]
            return buf.get("dX")

        def dx_set(t):
            if w.kind in ("lnlayer", "splayer", "layer"):
                buf["grads"]["dX"] = t
            else:
                buf["dX"] = t

        z0, dx0 = buf[zkey], (dx_get() if w.backward else None)
        x_in = [torch.empty_like(d["X"]) for _ in range(2)]
        dz_in = [torch.empty_like(d["dZ"]) for _ in range(2)] if hdZ is not None else None
        z_out = [z0, torch.empty_like(z0)]
        dx_out = [dx0, torch.empty_like(dx0)] if dx0 is not None else None
        out_z = torch.empty(z0.shape, dtype=z0.dtype).pin_memory()
        out_dx = torch.empty(dx0.shape, dtype=dx0.dtype).pin_memory() if dx0 is not None else None
        h2d = hX.numel() * hX.element_size() + (hdZ.numel() * hdZ.element_size() if hdZ is not None else 0)
        d2h = out_z.numel() * out_z.element_size() + (out_dx.numel() * out_dx.element_size() if out_dx is not None else 0)
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def e2e_run(nsteps, start_ev):
            ev_in, ev_comp, ev_out = [None] * nsteps, [None] * nsteps, [None] * nsteps

            def copy_in(i):
                with torch.cuda.stream(s_in):
                    s_in.wait_event(start_ev if i < 2 else ev_comp[i - 2])  # step i-2 has read the buffers
                    x_in[i % 2].copy_(hX, non_blocking=True)
                    if dz_in is not None:
                        dz_in[i % 2].copy_(hdZ, non_blocking=True)
                    ev_in[i] = torch.cuda.Event()
                    ev_in[i].record(s_in)

            copy_in(0)
            for i in range(nsteps):
                if i + 1 < nsteps:
                    copy_in(i + 1)
                stream.wait_event(ev_in[i])
                if i >= 2:
                    stream.wait_event(ev_out[i - 2])  # step i-2's outputs have been copied out
                buf[zkey] = z_out[i % 2]
                if dx_out is not None:
                    dx_set(dx_out[i % 2])
                step(x_in[i % 2], dz_in[i % 2] if dz_in is not None else None)
                ev_comp[i] = torch.cuda.Event()
                ev_comp[i].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_comp[i])
                    out_z.copy_(z_out[i % 2], non_blocking=True)
                    if out_dx is not None:
                        out_dx.copy_(dx_out[i % 2], non_blocking=True)
                    ev_out[i] = torch.cuda.Event()
                    ev_out[i].record(s_out)
            stream.wait_event(ev_out[-1])

        w0 = torch.cuda.Event()
        w0.record(stream)
        e2e_run(max(1, args.warmup // 2), w0)
        torch.cuda.synchronize(dev)
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with ClockSampler(gpu_id) as cs_e2e:
            e0.record(stream)
            e2e_run(args.steps, e0)
            e1.record(stream)
            torch.cuda.synchronize(dev)
        barrier()
        buf[zkey] = z0
        if dx0 is not None:
            dx_set(dx0)
        ems = max_over_ranks(e0.elapsed_time(e1), world, dev)
        e2e = {"value": whole_job_tflops(flops, args.steps, ems, world), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ems / args.steps,
               "clocks": cs_e2e.summary(),
               "path": "pinned host -> device copies of each step's inputs on a copy stream, tp_* C-ABI calls on "
                       "the compute stream, device -> pinned host copies of each step's outputs on a second copy "
                       "stream; inputs and outputs double-buffered on the device so that the copies of the "
                       "neighbouring steps overlap the compute.  The copies are the activations (X and dZ in; "
                       "Z and dX out); the weights and their gradients stay resident on the device as model "
                       "state and are not copied"}

    lib = None
    if world == 1 and not args.no_library_baseline:
        Xt = inp_tok["X"].to(dev) if w.kind == "splayer" else d["X"]
        dZt = (inp_tok["dZ"].to(dev) if w.kind == "splayer" else d.get("dZ")) if w.backward else None
        lib = library_baseline(w, d, Xt, dZt, args.steps, args.warmup, dev, gpu_id)
        torch.cuda.synchronize(dev)

    # peaks: measured copies, NVIDIA's nominal dense figure, and the clock the run saw
    nominal = NOMINAL_DENSE_BF16_TFLOPS
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    clock_peak = None
    if clocks and clocks.get("sm_mhz"):
        # one M=128, N=256, K=16 bf16 tcgen05 MMA per 128 SM cycles = 8192 flop per clock per SM;
        # at 152 SMs and ~1.81 GHz this is the nominal 2.25 PFLOP/s
        tf = sms * 8192 * clocks["sm_mhz"] * 1e6 / 1e12
        clock_peak = {"tflops": tf, "frac": value / world / tf, "sm_count": sms, "flop_per_clk_per_sm": 8192,
                      "sm_mhz": clocks["sm_mhz"]}

    cpu = None
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        import torch as _t  # noqa: F401
        cpu = cpu_baseline(w, {k: v.to(torch.float64).numpy() for k, v in inp_tok.items()}, args.cpu_seconds)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded normals; weights random-init)",
                "config": {"workload": w.name, "description": describe(w), "parallelism": "tp" + str(N) +
                           " logical shards on one GPU" + (f", {world} independent replicas" if world > 1 else ""),
                           "flops_per_step": flops,
                           "launch_overlap": bool(args.launch_overlap),
                           "l2": ("flushed before each step (256 MiB write, outside the step's CUDA events)"
                                  if flush is not None else
                                  (f"inputs larger than L2 (step working set {work_bytes / 2**30:.2f} GiB); no flush"
                                   if work_bytes > (129 << 20) else
                                   f"not flushed (--l2 none; the step working set, {work_bytes / 2**30:.2f} GiB, "
                                   f"fits in L2)"))},
                "pct_of_peak": {"of_measured_burst": value / world / pk["bf16_tflops"],
                                "of_measured_sustained": value / world / pk["bf16_tflops_sustained"],
                                "peaks": pk["source"], "of_nominal_dense": value / world / nominal,
                                "nominal_dense_tflops": nominal, "nominal_source": NOMINAL_SOURCE,
                                "clock_based": clock_peak},
                "ms_per_step_median": ms_median,
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
                "library_baseline": lib,
                "kernels": {k: {"launches": v[0], "ms_total": v[1]} for k, v in rep.items()},
                "clocks": clocks}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="tpblock", choices=["tpblock", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-library-baseline", action="store_true",
                    help="skip timing the torch library composition of the step")
    ap.add_argument("--l2", default="auto", choices=["auto", "flush", "none"],
                    help="L2 between timed steps: auto flushes when a step's working set is under 4x L2")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--gemm-tiling", type=int, default=0, choices=[0, 1, 2],
                    help="0 automatic, 1 one CTA per 128x256 tile, 2 CTA pairs per 256x256 tile")
    ap.add_argument("--launch-overlap", type=int, default=1, choices=[0, 1],
                    help="1: each kernel's prologue overlaps the previous kernel's tail (programmatic "
                         "dependent launch); 0: ordinary stream order")
    ap.add_argument("--override", action="append", default=[],
                    help="KEY=VALUE shape override of the workload (a smaller case for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    from tensor_transformer_block_gb300.inputs import WORKLOADS
    if args.workload not in WORKLOADS:
        raise SystemExit(f"unknown workload {args.workload}; choose from {sorted(WORKLOADS)}")
    w = WORKLOADS[args.workload]
    if args.override:
        import dataclasses
        kv = {}
        for item in args.override:
            k, v = item.split("=", 1)
            kv[k] = type(getattr(w, k))(v)
        if "B" in kv or "S" in kv:
            kv.setdefault("T", kv.get("B", w.B) * kv.get("S", w.S))
        w = dataclasses.replace(w, name=w.name + "+" + ",".join(args.override), **kv)
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_gpu(args, w)


if __name__ == "__main__":
    main()
