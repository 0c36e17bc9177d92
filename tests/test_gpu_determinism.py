"""Run-to-run determinism of every call: each output is bit-identical over repeated
runs, with other launches of different shapes in between to perturb the order in
which CTAs are scheduled.  Every reduction in the library has a fixed order (shard
sums in the accumulator, split-K partials added in split order, dK/dV summed over
a group in one CTA, dQ over key blocks in one CTA, LayerNorm column sums in CTA
order); no result may depend on timing."""
import pytest
import torch

import tensor_transformer_block_gb300 as tp
from tensor_transformer_block_gb300 import block, inputs

pytestmark = pytest.mark.gpu

RUNS = 4


def _perturb():
    # a launch of another shape between the runs (different grids and tilings)
    d = {k: v.cuda() for k, v in inputs.mlp_inputs(333, 200, 264, 3, seed=99).items()}
    block.mlp_forward(d["X"], d["W1s"], d["W2s"])


def _repeat(run):
    first = None
    for i in range(RUNS):
        out = {k: v.clone() for k, v in run().items() if isinstance(v, torch.Tensor)}
        torch.cuda.synchronize()
        assert tp.tp_sync_status() == 0
        if first is None:
            first = out
        else:
            for k in first:
                assert torch.equal(first[k], out[k]), f"{k} differs on run {i}"
        _perturb()


def test_prenorm_layer_deterministic():
    B, S, h, H, d, f, N = 2, 1024, 1024, 8, 128, 4096, 4
    p = {k: v.cuda() for k, v in inputs.prenorm_inputs(B, S, h, H, d, f, N, seed=21).items()}

    def run():
        fw = block.prenorm_layer_forward(p["X"], p, B, S)
        bw = block.prenorm_layer_backward(p["X"], p, fw["save"], p["dZ"], B, S)
        return {"Z": fw["Z"], **bw}

    _repeat(run)


def test_gqa_deterministic():
    B, S, h, H, Hkv, d, N = 2, 1024, 1024, 16, 4, 128, 4
    p = {k: v.cuda() for k, v in inputs.gqa_inputs(B, S, h, H, Hkv, d, N, seed=22).items()}

    def run():
        fw = block.gqa_forward(p["X"], p["Wqkv"], p["Wo"], H, Hkv, d, B, S)
        bw = block.gqa_backward(p["X"], p["Wqkv"], p["Wo"], fw["QKV"], fw["O"], fw["LSE"], p["dZ"], H, Hkv, d, B, S)
        return {**fw, **bw}

    _repeat(run)


def test_attn_mlp_layer_deterministic():
    B, S, h, H, d, f, N = 1, 1024, 1024, 8, 128, 4096, 8
    p = {k: v.cuda() for k, v in inputs.layer_inputs(B, S, h, H, d, f, N, seed=23).items()}

    def run():
        fw = block.attn_mlp_forward(p["X"], p, B, S)
        bw = block.attn_mlp_backward(p["X"], p, fw["save"], p["dZ"], B, S)
        return {"Z": fw["Z"], **bw}

    _repeat(run)


def test_small_mlp_split_k_deterministic():
    """The small MLP shape, whose row-parallel GEMMs run split-K."""
    d = {k: v.cuda() for k, v in inputs.mlp_inputs(2048, 1024, 4096, 4, seed=24).items()}

    def run():
        fw = block.mlp_forward(d["X"], d["W1s"], d["W2s"])
        return {**fw, **block.mlp_backward(d["X"], d["W1s"], d["W2s"], fw["Y"], fw["A"], d["dZ"])}

    _repeat(run)


def test_f32_mlp_deterministic():
    """The fp32 forward, whose K loop is split over a cluster."""
    d = {k: v.cuda() for k, v in inputs.mlp_inputs(64, 256, 1024, 2, dtype="f32", seed=25).items()}
    _repeat(lambda: block.mlp_forward(d["X"], d["W1s"], d["W2s"]))
