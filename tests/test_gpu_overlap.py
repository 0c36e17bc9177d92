"""Programmatic dependent launch changes when each kernel starts (its prologue
overlapping the previous kernel's tail), not what any kernel computes: every
output of each call is bit-identical with the overlap on and off."""
import pytest
import torch

import tensor_transformer_block_gb300 as tp
from tensor_transformer_block_gb300 import block, inputs

pytestmark = pytest.mark.gpu


def _same_both_ways(run):
    outs = {}
    try:
        for on in (False, True):
            tp.tp_set_launch_overlap(on)
            outs[on] = {k: v.clone() for k, v in run().items() if isinstance(v, torch.Tensor)}
            torch.cuda.synchronize()
            assert tp.tp_sync_status() == 0
    finally:
        tp.tp_set_launch_overlap(True)
    assert outs[True].keys() == outs[False].keys()
    for k in outs[True]:
        assert torch.equal(outs[True][k], outs[False][k]), k


def test_overlap_mlp():
    """The small MLP shape: split-K GEMMs and their fixed-order reduction."""
    d = {k: v.cuda() for k, v in inputs.mlp_inputs(2048, 1024, 4096, 4, seed=11).items()}

    def run():
        fw = block.mlp_forward(d["X"], d["W1s"], d["W2s"])
        bw = block.mlp_backward(d["X"], d["W1s"], d["W2s"], fw["Y"], fw["A"], d["dZ"])
        return {**fw, **bw}

    _same_both_ways(run)


def test_overlap_mlp_f32():
    """The fp32 forward (FFMA GEMMs)."""
    d = {k: v.cuda() for k, v in inputs.mlp_inputs(64, 256, 1024, 2, dtype="f32", seed=11).items()}
    _same_both_ways(lambda: block.mlp_forward(d["X"], d["W1s"], d["W2s"]))


def test_overlap_gated_mlp():
    d = {k: v.cuda() for k, v in inputs.gmlp_inputs(1000, 512, 1536, 4, seed=12).items()}

    def run():
        fw = block.gmlp_forward(d["X"], d["Wgus"], d["Wds"])
        bw = block.gmlp_backward(d["X"], d["Wgus"], d["Wds"], fw["GU"], fw["A"], d["dZ"])
        return {**fw, **bw}

    _same_both_ways(run)


def test_overlap_prenorm_layer():
    """LayerNorm, the bf16 -> fp16 weight copies, attention forward and backward
    (Dsum, dK/dV, dQ) and every GEMM epilogue, back to back in one stream."""
    B, S, h, H, d, f, N = 2, 384, 512, 4, 128, 1024, 2
    p = {k: v.cuda() for k, v in inputs.prenorm_inputs(B, S, h, H, d, f, N, seed=13).items()}

    def run():
        fw = block.prenorm_layer_forward(p["X"], p, B, S)
        bw = block.prenorm_layer_backward(p["X"], p, fw["save"], p["dZ"], B, S)
        return {"Z": fw["Z"], **bw}

    _same_both_ways(run)


def test_overlap_gqa():
    B, S, h, H, Hkv, d, N = 1, 640, 512, 8, 2, 64, 2
    p = {k: v.cuda() for k, v in inputs.gqa_inputs(B, S, h, H, Hkv, d, N, seed=14).items()}

    def run():
        fw = block.gqa_forward(p["X"], p["Wqkv"], p["Wo"], H, Hkv, d, B, S)
        bw = block.gqa_backward(p["X"], p["Wqkv"], p["Wo"], fw["QKV"], fw["O"], fw["LSE"], p["dZ"], H, Hkv, d, B, S)
        return {**fw, **bw}

    _same_both_ways(run)
