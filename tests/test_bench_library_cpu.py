"""bench.py's library baseline composes the same step from torch calls on the
unsharded weights.  On the CPU, in float64 and at tiny sizes, its forward must
give the oracle's Z for every workload kind: this checks that the shard-major
weights are viewed back as the unsharded matrices the pages split."""
import dataclasses
import importlib.util
import pathlib

import numpy as np
import pytest
import torch

from oracle import tp_oracle as O
from tensor_transformer_block_gb300 import inputs

ROOT = pathlib.Path(__file__).resolve().parents[1]
_spec = importlib.util.spec_from_file_location("bench_mod", ROOT / "bench.py")
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)

SMALL = {
    "mlp": dict(T=24, h=32, f=64, N=4),
    "gmlp": dict(T=24, h=32, f=64, N=4),
    "attn": dict(B=2, S=12, T=24, h=32, H=4, d=8, N=2),
    "gqa": dict(B=2, S=12, T=24, h=32, H=8, Hkv=4, d=8, N=2),
    "layer": dict(B=2, S=12, T=24, h=32, H=4, d=8, f=64, N=2),
    "lnlayer": dict(B=2, S=12, T=24, h=32, H=4, d=8, f=64, N=2),
}


def _workload(kind):
    base = next(w for w in inputs.WORKLOADS.values() if w.kind == kind and w.dtype == "bf16")
    return dataclasses.replace(base, dtype="f32", **SMALL[kind])


def _oracle_z(w, a):
    if w.kind == "mlp":
        return O.mlp_forward(a["X"], a["W1s"], a["W2s"])["Z"]
    if w.kind == "gmlp":
        return O.gated_mlp_forward(a["X"], a["Wgus"], a["Wds"])["Z"]
    if w.kind == "attn":
        return O.attention_forward(a["X"], a["Wqkv"], a["Wo"], w.B, w.S, w.causal)["Z"]
    if w.kind == "gqa":
        return O.gqa_attention_forward(a["X"], a["Wqkv"], a["Wo"], w.B, w.S, w.H, w.Hkv, w.causal)["Z"]
    if w.kind == "layer":
        return O.layer_forward(a["X"], a["Wqkv"], a["Wo"], a["W1s"], a["W2s"], w.B, w.S, True)["Z"]
    return O.prenorm_layer_forward(a["X"], a["ln1_g"], a["ln1_b"], a["Wqkv"], a["Wo"], a["ln2_g"], a["ln2_b"],
                                   a["W1s"], a["W2s"], w.B, w.S, True)["Z"]


@pytest.mark.parametrize("kind", sorted(SMALL))
def test_library_composition_matches_oracle(kind):
    w = _workload(kind)
    inp = inputs.workload_inputs(w)
    d = {k: v.to(torch.float64) for k, v in inp.items()}
    fwd, p = bench.library_composition(w, d)
    z = fwd(d["X"], p).numpy()
    ref = _oracle_z(w, {k: v.numpy() for k, v in d.items()})
    np.testing.assert_allclose(z, ref, rtol=1e-9, atol=1e-9 * np.abs(ref).max())
