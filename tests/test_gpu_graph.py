"""The compute calls enqueue kernels only (no synchronisation, allocation or host
round trip on the stream), so a step can be captured into a CUDA graph and
replayed: every output of a replay is bit-identical to the same calls run eagerly,
and a replay after the input buffers are refilled computes on the new inputs."""
import pytest
import torch

import tensor_transformer_block_gb300 as tp
from tensor_transformer_block_gb300 import block, inputs

pytestmark = pytest.mark.gpu


def _graph_matches_eager(step, refill):
    """step(): runs the calls on the current stream into preallocated outputs and
    returns them; refill(): writes new values into the input buffers."""
    eager = {k: v.clone() for k, v in step().items()}
    torch.cuda.synchronize()
    assert tp.tp_sync_status() == 0
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = step()
    g.replay()
    torch.cuda.synchronize()
    assert tp.tp_sync_status() == 0
    for k in eager:
        assert torch.equal(outs[k], eager[k]), k
    # new inputs: the replay must read the buffers, not values captured with the graph
    refill()
    eager2 = {k: v.clone() for k, v in step().items()}
    torch.cuda.synchronize()
    for k in eager2:
        outs[k].zero_()
    g.replay()
    torch.cuda.synchronize()
    assert tp.tp_sync_status() == 0
    for k in eager2:
        assert torch.equal(outs[k], eager2[k]), k
        assert not torch.equal(eager2[k], eager[k]), f"{k} did not change with the inputs"


def test_mlp_step_graph():
    T, h, f, N = 2048, 1024, 4096, 4  # split-K row-parallel GEMMs and their reduction
    d = {k: v.cuda() for k, v in inputs.mlp_inputs(T, h, f, N, seed=31).items()}
    dev = d["X"].device
    ws = block.workspace(tp.tp_mlp_workspace_bytes(tp.TP_BF16, T, h, f, N), dev)
    o = {"Z": torch.empty(T, h, dtype=torch.bfloat16, device=dev),
         "Y": torch.empty(N, T, f // N, dtype=torch.bfloat16, device=dev),
         "A": torch.empty(N, T, f // N, dtype=torch.bfloat16, device=dev),
         "dX": torch.empty(T, h, dtype=torch.bfloat16, device=dev),
         "dW1s": torch.empty_like(d["W1s"]), "dW2s": torch.empty_like(d["W2s"])}

    def step():
        tp.tp_mlp_fwd(tp.TP_BF16, T, h, f, N, d["X"], d["W1s"], d["W2s"], o["Y"], o["A"], o["Z"], ws)
        tp.tp_mlp_bwd(tp.TP_BF16, T, h, f, N, d["X"], d["W1s"], d["W2s"], o["Y"], o["A"], d["dZ"], o["dX"],
                      o["dW1s"], o["dW2s"], ws)
        return o

    def refill():
        d["X"].copy_(inputs.mlp_inputs(T, h, f, N, seed=32)["X"])

    _graph_matches_eager(step, refill)


def test_prenorm_layer_step_graph():
    B, S, h, H, dd, f, N = 1, 512, 512, 4, 128, 2048, 2
    p = {k: v.cuda() for k, v in inputs.prenorm_inputs(B, S, h, H, dd, f, N, seed=33).items()}
    dev = p["X"].device
    save = block.workspace(tp.tp_layer_save_bytes(tp.TP_BF16, B, S, h, H, dd, f, N), dev)
    lws = block.workspace(tp.tp_layer_workspace_bytes(tp.TP_BF16, B, S, h, H, dd, f, N), dev)
    Z = torch.empty_like(p["X"])
    grads = {"dX": torch.empty_like(p["X"]), "dln1_g": torch.empty_like(p["ln1_g"]),
             "dln1_b": torch.empty_like(p["ln1_b"]), "dWqkv": torch.empty_like(p["Wqkv"]),
             "dWo": torch.empty_like(p["Wo"]), "dln2_g": torch.empty_like(p["ln2_g"]),
             "dln2_b": torch.empty_like(p["ln2_b"]), "dW1s": torch.empty_like(p["W1s"]),
             "dW2s": torch.empty_like(p["W2s"])}

    def step():
        fw = block.prenorm_layer_forward(p["X"], p, B, S, save=save)
        Z.copy_(fw["Z"])
        block.prenorm_layer_backward(p["X"], p, save, p["dZ"], B, S, ws=lws, out=grads)
        return {"Z": Z, **grads}

    def refill():
        p["dZ"].copy_(inputs.prenorm_inputs(B, S, h, H, dd, f, N, seed=34)["dZ"])
        p["X"].copy_(inputs.prenorm_inputs(B, S, h, H, dd, f, N, seed=35)["X"])

    _graph_matches_eager(step, refill)
