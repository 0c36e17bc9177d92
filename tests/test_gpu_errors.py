"""Device-side failure detection without a GPU fault: the bounded wait runs out on
a barrier nothing signals, the status surfaces through tp_sync_status, and the
context stays usable afterwards."""
import pytest
import torch

import tensor_transformer_block_gb300 as tp
from tensor_transformer_block_gb300 import block, inputs

pytestmark = pytest.mark.gpu


def test_device_is_sm103():
    assert tp.tp_device_check() == 0


def test_timeout_status_then_normal_call():
    assert tp.tp_sync_status() == 0
    tp.tp_debug_timeout_probe(50_000_000)
    assert tp.tp_sync_status() == 6  # TP_ERR_TIMEOUT
    assert tp.tp_sync_status() == 0  # cleared
    inp = inputs.mlp_inputs(64, 64, 128, 2, backward=False)
    dev = {k: v.cuda() for k, v in inp.items()}
    z = block.mlp_forward(dev["X"], dev["W1s"], dev["W2s"])["Z"]
    torch.cuda.synchronize()
    assert tp.tp_sync_status() == 0
    assert torch.isfinite(z.float()).all()
