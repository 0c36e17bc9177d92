"""tp_mlp_fwd_noalloc: the MLP forward for callers that cannot allocate device
memory (a plug-in whose host framework owns all allocations, a runtime that
forbids cudaMalloc once it is serving).  Its activation scratch is a fixed array
inside the library.  The test calls it through the C-ABI twice in a row, on
different inputs.  Each result must equal tp_mlp_fwd's bit for bit when that
call is given the activation-sized scratch alone (the same kernels run on the same
operands; only the scratch address differs) and pass
the parity criteria the other tests use, and the second call must leave the
device's free memory unchanged (an allocation inside the call, even one that
bypasses torch's allocator, would show there).  The file sorts last so that a
run stopping at the first failure has already run every other test."""
import pytest
import torch

import tensor_transformer_block_gb300 as tp
from parity import assert_bf16_parity, assert_f32_parity
from tensor_transformer_block_gb300 import block, inputs

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_matches_workspace_path_twice(dtype):
    lib = tp.load_library()
    code = tp.TP_BF16 if dtype == "bf16" else tp.TP_F32
    check = assert_bf16_parity if dtype == "bf16" else assert_f32_parity
    for i, (T, h, f, N, seed) in enumerate(((2048, 1024, 4096, 4, 0), (333, 200, 264, 3, 7))):
        inp = inputs.mlp_inputs(T, h, f, N, dtype=dtype, seed=seed, backward=False)
        d = {k: v.cuda() for k, v in inp.items()}
        # the workspace path with exactly the activation-sized scratch: the same
        # kernels as the fixed-array path (a larger workspace may split small GEMMs)
        ws = block.workspace((T * f * (2 if dtype == "bf16" else 4) + 255) // 256 * 256, d["X"].device)
        z_ref = block.mlp_forward(d["X"], d["W1s"], d["W2s"], save=False, ws=ws)["Z"]
        z = torch.full_like(z_ref, float("nan"))
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        st = lib.tp_mlp_fwd_noalloc(code, T, h, f, N, d["X"].data_ptr(), d["W1s"].data_ptr(),
                                    d["W2s"].data_ptr(), z.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert st == 0, tp.tp_status_string(st)
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        assert tp.tp_sync_status() == 0
        if i > 0:  # the first call may load kernels; the second must not change free memory
            assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
        assert torch.equal(z, z_ref), f"noalloc Z differs from tp_mlp_fwd's ({T}, {h}, {f}, {N})"
        check(_np(z), _np(z_ref), f"noalloc Z ({T}, {h}, {f}, {N})")


def test_noalloc_rejects_oversize():
    lib = tp.load_library()
    # T * f * 2 bytes = 64 MiB > the 32 MiB array
    st = lib.tp_mlp_fwd_noalloc(tp.TP_BF16, 8192, 1024, 4096, 4, 16, 16, 16, 16, None)
    assert st == 4  # TP_ERR_WORKSPACE
