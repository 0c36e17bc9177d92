"""Host-side checks that need no GPU: the library loads, exports every function
the header declares, and its argument validation rejects bad calls before any
CUDA call is made."""
import ctypes
import json
import os
import subprocess

import pytest

import tensor_transformer_block_gb300 as tp
from tensor_transformer_block_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLD = json.load(open(os.path.join(ROOT, "tests", "golden", "split_shapes.json")))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return tp.load_library()


def test_exports_every_header_function(lib):
    names = tp.header_functions()
    assert len(names) >= 11
    out = subprocess.run(["nm", "-D", "--defined-only", tp.LIB_PATH], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n)
    # nothing else of the library's internals is exported
    assert all(e.startswith("tp_") for e in exported)


def test_status_strings(lib):
    for s in range(10):
        assert tp.tp_status_string(s) != "unknown status"
    assert tp.tp_status_string(99) == "unknown status"
    assert tp.tp_version() > 0


def test_workspace_queries(lib):
    assert tp.tp_mlp_workspace_bytes(tp.TP_BF16, 64, 256, 1000, 3) == 0   # 3 does not divide 1000
    assert tp.tp_mlp_workspace_bytes(tp.TP_BF16, 64, 256, 1024, 2) == 64 * 1024 * 2
    assert tp.tp_mlp_workspace_bytes(tp.TP_F32, 64, 256, 1024, 2) == 64 * 1024 * 4
    assert tp.tp_mlp_workspace_bytes(tp.TP_BF16, 64, 256, 1024, 128) > 0   # f/N = 8: one 16-byte row
    assert tp.tp_mlp_workspace_bytes(tp.TP_BF16, 64, 256, 1024, 256) == 0  # f/N = 4: rows under 16 bytes
    assert tp.tp_attn_workspace_bytes(tp.TP_BF16, 2, 2048, 4096, 32, 128, 8) > 0
    assert tp.tp_attn_workspace_bytes(tp.TP_BF16, 2, 2048, 4096, 32, 128, 5) == 0
    assert tp.tp_attn_workspace_bytes(tp.TP_F32, 2, 2048, 4096, 32, 128, 8) == 0


def _mlp_fwd(lib, dtype=1, T=64, h=256, f=1024, N=2, X=16, W1=16, W2=16, Z=16, ws=None, wsb=0):
    return lib.tp_mlp_fwd(dtype, T, h, f, N, X, W1, W2, None, None, Z, ws, wsb, None)


def test_mlp_validation_before_cuda(lib):
    assert _mlp_fwd(lib, N=3, f=1000) == 2              # N does not divide f
    assert _mlp_fwd(lib, T=0) == 2
    assert _mlp_fwd(lib, h=250) == 2                    # row not a multiple of 8 (bf16)
    assert _mlp_fwd(lib, dtype=7) == 3
    assert _mlp_fwd(lib, X=None) == 1
    assert _mlp_fwd(lib, X=8) == 7                      # misaligned pointer
    assert _mlp_fwd(lib, ws=None) == 4                  # A_save NULL needs a workspace
    assert _mlp_fwd(lib, ws=256, wsb=16) == 4           # workspace too small
    assert _mlp_fwd(lib, ws=272, wsb=1 << 30) == 7      # workspace not 256-aligned
    bwd = lib.tp_mlp_bwd(0, 64, 256, 1024, 2, 16, 16, 16, 16, 16, 16, 16, 16, 16, 256, 1 << 30, None)
    assert bwd == 3                                     # fp32 backward is not provided


def test_gmlp_validation_before_cuda(lib):
    g = lambda **k: lib.tp_gmlp_fwd(k.get("dt", 1), k.get("T", 64), k.get("h", 256), k.get("f", 1024),
                                    k.get("N", 2), k.get("X", 16), 16, 16, None, None, 16, k.get("ws", None),
                                    k.get("wsb", 0), None)
    assert g(N=3, f=1000) == 2                          # N does not divide f
    assert g(dt=0) == 3                                 # bf16 only
    assert g(h=250) == 2
    assert g(X=None) == 1
    assert g(X=8) == 7
    assert g() == 4                                     # A_save NULL needs a workspace
    assert tp.tp_gmlp_workspace_bytes(tp.TP_BF16, 64, 256, 1024, 2) == 2 * 64 * 1024 * 2
    assert tp.tp_gmlp_workspace_bytes(tp.TP_F32, 64, 256, 1024, 2) == 0
    bwd = lib.tp_gmlp_bwd(1, 64, 256, 1024, 2, 16, 16, 16, None, 16, 16, 16, 16, 16, 256, 1 << 30, None)
    assert bwd == 1                                     # GU_save is required


def test_gqa_validation_before_cuda(lib):
    f = lambda **k: lib.tp_gqa_fwd(1, 2, 128, 512, k.get("H", 8), k.get("Hkv", 2), 64, k.get("N", 2), 1, 16, 16, 16,
                                   None, None, None, 16, None, 0, None)
    assert f(Hkv=3) == 2                                # Hkv does not divide H
    assert f(Hkv=2, N=4) == 2                           # N does not divide Hkv
    assert f() == 4                                     # valid: wants a workspace for the unsaved tensors
    assert tp.tp_gqa_workspace_bytes(tp.TP_BF16, 2, 128, 512, 8, 8, 64, 2) == \
        tp.tp_attn_workspace_bytes(tp.TP_BF16, 2, 128, 512, 8, 64, 2)
    assert tp.tp_gqa_workspace_bytes(tp.TP_BF16, 2, 128, 512, 8, 2, 64, 2) < \
        tp.tp_attn_workspace_bytes(tp.TP_BF16, 2, 128, 512, 8, 64, 2)


def test_sp_layer_validation_before_cuda(lib):
    f = lambda S, N: lib.tp_sp_layer_fwd(1, 2, S, 512, 4, 128, 1024, N, 1, 1e-5, *([16] * 9), 256, 0, 16, None)
    assert f(384, 2) == 2                               # S/N = 192: not a multiple of 128
    assert f(256, 3) == 2                               # N does not divide S
    assert f(256, 2) == 4                               # valid shape: the empty save buffer is reported


def test_attention_validation_before_cuda(lib):
    f = lambda **k: lib.tp_attn_fwd(k.get("dt", 1), k.get("B", 2), k.get("S", 128), k.get("h", 512),
                                    k.get("H", 8), k.get("d", 64), k.get("N", 2), 1, k.get("X", 16), 16, 16,
                                    None, None, None, 16, k.get("ws", None), k.get("wsb", 0), None)
    assert f(N=3) == 2
    assert f(d=96) == 2
    assert f(dt=0) == 3
    assert f(X=None) == 1
    assert f(X=24) == 7
    assert f() == 4


@pytest.mark.parametrize("case", [c for c in GOLD["cases"] if c["kind"] == "heads"], ids=lambda c: c["id"])
def test_golden_head_split_rule(lib, case):
    """The pages' head-split facts at the boundary: 32 heads on 4 shards is valid
    (8 per shard), on 5 shards it is rejected."""
    ws = tp.tp_attn_workspace_bytes(tp.TP_BF16, 1, 128, 4096, case["H"], 128, case["N"])
    assert (ws > 0) == case["valid"]
    if not case["valid"]:
        st = lib.tp_attn_fwd(1, 1, 128, 4096, case["H"], 128, case["N"], 1, 16, 16, 16, None, None, None, 16,
                             None, 0, None)
        assert st == 2


def test_gemm_tiling_modes(lib):
    """Tilings 0-2 are accepted; any other value is rejected and leaves the setting."""
    for m in (1, 2, 0):
        assert lib.tp_set_gemm_tiling(m) == 0
    for m in (3, -1, 4):
        assert lib.tp_set_gemm_tiling(m) == 2


def test_launch_overlap_setting(lib):
    """Overlap 0 and 1 are accepted; any other value is rejected."""
    for v in (0, 1):
        assert lib.tp_set_launch_overlap(v) == 0
    for v in (2, -1):
        assert lib.tp_set_launch_overlap(v) == 2
