"""Every C-ABI call of libtpblock opens an NVTX range named after the call in the
"libtpblock" domain.  The test loads a recording NVTX tool (tests/nvtx_record.c,
compiled here with the system C compiler) through NVTX_INJECTION64_PATH in a fresh
process, makes calls that fail argument validation (so no GPU is needed: the
range is opened before validation and closed on return) and reads the record."""
import os
import shutil
import subprocess
import sys

import pytest

from tensor_transformer_block_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path.insert(0, sys.argv[1])
import tensor_transformer_block_gb300 as tp
lib = tp.load_library()
assert lib.tp_mlp_fwd(1, 64, 256, 1000, 3, 16, 16, 16, None, None, 16, None, 0, None) == 2
assert lib.tp_attn_fwd(1, 1, 128, 4096, 32, 128, 5, 1, 16, 16, 16, None, None, None, 16, None, 0, None) == 2
assert lib.tp_layernorm_fwd(0, 4, 8, 1e-5, 16, 16, 16, 16, 16, 16, None) == 3
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_every_call_opens_a_named_range(tmp_path):
    build.build()
    so = str(tmp_path / "nvtx_record.so")
    subprocess.run(["gcc", "-shared", "-fPIC", "-O1", "-I", "/usr/local/cuda/include", "-o", so,
                    os.path.join(ROOT, "tests", "nvtx_record.c")], check=True)
    rec = tmp_path / "record.txt"
    env = dict(os.environ, NVTX_INJECTION64_PATH=so, TP_NVTX_RECORD=str(rec))
    subprocess.run([sys.executable, "-c", CHILD, ROOT], check=True, env=env, timeout=300)
    lines = rec.read_text().splitlines()
    assert lines.count("domain libtpblock") == 1
    pushes = [ln[5:] for ln in lines if ln.startswith("push ")]
    # tp_attn_fwd is the grouped-query call with Hkv = H: its range holds that call's
    assert pushes == ["tp_mlp_fwd", "tp_attn_fwd", "tp_gqa_fwd", "tp_layernorm_fwd"]
    assert lines.count("pop") == len(pushes)
