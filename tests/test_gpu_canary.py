"""Guard bands around every output, save buffer and workspace of every C-ABI call
(tests/canary_calls.py): with the release library in this process, and with the
bounds-checked debug build (compiled with -DTPBLOCK_DEBUG: device-side index and
TMA-alignment checks that latch TP_ERR_BOUNDS) in a fresh process, where the
error word must also come back clean."""
import os
import subprocess
import sys

import pytest

import tensor_transformer_block_gb300 as tp
from tensor_transformer_block_gb300 import build

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_release_build_guard_bands():
    import canary_calls
    hit = canary_calls.run_calls()
    assert not hit, f"writes past a buffer's end: {hit}"
    assert tp.tp_sync_status() == 0


def test_debug_build_guard_bands_and_error_word():
    lib = build.build(debug=True)
    env = dict(os.environ, TPBLOCK_LIB=lib, PYTHONPATH=os.pathsep.join([os.path.dirname(HERE), HERE]))
    r = subprocess.run([sys.executable, os.path.join(HERE, "canary_calls.py")], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "libtpblock_debug.so" in r.stdout, r.stdout
