"""The debug-bounds build (libssm_debug.so, SSM_DEBUG_BOUNDS=1): its kernels check the
indices of their global writes and TMA coordinates in-kernel and record SSM_ERR_BOUNDS
in the status word instead of faulting.  On correct shapes no check may fire and the
results must still match the oracle."""
import ctypes
import json
import os
import subprocess
import sys

import pytest

from selective_state_space_132_b300 import binding as bd
from selective_state_space_132_b300.build import LIB_DEBUG, build

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def debug_lib():
    build(debug_bounds=True)
    return LIB_DEBUG


def test_debug_library_exports_the_abi(debug_lib):
    lib = ctypes.CDLL(debug_lib)
    for name in bd.EXPORTED:
        assert hasattr(lib, name), name
    lib.ssm_status_string.restype = ctypes.c_char_p
    assert b"index check" in lib.ssm_status_string(7)


@pytest.mark.gpu
def test_no_index_check_fires_on_valid_calls(debug_lib):
    env = dict(os.environ, SSM_LIBRARY=debug_lib)
    r = subprocess.run([sys.executable, os.path.join(HERE, "_debug_bounds_run.py")],
                       capture_output=True, text=True, env=env, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    rows = [json.loads(ln) for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(rows) == 14, r.stdout
    for row in rows:
        assert row["status"] == 0, row
        # (the parity suites hold the exact bounds; this only catches a skipped access)
        assert row["rel_l2"] < 5e-3, row
