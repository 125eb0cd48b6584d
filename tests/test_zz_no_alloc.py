"""ssm_scan_fwd_noalloc: the scan for callers that cannot allocate device memory on
the call path (a plugin inside a runtime that owns all device memory, a latency-
critical loop that cannot take cudaMalloc's implicit synchronisation, a process
held to memory reserved at start-up).  It must give what ssm_scan_fwd gives, using
the library's fixed scratch buffer instead of a caller workspace.

This file is collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test.  Each call below goes through the C ABI.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from selective_state_space_132_b300 import binding as bd
from selective_state_space_132_b300 import workloads as W

from _parity import assert_close, dev, host, io_dtype

pytestmark = pytest.mark.gpu


def _buffers(p):
    io = io_dtype(p.io)
    ins = dict(x=dev(p.x, io), delta=dev(p.delta, io), A=dev(p.A), B=dev(p.B, io),
               C=dev(p.C, io), D=dev(p.D), z=dev(p.z, io), delta_bias=dev(p.bias), h0=dev(p.h0))
    return ins


def _args(ins, y, hf, time_chunk, disc="euler"):
    return bd._scan_args(ins["x"], ins["delta"], ins["A"], ins["B"], ins["C"], ins["D"], ins["z"],
                         ins["delta_bias"], True, ins["h0"], y, hf, time_chunk, disc)


def _run_both(p, time_chunk, disc="euler"):
    lib = bd.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    ins = _buffers(p)
    # the existing entry point, with a workspace
    y_ref = torch.empty_like(ins["x"])
    h_ref = torch.empty((p.batch, p.dim, p.dstate), dtype=torch.float32, device="cuda")
    a = _args(ins, y_ref, h_ref, time_chunk, disc)
    need = ctypes.c_size_t(0)
    assert lib.ssm_scan_workspace_size(ctypes.byref(a), ctypes.byref(need)) == 0
    ws = torch.empty(max(int(need.value), 256), dtype=torch.uint8, device="cuda")
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    assert lib.ssm_scan_fwd(ctypes.byref(a), stream) == 0
    # the no-allocation entry point: workspace fields left empty
    y = torch.full_like(ins["x"], float("nan"))
    hf = torch.full((p.batch, p.dim, p.dstate), float("nan"), dtype=torch.float32,
                    device="cuda")
    b = _args(ins, y, hf, time_chunk, disc)
    assert lib.ssm_scan_fwd_noalloc(ctypes.byref(b), stream) == 0
    torch.cuda.synchronize()
    return host(y), host(hf), host(y_ref), host(h_ref)


@pytest.mark.parametrize("disc", ["euler", "zoh"])
@pytest.mark.parametrize("time_chunk", [64, 0])
def test_noalloc_matches_scan_on_two_calls_in_a_row(time_chunk, disc):
    """Two different problems back to back (the second must not see the first's
    scratch): the no-allocation call runs the same kernels on the same plan as
    ssm_scan_fwd, so its results are identical bit for bit; the first problem is also
    checked against the fp64 oracle."""
    for i, seed in enumerate((201, 202)):
        p = W.scan_problem(2, 300 + seed % 7, 72, 16, io="bf16", seed=seed, h0=True)
        p.zoh = disc == "zoh"
        y, hf, y_ref, h_ref = _run_both(p, time_chunk, disc)
        assert np.all(np.isfinite(y)) and np.all(np.isfinite(hf))
        np.testing.assert_array_equal(y, y_ref)
        np.testing.assert_array_equal(hf, h_ref)
        if i == 0:
            yr, hr = oracle.scan(**p.oracle_args())
            assert_close(y, yr, "bf16", "no-alloc y", row_axes=(0, 2))
            assert_close(hf, hr, "bf16", "no-alloc h_final")


def test_noalloc_long_sequence_uses_the_scratch():
    """A sequence the library splits over time on its own (chunk summaries in scratch)."""
    p = W.scan_problem(1, 8192, 64, 16, io="f32", seed=203, h0=True)
    _, k, _ = bd.scan_plan(1, 8192, 64, 16, torch.float32)
    assert k > 1
    for _ in range(2):
        y, hf, y_ref, h_ref = _run_both(p, 0)
        np.testing.assert_array_equal(y, y_ref)
        np.testing.assert_array_equal(hf, h_ref)
    yr, hr = oracle.scan(**p.oracle_args())
    assert_close(y, yr, "f32", "no-alloc y (time split)", row_axes=(0, 2))
    assert_close(hf, hr, "f32", "no-alloc h_final (time split)")
