"""Failure detection without a GPU fault: every spin-wait in the kernels is bounded.

ssm_check_bounded_wait runs one thread that waits, through the same acquire-and-back-off
routine the SSD kernel uses to take over the state of the block before it, on a flag
nothing sets.  The wait must give up, the status word must say SSM_ERR_TIMEOUT, and the
CUDA context must stay usable for the next call."""
import ctypes
import time

import numpy as np
import pytest

import oracle
from selective_state_space_132_b300 import binding as bd
from selective_state_space_132_b300 import workloads as W

TIMEOUT = 6


def test_bounded_wait_rejects_bad_arguments_on_host():
    lib = bd.load_library()
    assert lib.ssm_check_bounded_wait(None, 1000, None) == 1          # no workspace
    assert lib.ssm_check_bounded_wait(0x10000, 0, None) == 1          # empty budget
    assert lib.ssm_check_bounded_wait(0x10000, 3_000_000_000, None) == 1
    assert lib.ssm_check_bounded_wait(0x10010, 1000, None) == 3       # unaligned


@pytest.mark.gpu
def test_expired_wait_reports_timeout_and_context_survives():
    import torch
    from _parity import run_scan, assert_close

    lib = bd.load_library()
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.time()
    assert lib.ssm_check_bounded_wait(ws.data_ptr(), 2_000_000, stream) == 0
    assert bd.read_device_status(ws) == TIMEOUT
    assert time.time() - t0 < 30.0
    # the context is still usable: a normal call runs and is correct
    p = W.scan_problem(1, 70, 32, 16, io="bf16", seed=11)
    y, _ = run_scan(p)
    yr, _ = oracle.scan(**p.oracle_args())
    assert_close(y, yr, "bf16", "y after an expired wait")


def test_lookback_self_test_rejects_bad_arguments_on_host():
    import torch
    lib = bd.load_library()
    a = bd.ScanArgs(1, 8192, 64, 16, 0, 1, 1, None, None, None, None, None, None, None, None,
                    None, None, None, None, 0)
    assert lib.ssm_check_scan_lookback(ctypes.byref(a), 0, None) == 1          # empty budget
    assert lib.ssm_check_scan_lookback(None, 1000, None) == 1                  # no arguments
    one = bd.ScanArgs(1, 64, 64, 16, 0, 1, 1, None, None, None, None, None, None, None, None,
                      None, None, None, None, 0)
    assert lib.ssm_check_scan_lookback(ctypes.byref(one), 1000, None) in (1, 2)


@pytest.mark.gpu
def test_scan_lookback_wait_times_out_and_context_survives():
    """The single-launch scan with its chunk summaries left unpublished: the blocks of the
    later chunks wait for a predecessor that never publishes, give up after the budget,
    record SSM_ERR_TIMEOUT and return; the next normal call runs and is correct."""
    import torch
    from _parity import assert_close, dev, run_scan

    lib = bd.load_library()
    p = W.scan_problem(1, 4096, 64, 16, io="bf16", seed=12)
    cl, k, launches = bd.scan_plan(1, 4096, 64, 16, torch.bfloat16, time_chunk=1024)
    assert k == 4 and launches == 1
    io = torch.bfloat16
    x, dl, B, C, z = dev(p.x, io), dev(p.delta, io), dev(p.B, io), dev(p.C, io), dev(p.z, io)
    A, D, bias = dev(p.A), dev(p.D), dev(p.bias)
    y = torch.zeros_like(x)
    hf = torch.zeros((1, 64, 16), dtype=torch.float32, device="cuda")
    args = bd._scan_args(x, dl, A, B, C, D, z, bias, True, None, y, hf, 1024)
    ws = torch.empty(bd.scan_workspace_size(1, 4096, 64, 16, io, 1024), dtype=torch.uint8,
                     device="cuda")
    args.workspace, args.workspace_bytes = ws.data_ptr(), ws.numel()
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.time()
    assert lib.ssm_check_scan_lookback(ctypes.byref(args), 2_000_000, stream) == 0
    assert bd.read_device_status(ws) == TIMEOUT
    assert time.time() - t0 < 30.0
    # the first chunk needs no predecessor: its outputs were written and are correct
    yr, hr = oracle.scan(**p.oracle_args())
    assert_close(y[:, :1024].float().cpu().numpy().astype(np.float64), yr[:, :1024], "bf16",
                 "first chunk")
    # a normal call on the same workspace runs, reports no timeout and is correct
    y2, h2 = run_scan(p, time_chunk=1024)
    assert_close(y2, yr, "bf16", "y after an expired look-back", row_axes=(0, 2))
    assert_close(h2, hr, "bf16", "h_final after an expired look-back")
