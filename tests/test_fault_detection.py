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
