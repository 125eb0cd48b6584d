"""GPU parity of ssm_scan_fwd against the fp64 oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_132_b300 import workloads as W

from _parity import Parity, assert_close, run_scan

pytestmark = pytest.mark.gpu


def _check(p, time_chunk=0, h_final=True):
    """y is compared with channels (b, d) as rows (each a channel over time), so one
    wrong carry or one wrong tile of a channel shows in its row; h_final by (b, d)."""
    y, hf = run_scan(p, time_chunk=time_chunk, h_final=h_final)
    yr, hr = oracle.scan(**p.oracle_args())
    assert np.all(np.isfinite(y))
    e_y = assert_close(y, yr, p.io, "y", row_axes=(0, 2))
    e_h = assert_close(hf, hr, p.io, "h_final") if h_final else 0.0
    return e_y, e_h


def test_tiny_fp32_workload():
    """Reference workload: fp32, batch 1, d_inner 16, L 64, N 4, gate on."""
    _check(W.config_problem(0))


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 3, 4, 5, 8, 12, 16, 24, 32, 33, 64])
def test_state_sizes(io, N):
    p = W.scan_problem(2, 83, 40, N, io=io, seed=100 + N, A="random")
    _check(p)


@pytest.mark.parametrize("gate,use_D,use_bias,softplus,h0", [
    (False, True, True, True, False),
    (True, False, True, True, True),
    (True, True, False, True, True),
    (True, True, True, False, False),
    (False, False, False, False, True),
])
def test_optional_inputs(gate, use_D, use_bias, softplus, h0):
    p = W.scan_problem(3, 150, 70, 16, io="bf16", seed=7, gate=gate, use_D=use_D,
                       use_bias=use_bias, softplus=softplus, h0=h0)
    if not softplus:  # keep the step positive: small |raw| plus a small positive bias
        p.delta = W.round_bf16(np.abs(p.delta) * np.float32(0.1))
        if p.bias is not None:
            p.bias = np.abs(p.bias) * np.float32(0.01)
    _check(p)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("time_chunk", [32, 64, 96, 224])
def test_forced_time_split_carry(io, time_chunk):
    """Several blocks along time joined by the chunk-summary carry."""
    p = W.scan_problem(2, 300, 72, 16, io=io, seed=21, h0=True)
    _check(p, time_chunk=time_chunk)


def test_time_split_matches_single_pass_closely():
    p = W.scan_problem(2, 1000, 64, 16, io="f32", seed=22, h0=True)
    y1, h1 = run_scan(p)
    y2, h2 = run_scan(p, time_chunk=128)
    assert oracle.rel_l2(y2, y1) < 2e-6 and oracle.rel_l2(h2, h1) < 2e-6


def test_ragged_and_empty():
    _check(W.scan_problem(1, 1, 1, 16, io="bf16", seed=3))              # one step, one channel
    _check(W.scan_problem(2, 33, 33, 16, io="bf16", seed=4, h0=True))   # ragged tile and block
    p = W.scan_problem(2, 0, 24, 16, io="f32", seed=5, h0=True)         # empty sequence
    y, hf = run_scan(p)
    assert y.shape == (2, 0, 24)
    np.testing.assert_array_equal(hf, p.h0.astype(np.float64))


def test_no_final_state_and_other_stream():
    p = W.scan_problem(2, 70, 48, 16, io="bf16", seed=6)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y, hf = run_scan(p, h_final=False, stream=s)
    assert hf is None
    yr, _ = oracle.scan(**p.oracle_args())
    assert_close(y, yr, "bf16", "y")


def test_deterministic_bitwise():
    p = W.scan_problem(2, 200, 64, 16, io="bf16", seed=8)
    a = run_scan(p, time_chunk=64)
    b = run_scan(p, time_chunk=64)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.slow
def test_mamba130m_layer_full_size():
    """Reference workload: bf16, batch 8, d_inner 1536, L 2048, N 16, compared in full."""
    _check(W.config_problem(1))


@pytest.mark.slow
def test_long_context_full_size():
    """Reference workload: bf16, batch 1, d_inner 2048, L 131072, N 16, run in full on the
    GPU (multi-block carry along time) and compared with the oracle on every output and
    every final state, in blocks of 256 channels (each block is an independent oracle
    call over the whole sequence)."""
    p = W.config_problem(2)
    y, hf = run_scan(p)
    py = Parity("bf16", "y (long context)", p.batch * p.dim)
    ph = Parity("bf16", "h_final (long context)", p.batch * p.dim)
    for d0 in range(0, p.dim, 256):
        sel = slice(d0, min(p.dim, d0 + 256))
        args = p.oracle_args()
        for k in ("x", "delta", "z"):
            args[k] = np.ascontiguousarray(getattr(p, k)[:, :, sel])
        args["A"], args["Dv"], args["bias"] = p.A[sel], p.D[sel], p.bias[sel]
        yr, hr = oracle.scan(**args)
        # rows (b, d) over time; batch 1, so the row of channel d is d
        py.add(y[0, :, sel].T, yr[0].T, rows=sel)
        ph.add(hf[0, sel], hr[0], rows=sel)
    py.check()
    ph.check()


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N,time_chunk", [(16, 0), (16, 64), (5, 0), (64, 96)])
def test_zero_order_hold(io, N, time_chunk):
    """B̄ = (exp(dl A) - 1) / A B (the tildalice page's zero-order hold): TMA and general
    kernels, single pass and time split, including a channel with A = 0 (limit dl B)."""
    p = W.scan_problem(2, 150, 40, N, io=io, seed=140 + N, h0=True, A="random")
    p.A[3, :] = 0.0
    p.zoh = True
    _check(p, time_chunk=time_chunk)
