"""GPU parity of ssm_step_decode against the fp64 oracle (state carried across calls)."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_132_b300 as ssm
from selective_state_space_132_b300 import workloads as W

from _parity import Parity, assert_close, dev, host, io_dtype

pytestmark = pytest.mark.gpu


def _decode_run(p, steps, rows=None):
    """Run `steps` decode calls on the GPU and the oracle; compare every step's y
    (on `rows` of the batch, all rows when None) and the final state."""
    io = io_dtype(p.io)
    state = dev(p.state0)
    A, Dv, bias = dev(p.A), dev(p.D), dev(p.bias)
    sel = np.arange(p.batch) if rows is None else np.asarray(rows)
    ref_state = p.state0[sel].astype(np.float64).copy()
    ys, yrs = [], []
    for s in range(steps):
        tok = p.tokens(s)
        y = ssm.step_decode(state, dev(tok["x"], io), dev(tok["delta"], io), A, dev(tok["B"], io),
                            dev(tok["C"], io), D=Dv, z=dev(tok["z"], io), delta_bias=bias)
        ys.append(host(y)[sel])
        yrs.append(oracle.decode_step(ref_state, tok["x"][sel], tok["delta"][sel], p.A,
                                      tok["B"][sel], tok["C"][sel], Dv=p.D,
                                      z=None if tok["z"] is None else tok["z"][sel],
                                      bias=p.bias, softplus=True))
    torch.cuda.synchronize()
    assert_close(np.stack(ys), np.stack(yrs), p.io, "y over all steps")
    assert_close(host(state)[sel], ref_state, p.io, "state")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 4, 6, 16, 32, 64])
def test_decode_small(io, N):
    p = W.decode_problem(5, 37, N, 12, io=io, seed=40 + N)
    _decode_run(p, 12)


def test_decode_equals_scan():
    """L decode calls on the GPU equal one GPU scan over the same L tokens."""
    p = W.scan_problem(3, 24, 40, 16, io="f32", seed=50, h0=True)
    io = io_dtype(p.io)
    y_scan, h_scan = ssm.scan_fwd(dev(p.x, io), dev(p.delta, io), dev(p.A), dev(p.B, io),
                                  dev(p.C, io), D=dev(p.D), z=dev(p.z, io),
                                  delta_bias=dev(p.bias), h0=dev(p.h0))
    state = dev(p.h0)
    ys = []
    for t in range(p.seqlen):
        ys.append(ssm.step_decode(state, dev(p.x[:, t], io), dev(p.delta[:, t], io), dev(p.A),
                                  dev(p.B[:, t], io), dev(p.C[:, t], io), D=dev(p.D),
                                  z=dev(p.z[:, t], io), delta_bias=dev(p.bias)))
    y_dec = torch.stack(ys, dim=1)
    assert oracle.rel_l2(host(y_dec), host(y_scan)) < 2e-6
    assert oracle.rel_l2(host(state), host(h_scan)) < 2e-6


@pytest.mark.slow
def test_decode_full_size():
    """Reference workload: batch 256, d_inner 5120, N 16, fp32 state, bf16 tokens, 1000
    steps in place; every step's y for every sequence and channel, and the whole final
    state, against the streaming oracle.  Rows are the (b, d) channels over the steps."""
    p = W.config_problem(4)
    io = io_dtype(p.io)
    state = dev(p.state0)
    A, Dv, bias = dev(p.A), dev(p.D), dev(p.bias)
    ref_state = p.state0.astype(np.float64).copy()
    rows = p.batch * p.dim
    py = Parity(p.io, "y (decode, 1000 steps)", rows)
    for s in range(p.steps):
        tok = p.tokens(s)
        y = ssm.step_decode(state, dev(tok["x"], io), dev(tok["delta"], io), A, dev(tok["B"], io),
                            dev(tok["C"], io), D=Dv, z=dev(tok["z"], io), delta_bias=bias)
        yr = oracle.decode_step(ref_state, tok["x"], tok["delta"], p.A, tok["B"], tok["C"],
                                Dv=p.D, z=tok["z"], bias=p.bias, softplus=True)
        py.add(host(y).reshape(rows, 1), yr.reshape(rows, 1))
    py.check()
    assert_close(host(state), ref_state, p.io, "state after 1000 steps")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_decode_zero_order_hold(io):
    p = W.decode_problem(4, 40, 16, 6, io=io, seed=150)
    io_t = io_dtype(p.io)
    state = dev(p.state0)
    ref = p.state0.astype(np.float64).copy()
    A, Dv, bias = dev(p.A), dev(p.D), dev(p.bias)
    for s in range(6):
        tok = p.tokens(s)
        y = ssm.step_decode(state, dev(tok["x"], io_t), dev(tok["delta"], io_t), A,
                            dev(tok["B"], io_t), dev(tok["C"], io_t), D=Dv, z=dev(tok["z"], io_t),
                            delta_bias=bias, discretization="zoh")
        yr = oracle.decode_step(ref, tok["x"], tok["delta"], p.A, tok["B"], tok["C"], Dv=p.D,
                                z=tok["z"], bias=p.bias, zoh=True)
        assert_close(host(y), yr, p.io, f"y step {s}")
    assert_close(host(state), ref, p.io, "state")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_decode_four_rows_per_thread_ragged_batch(io):
    """Enough rows for the kernel to give each thread four batch rows of its channel;
    130 rows leave a ragged last group of two."""
    p = W.decode_problem(130, 1024, 16, 3, io=io, seed=160)
    _decode_run(p, 3, rows=[0, 1, 2, 3, 64, 127, 128, 129])
