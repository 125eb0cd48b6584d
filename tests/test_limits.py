"""Sizes at the edges of the launch grids and of the time split: the largest batch the
scan accepts (one grid row per batch row), a million-step sequence (hundreds of time
chunks), a very wide channel count, and the same for conv1d and the backward."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_132_b300 as ssm
from selective_state_space_132_b300 import workloads as W

from _parity import assert_close, dev, host, io_dtype, run_scan

pytestmark = pytest.mark.gpu


def test_scan_largest_batch():
    """65535 batch rows (the grid's y limit), checked on sampled rows."""
    p = W.scan_problem(65535, 3, 32, 16, io="bf16", seed=40)
    y, hf = run_scan(p)
    rows = [0, 1, 12345, 40000, 65534]
    sub = dict(p.oracle_args())
    for k in ("x", "delta", "Bm", "Cm", "z"):
        sub[k] = sub[k][rows]
    yr, hr = oracle.scan(**sub)
    assert_close(y[rows], yr, "bf16", "y")
    assert_close(hf[rows], hr, "bf16", "h_final")
    assert ssm.scan_plan(65535, 3, 32, 16)[2] == 1


@pytest.mark.slow
def test_scan_million_steps():
    """One batch row of 2^20 steps over 32 channels: the plan cuts it into hundreds of
    time chunks whose summaries are published and folded in one launch."""
    p = W.scan_problem(1, 1 << 20, 32, 16, io="bf16", seed=41)
    cl, k, launches = ssm.scan_plan(1, 1 << 20, 32, 16)
    assert k > 100 and launches == 1
    y, hf = run_scan(p)
    yr, hr = oracle.scan(**p.oracle_args())
    assert_close(y, yr, "bf16", "y")
    assert_close(hf, hr, "bf16", "h_final")


def test_scan_wide_channels():
    p = W.scan_problem(1, 64, 1 << 17, 16, io="bf16", seed=42)
    y, hf = run_scan(p)
    yr, hr = oracle.scan(**p.oracle_args())
    assert_close(y, yr, "bf16", "y")
    assert_close(hf, hr, "bf16", "h_final")


def test_conv1d_million_steps():
    rng = np.random.default_rng(43)
    t = torch.bfloat16
    x = rng.standard_normal((1, 1 << 20, 64)).astype(np.float32)
    w = rng.standard_normal((64, 4)).astype(np.float32) / 2
    xd = dev(x, t)
    out = ssm.conv1d(xd, dev(w))
    torch.cuda.synchronize()
    ref = oracle.conv1d(host(xd), w)
    assert_close(host(out), ref, "bf16", "conv1d")


@pytest.mark.parametrize("nb,L,D", [(2048, 40, 32), (1, 1 << 16, 32)])
def test_scan_bwd_at_limits(nb, L, D):
    """Many batch rows, and one long sequence (4096 checkpoint tiles), sampled rows."""
    p = W.scan_problem(nb, L, D, 16, io="f32", seed=44, h0=True)
    rng = np.random.default_rng(45)
    gy = rng.standard_normal((nb, L, D)).astype(np.float32)
    g = ssm.scan_bwd(dev(gy), dev(p.x), dev(p.delta), dev(p.A), dev(p.B), dev(p.C), D=dev(p.D),
                     z=dev(p.z), delta_bias=dev(p.bias), h0=dev(p.h0))
    torch.cuda.synchronize()
    rows = [0, nb // 2, nb - 1] if nb > 1 else [0]
    ref = oracle.scan_bwd(gy[rows], p.x[rows], p.delta[rows], p.A, p.B[rows], p.C[rows],
                          Dv=p.D, z=p.z[rows], bias=p.bias, h0=p.h0[rows])
    for mine, theirs in (("dx", "gx"), ("ddelta", "gdelta"), ("dB", "gB"), ("dC", "gC"),
                         ("dz", "gz"), ("dh0", "gh0")):
        assert_close(host(g[mine])[rows], ref[theirs], "f32", mine)
    if nb == 1:
        for mine, theirs in (("dA", "gA"), ("dD", "gD"), ("ddelta_bias", "gbias")):
            assert_close(host(g[mine]), ref[theirs], "f32", mine)
