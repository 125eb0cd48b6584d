"""GPU parity of ssm_scan_bwd (gradients with recomputed states) against the fp64
adjoint oracle, on the same seeded inputs (rounded to the I/O type first)."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_132_b300 as ssm
from selective_state_space_132_b300 import workloads as W

from _parity import assert_close, dev, host, io_dtype

pytestmark = pytest.mark.gpu

_NAMES = [("dx", "gx"), ("ddelta", "gdelta"), ("dA", "gA"), ("dB", "gB"), ("dC", "gC"),
          ("dD", "gD"), ("ddelta_bias", "gbias"), ("dh0", "gh0"), ("dz", "gz")]


def _run(p, seed, zoh=False, dh_final=True, rows=None, check_sums=True):
    io = io_dtype(p.io)
    rng = np.random.default_rng(seed)
    gy = rng.standard_normal((p.batch, p.seqlen, p.dim)).astype(np.float32)
    ghf = rng.standard_normal((p.batch, p.dim, p.dstate)).astype(np.float32) if dh_final else None
    gy_d = dev(gy, io)
    disc = "zoh" if zoh else "euler"
    g = ssm.scan_bwd(gy_d, dev(p.x, io), dev(p.delta, io), dev(p.A), dev(p.B, io), dev(p.C, io),
                     D=dev(p.D), z=dev(p.z, io), delta_bias=dev(p.bias),
                     delta_softplus=p.softplus, h0=dev(p.h0), dh_final=dev(ghf),
                     discretization=disc)
    torch.cuda.synchronize()
    sel = slice(None) if rows is None else rows
    rnd = lambda a: None if a is None else host(dev(a, io))[sel]          # noqa: E731
    ref = oracle.scan_bwd(rnd(gy), rnd(p.x), rnd(p.delta), p.A, rnd(p.B), rnd(p.C), Dv=p.D,
                          z=rnd(p.z), bias=p.bias, softplus=p.softplus,
                          h0=None if p.h0 is None else p.h0[sel],
                          gh_final=None if ghf is None else ghf[sel], zoh=zoh)
    errs = {}
    for mine, theirs in _NAMES:
        if theirs not in ref:
            continue
        if mine in ("dA", "dD", "ddelta_bias") and not check_sums:
            continue
        got = host(g[mine])
        if mine not in ("dA", "dD", "ddelta_bias"):
            got = got[sel]
        errs[mine] = assert_close(got, ref[theirs], p.io, mine)
    return errs


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [16, 4, 1, 5, 8, 32, 64])
def test_scan_bwd(io, N):
    # 3 batch rows, 2 channel blocks (the second ragged), several tiles with a ragged tail
    p = W.scan_problem(3, 77, 45, N, io=io, seed=300 + N, h0=True)
    _run(p, seed=N)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [16, 5])
def test_scan_bwd_zero_order_hold(io, N):
    p = W.scan_problem(2, 70, 40, N, io=io, seed=320 + N, h0=True)
    p.A[3, :] = 0.0                                    # the A -> 0 limit
    p.A[5, :] = -1e-3
    _run(p, seed=7, zoh=True)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_scan_bwd_without_optional_inputs(io):
    p = W.scan_problem(2, 50, 33, 16, io=io, seed=330, gate=False, use_D=False,
                       use_bias=False, softplus=False)
    p.delta = np.abs(p.delta) * 0.2 + 0.01            # positive steps without softplus
    if io == "bf16":
        p.delta = host(dev(p.delta, torch.bfloat16)).astype(np.float32)
    _run(p, seed=8, dh_final=False)


def test_scan_bwd_single_step_and_empty():
    p = W.scan_problem(2, 1, 16, 16, io="f32", seed=340, h0=True)
    _run(p, seed=9)
    x = torch.empty(2, 0, 16, device="cuda")
    A = -torch.ones(16, 16, device="cuda")
    e = torch.empty(2, 0, 16, device="cuda")
    dhf = torch.randn(2, 16, 16, device="cuda")
    g = ssm.scan_bwd(e, x, e, A, e[..., :16], e[..., :16], dh_final=dhf)
    torch.cuda.synchronize()
    assert torch.equal(g["dh0"], dhf)                  # no steps: the gradient passes through
    assert torch.count_nonzero(g["dA"]) == 0


def test_scan_bwd_time_reversal_consistency_with_forward():
    """<dy, y(x + e v)> - <dy, y(x - e v)> over 2e equals <dx, v> (GPU forward, GPU
    backward): the two GPU entry points agree with each other in fp32."""
    p = W.scan_problem(1, 64, 32, 16, io="f32", seed=350, h0=True)
    rng = np.random.default_rng(5)
    gy = rng.standard_normal(p.x.shape).astype(np.float32)
    v = rng.standard_normal(p.x.shape).astype(np.float32)
    args = lambda xx: (dev(xx), dev(p.delta), dev(p.A), dev(p.B), dev(p.C))   # noqa: E731
    kw = dict(D=dev(p.D), z=dev(p.z), delta_bias=dev(p.bias), h0=dev(p.h0))
    eps = 1e-2
    yp, _ = ssm.scan_fwd(*args(p.x + eps * v), **kw)
    ym, _ = ssm.scan_fwd(*args(p.x - eps * v), **kw)
    g = ssm.scan_bwd(dev(gy), *args(p.x), **kw)
    torch.cuda.synchronize()
    fd = float(np.sum(gy * (host(yp) - host(ym)))) / (2 * eps)
    an = float(np.sum(host(g["dx"]) * v))
    assert abs(fd - an) <= 1e-4 * max(1.0, abs(an))


@pytest.mark.slow
def test_scan_bwd_block_shape_full():
    """The 130M layer's shape (batch 8, length 2048, d_inner 1536, N 16, bf16): every
    gradient, the per-row ones and the sums over batch rows and channels, against the
    oracle's adjoint of the whole problem."""
    _run(W.config_problem(1), seed=11)
