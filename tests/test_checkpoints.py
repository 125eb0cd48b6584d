"""State checkpoints kept from the forward pass for the backward pass
(ssm_scan_fwd_ckpt / ssm_scan_bwd_ckpt).

The forward scan also writes the state before every T-th step; the checkpoints are
checked against the oracle's states at those steps (the final state of the oracle run
on each prefix), and the backward pass that starts from them against the oracle's
adjoint.  Host-side argument checks run without a GPU."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import selective_state_space_132_b300 as ssm
from selective_state_space_132_b300 import binding as bd
from selective_state_space_132_b300 import workloads as W

from _parity import assert_close, dev, host, io_dtype

OK, INVALID, ALIGN = 0, 1, 3


# ---------------------------------------------------------------- host side (no GPU)
def _scan(**kw):
    base = dict(batch=2, seqlen=64, dim=32, dstate=16, time_chunk=0, io_dtype=1,
                delta_softplus=1, x=0x10000, delta=0x20000, B=0x30000, C=0x40000, z=None,
                A=0x50000, D=None, delta_bias=None, h0=None, y=0x60000, h_final=None,
                workspace=None, workspace_bytes=0)
    base.update(kw)
    return bd.ScanArgs(**base)


def test_checkpoint_size_and_steps():
    lib = ssm.load_library()
    steps, nbytes = ctypes.c_int64(0), ctypes.c_size_t(0)
    for N, T in [(1, 32), (8, 32), (9, 16), (16, 16), (17, 8), (32, 8), (33, 4), (64, 4)]:
        a = _scan(dstate=N, seqlen=100)
        assert lib.ssm_scan_ckpt_size(ctypes.byref(a), ctypes.byref(steps),
                                      ctypes.byref(nbytes)) == OK
        assert steps.value == T
        # (B, ceil(L / T), D, N) fp32
        assert nbytes.value == 2 * (-(-100 // T)) * 32 * N * 4
    assert ssm.scan_ckpt_shape(8, 2048, 1536, 16) == (8, 128, 1536, 16)
    assert lib.ssm_scan_ckpt_size(None, ctypes.byref(steps), ctypes.byref(nbytes)) == INVALID
    assert lib.ssm_scan_ckpt_size(ctypes.byref(_scan(dstate=0)), ctypes.byref(steps),
                                  ctypes.byref(nbytes)) == INVALID


def test_checkpoint_calls_reject_bad_buffers_on_the_host():
    """Every case returns from the host checks before any CUDA call (the pointers are
    never dereferenced)."""
    lib = ssm.load_library()
    a = _scan()
    need = 2 * 4 * 32 * 16 * 4
    base = 0x1000000
    assert lib.ssm_scan_fwd_ckpt(ctypes.byref(a), None, need, None) == INVALID
    assert lib.ssm_scan_fwd_ckpt(ctypes.byref(a), base, need - 4, None) == INVALID
    assert lib.ssm_scan_fwd_ckpt(ctypes.byref(a), base + 8, need, None) == ALIGN
    assert lib.ssm_scan_fwd_ckpt(ctypes.byref(a), 0x60000, need, None) == INVALID  # over y
    assert lib.ssm_scan_fwd_ckpt(ctypes.byref(a), 0x2f000, need, None) == INVALID  # over B
    assert lib.ssm_scan_fwd_ckpt(ctypes.byref(_scan(x=0x10001)), base, need, None) == ALIGN
    b = bd.ScanBwdArgs(batch=2, seqlen=64, dim=32, dstate=16, io_dtype=1, delta_softplus=1,
                       discretization=0, reserved=0, x=0x100000, delta=0x200000, B=0x300000,
                       C=0x400000, z=None, A=0x500000, D=None, delta_bias=None, h0=None,
                       dy=0x600000, dh_final=None, dx=0x700000, ddelta=0x800000, dz=None,
                       dA=0x900000, dB=0xa00000, dC=0xb00000, dD=None, ddelta_bias=None,
                       dh0=None, workspace=None, workspace_bytes=0)
    assert lib.ssm_scan_bwd_ckpt(ctypes.byref(b), None, need, None) == INVALID
    assert lib.ssm_scan_bwd_ckpt(ctypes.byref(b), base, need - 4, None) == INVALID
    assert lib.ssm_scan_bwd_ckpt(ctypes.byref(b), base + 4, need, None) == ALIGN


# ---------------------------------------------------------------- GPU
def _oracle_states(p, T):
    """The oracle's state before every step t = s T: h0 (or zero) at t = 0, else the
    final state of the oracle scan of the first t steps."""
    L = p.seqlen
    out = []
    for t in range(0, L, T):
        if t == 0:
            out.append(np.zeros((p.batch, p.dim, p.dstate)) if p.h0 is None else p.h0)
            continue
        args = p.oracle_args()
        for k in ("x", "delta", "Bm", "Cm", "z"):
            if args[k] is not None:
                args[k] = args[k][:, :t]
        out.append(oracle.scan(**args)[1])
    return np.stack(out, axis=1)            # (B, ceil(L / T), D, N)


def _fwd(p, zoh, time_chunk, checkpoints):
    io = io_dtype(p.io)
    return ssm.scan_fwd(dev(p.x, io), dev(p.delta, io), dev(p.A), dev(p.B, io), dev(p.C, io),
                        D=dev(p.D), z=dev(p.z, io), delta_bias=dev(p.bias),
                        delta_softplus=p.softplus, h0=dev(p.h0), time_chunk=time_chunk,
                        discretization="zoh" if zoh else "euler", checkpoints=checkpoints)


# (io, N, D, time_chunk, zoh): the TMA kernel (bf16 with D a multiple of 8, fp32 with N a
# multiple of 4), the general kernel (ragged D or N), whole and split over time chunks
CASES = [("bf16", 16, 64, 0, False), ("bf16", 16, 64, 64, False), ("bf16", 16, 45, 96, False),
         ("f32", 4, 40, 0, False), ("f32", 5, 33, 64, True), ("bf16", 64, 32, 0, False),
         ("bf16", 8, 48, 128, True), ("f32", 32, 36, 0, False)]


@pytest.mark.gpu
@pytest.mark.parametrize("io,N,D,tc,zoh", CASES)
def test_forward_checkpoints_are_the_scan_states(io, N, D, tc, zoh):
    p = W.scan_problem(2, 300, D, N, io=io, seed=500 + N + D, h0=True)
    p.zoh = zoh
    y0, h0f = _fwd(p, zoh, tc, None)
    y, hf, ck = _fwd(p, zoh, tc, True)
    torch.cuda.synchronize()
    # the outputs are those of the plain call, bit for bit
    assert torch.equal(y, y0) and torch.equal(hf, h0f)
    T = ssm.scan_ckpt_steps(N)
    assert ck.shape == (2, -(-300 // T), D, N)
    ref = _oracle_states(p, T)
    assert_close(host(ck), ref, p.io, "checkpoints", row_axes=(0, 2, 3))


def _grads(p, seed, zoh, checkpoints, time_chunk=0):
    io = io_dtype(p.io)
    rng = np.random.default_rng(seed)
    gy = rng.standard_normal((p.batch, p.seqlen, p.dim)).astype(np.float32)
    ghf = rng.standard_normal((p.batch, p.dim, p.dstate)).astype(np.float32)
    ck = None
    if checkpoints:
        ck = _fwd(p, zoh, time_chunk, True)[2]
    g = ssm.scan_bwd(dev(gy, io), dev(p.x, io), dev(p.delta, io), dev(p.A), dev(p.B, io),
                     dev(p.C, io), D=dev(p.D), z=dev(p.z, io), delta_bias=dev(p.bias),
                     delta_softplus=p.softplus, h0=dev(p.h0), dh_final=dev(ghf),
                     discretization="zoh" if zoh else "euler", checkpoints=ck)
    torch.cuda.synchronize()
    return g, gy, ghf


@pytest.mark.gpu
@pytest.mark.parametrize("io,N,D,tc,zoh", CASES[:5])
def test_backward_from_forward_checkpoints(io, N, D, tc, zoh):
    """The backward pass that starts from the forward pass's checkpoints (ragged last
    tile: L = 300) against the fp64 adjoint, gradient by gradient."""
    p = W.scan_problem(2, 300, D, N, io=io, seed=520 + N + D, h0=True)
    p.zoh = zoh
    g, gy, ghf = _grads(p, 11, zoh, True, tc)
    io_t = io_dtype(p.io)
    rnd = lambda a: None if a is None else host(dev(a, io_t))          # noqa: E731
    ref = oracle.scan_bwd(rnd(gy), rnd(p.x), rnd(p.delta), p.A, rnd(p.B), rnd(p.C), Dv=p.D,
                          z=rnd(p.z), bias=p.bias, softplus=p.softplus, h0=p.h0,
                          gh_final=ghf, zoh=zoh)
    for mine, theirs in [("dx", "gx"), ("ddelta", "gdelta"), ("dA", "gA"), ("dB", "gB"),
                         ("dC", "gC"), ("dD", "gD"), ("ddelta_bias", "gbias"),
                         ("dh0", "gh0"), ("dz", "gz")]:
        if theirs in ref and mine in g:
            assert_close(host(g[mine]), ref[theirs], p.io, mine)


@pytest.mark.gpu
def test_backward_from_checkpoints_matches_recomputation():
    """Unsplit forward on the TMA kernel: its checkpoints are the states the backward
    kernel computes itself, so both backward calls return the same gradients."""
    p = W.scan_problem(2, 300, 64, 16, io="bf16", seed=540, h0=True)
    g1, _, _ = _grads(p, 12, False, False)
    g2, _, _ = _grads(p, 12, False, True)
    for k in g1:
        a, b = host(g1[k]), host(g2[k])
        # dA, dB, dC, dD and dbias are sums with atomic adds in any order
        tol = 0 if k in ("dx", "ddelta", "dz", "dh0") else 1e-5 * (np.abs(a).max() + 1e-30)
        assert np.max(np.abs(a - b)) <= tol, k


@pytest.mark.gpu
def test_autograd_with_checkpoint_states():
    p = W.scan_problem(2, 200, 64, 16, io="f32", seed=550, h0=True)
    grads = []
    for keep in (False, True):
        ins = [dev(a).requires_grad_() for a in (p.x, p.delta, p.A, p.B, p.C, p.D, p.z,
                                                 p.bias, p.h0)]
        x, dl, A, B, C, Dv, z, bias, h0 = ins
        y, hf = ssm.selective_scan(x, dl, A, B, C, D=Dv, z=z, delta_bias=bias, h0=h0,
                                   checkpoint_states=keep)
        (y.square().sum() + hf.sum()).backward()
        grads.append([t.grad.detach().cpu().numpy().astype(np.float64) for t in ins])
    for a, b in zip(*grads):
        assert np.allclose(a, b, rtol=1e-4, atol=1e-5 * (np.abs(a).max() + 1e-30))
