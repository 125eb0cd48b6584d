"""The method's degenerate cases on the GPU, against the oracle: a zero step (the state
passes through unchanged), a huge step (the state forgets at once) and no decay
(A = 0: the state accumulates), for the scan, the SSD kernel, the decode step and the
backward."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_132_b300 as ssm
from selective_state_space_132_b300 import workloads as W

from _parity import assert_close, dev, host, io_dtype, run_scan, run_ssd, ssd_tc_allowance

pytestmark = pytest.mark.gpu


def _degenerate(p, kind):
    if kind == "zero_step":          # dl = 0 exactly: softplus off, no bias, raw 0
        p.softplus, p.bias = False, None
        p.delta = np.zeros_like(p.delta)
    elif kind == "huge_step":        # dl = softplus(40) = 40: exp(40 A) underflows to 0
        p.delta = np.full_like(p.delta, 40.0)
        p.bias = None
    elif kind == "no_decay":         # A = 0 on every other channel / head
        p.A[::2] = 0.0
    return p


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("kind", ["zero_step", "huge_step", "no_decay"])
@pytest.mark.parametrize("N", [16, 5])
def test_scan(io, kind, N):
    p = _degenerate(W.scan_problem(2, 150, 64, N, io=io, seed=50, h0=True), kind)
    y, hf = run_scan(p)
    yr, hr = oracle.scan(**p.oracle_args())
    assert_close(y, yr, io, f"y ({kind})")
    assert_close(hf, hr, io, f"h_final ({kind})")
    if kind == "zero_step":
        # the state passes through and y = (C h0 + D x) silu(z)
        np.testing.assert_array_equal(hf, p.h0)
        x, z = p.x.astype(np.float64), p.z.astype(np.float64)
        ch = np.einsum("bln,bdn->bld", p.C.astype(np.float64), p.h0.astype(np.float64))
        closed = (ch + p.D[None, None, :] * x) * z / (1 + np.exp(-z))
        assert_close(y, closed, io, "closed form")


@pytest.mark.parametrize("kind", ["zero_step", "huge_step", "no_decay"])
def test_ssd_tensor_core(kind):
    p = _degenerate(W.ssd_problem(1, 300, 4, 64, 1, 128, chunk=128, io="bf16", seed=51, h0=True),
                    kind)
    ay, ah = ssd_tc_allowance(p)
    y, hf = run_ssd(p)
    yr, hr = oracle.ssd(**p.oracle_args())
    assert_close(y, yr, "bf16", f"y ({kind})", allow=ay)
    assert_close(hf, hr, "bf16", f"h_final ({kind})", allow=ah)


@pytest.mark.parametrize("kind", ["zero_step", "huge_step", "no_decay"])
def test_decode(kind):
    p = W.decode_problem(4, 64, 16, 2, io="f32", seed=52)
    if kind == "no_decay":
        p.A[::2] = 0.0
    state = dev(p.state0)
    ref = p.state0.astype(np.float64).copy()
    for s in range(2):
        tok = p.tokens(s)
        if kind == "zero_step":
            tok["delta"] = np.zeros_like(tok["delta"])
        if kind == "huge_step":
            tok["delta"] = np.full_like(tok["delta"], 40.0)
        sp = kind != "zero_step"
        bias = None if kind in ("zero_step", "huge_step") else p.bias
        y = ssm.step_decode(state, dev(tok["x"]), dev(tok["delta"]), dev(p.A), dev(tok["B"]),
                            dev(tok["C"]), D=dev(p.D), z=dev(tok["z"]), delta_bias=dev(bias),
                            delta_softplus=sp)
        yr = oracle.decode_step(ref, tok["x"], tok["delta"], p.A, tok["B"], tok["C"], Dv=p.D,
                                z=tok["z"], bias=bias, softplus=sp)
        torch.cuda.synchronize()
        assert_close(host(y), yr, "f32", f"y ({kind})")
    assert_close(host(state), ref, "f32", f"state ({kind})")
    if kind == "zero_step":
        np.testing.assert_array_equal(host(state), p.state0)


@pytest.mark.parametrize("kind", ["zero_step", "huge_step", "no_decay"])
def test_scan_bwd(kind):
    p = _degenerate(W.scan_problem(2, 90, 40, 16, io="f32", seed=53, h0=True), kind)
    rng = np.random.default_rng(54)
    gy = rng.standard_normal((2, 90, 40)).astype(np.float32)
    g = ssm.scan_bwd(dev(gy), dev(p.x), dev(p.delta), dev(p.A), dev(p.B), dev(p.C), D=dev(p.D),
                     z=dev(p.z), delta_bias=dev(p.bias), delta_softplus=p.softplus,
                     h0=dev(p.h0))
    torch.cuda.synchronize()
    ref = oracle.scan_bwd(gy, p.x, p.delta, p.A, p.B, p.C, Dv=p.D, z=p.z, bias=p.bias,
                          softplus=p.softplus, h0=p.h0)
    for mine, theirs in (("dx", "gx"), ("ddelta", "gdelta"), ("dA", "gA"), ("dB", "gB"),
                         ("dC", "gC"), ("dD", "gD"), ("ddelta_bias", "gbias"), ("dh0", "gh0"),
                         ("dz", "gz")):
        got, want = host(g[mine]), ref[theirs]
        assert np.all(np.isfinite(got)), mine
        if np.linalg.norm(want) == 0:
            assert np.all(got == 0), mine
        else:
            assert_close(got, want, "f32", f"{mine} ({kind})")
