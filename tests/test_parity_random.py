"""Seeded random parity cases: every GPU entry point against the oracle on randomly
drawn ragged shapes, dtypes and optional-input combinations (a fixed list, the same
on every run)."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_132_b300 as ssm
from selective_state_space_132_b300 import workloads as W

from _parity import TOL, assert_close, dev, host, io_dtype, run_scan, run_ssd, ssd_tc_allowance

pytestmark = pytest.mark.gpu

CASES = 24


def _positive_steps(p, io, rng):
    """Without softplus the raw step plus the bias is the step: keep both positive and
    small (the bias recipe stores inv_softplus of a small step, which is negative)."""
    p.delta = np.abs(p.delta) * 0.2 + 0.01
    if io == "bf16":
        p.delta = host(dev(p.delta, torch.bfloat16)).astype(np.float32)
    if p.bias is not None:
        p.bias = rng.uniform(0.0, 0.05, p.bias.shape).astype(np.float32)


@pytest.mark.parametrize("case", range(CASES))
def test_random_scan(case):
    rng = np.random.default_rng(500 + case)
    io = ("f32", "bf16")[case % 2]
    nb, L, D = int(rng.integers(1, 4)), int(rng.integers(1, 300)), int(rng.integers(1, 100))
    N = int(rng.choice([1, 2, 3, 4, 5, 8, 12, 16, 23, 32, 48, 64]))
    gate, use_D, bias, sp, h0, zoh = (bool(v) for v in rng.integers(0, 2, 6))
    p = W.scan_problem(nb, L, D, N, io=io, seed=600 + case, gate=gate, use_D=use_D,
                       use_bias=bias, softplus=sp, h0=h0, A="random")
    if not sp:
        _positive_steps(p, io, rng)
    p.zoh = zoh
    tc = int(rng.choice([0, 0, 32, 64, 96]))
    y, hf = run_scan(p, time_chunk=tc)
    yr, hr = oracle.scan(**p.oracle_args())
    assert_close(y, yr, io, f"y (B {nb} L {L} D {D} N {N} chunk {tc} zoh {zoh})")
    assert_close(hf, hr, io, "h_final")


@pytest.mark.parametrize("case", range(CASES))
def test_random_scan_bwd(case):
    rng = np.random.default_rng(700 + case)
    io = ("f32", "bf16")[case % 2]
    nb, L, D = int(rng.integers(1, 3)), int(rng.integers(1, 120)), int(rng.integers(1, 70))
    N = int(rng.choice([1, 3, 4, 7, 8, 16, 20, 32, 64]))
    gate, use_D, bias, sp, h0, zoh = (bool(v) for v in rng.integers(0, 2, 6))
    p = W.scan_problem(nb, L, D, N, io=io, seed=800 + case, gate=gate, use_D=use_D,
                       use_bias=bias, softplus=sp, h0=h0, A="random")
    if not sp:
        _positive_steps(p, io, rng)
    t = io_dtype(io)
    gy = rng.standard_normal((nb, L, D)).astype(np.float32)
    ghf = rng.standard_normal((nb, D, N)).astype(np.float32) if case % 3 else None
    disc = "zoh" if zoh else "euler"
    ck = None
    if case % 4 >= 2:
        # half of the cases start the backward from the forward pass's checkpoints (the
        # forward whole or split over time chunks)
        ck = ssm.scan_fwd(dev(p.x, t), dev(p.delta, t), dev(p.A), dev(p.B, t), dev(p.C, t),
                          D=dev(p.D), z=dev(p.z, t), delta_bias=dev(p.bias),
                          delta_softplus=sp, h0=dev(p.h0), discretization=disc,
                          time_chunk=int(rng.choice([0, 32, 64])), checkpoints=True)[2]
    g = ssm.scan_bwd(dev(gy, t), dev(p.x, t), dev(p.delta, t), dev(p.A), dev(p.B, t),
                     dev(p.C, t), D=dev(p.D), z=dev(p.z, t), delta_bias=dev(p.bias),
                     delta_softplus=sp, h0=dev(p.h0), dh_final=dev(ghf),
                     discretization=disc, checkpoints=ck)
    torch.cuda.synchronize()
    rnd = lambda a: None if a is None else host(dev(a, t))          # noqa: E731
    ref = oracle.scan_bwd(rnd(gy), rnd(p.x), rnd(p.delta), p.A, rnd(p.B), rnd(p.C), Dv=p.D,
                          z=rnd(p.z), bias=p.bias, softplus=sp, h0=p.h0, gh_final=ghf, zoh=zoh)
    for mine, theirs in (("dx", "gx"), ("ddelta", "gdelta"), ("dA", "gA"), ("dB", "gB"),
                         ("dC", "gC"), ("dD", "gD"), ("ddelta_bias", "gbias"), ("dh0", "gh0"),
                         ("dz", "gz")):
        if theirs in ref and mine in g:
            assert_close(host(g[mine]), ref[theirs], io, f"{mine} (B {nb} L {L} D {D} N {N})")


@pytest.mark.parametrize("case", range(CASES))
def test_random_conv1d(case):
    rng = np.random.default_rng(900 + case)
    io = ("f32", "bf16")[case % 2]
    nb, L = int(rng.integers(1, 4)), int(rng.integers(1, 400))
    D = int(rng.choice([8, 16, 24, 40, 64, 100, 128, 200, 264]))
    K = int(rng.integers(1, 9))
    x = rng.standard_normal((nb, L, D))
    w = rng.standard_normal((D, K)) / np.sqrt(K)
    b = rng.standard_normal(D) * 0.1 if case % 3 else None
    xp = rng.standard_normal((nb, K - 1, D)) if (case % 4 == 1 and K > 1) else None
    t = io_dtype(io)
    out = ssm.conv1d(dev(x, t), dev(w), dev(b), x_prev=dev(xp, t), silu=bool(case % 5))
    torch.cuda.synchronize()
    rnd = lambda a: None if a is None else host(dev(a, t))          # noqa: E731
    ref = oracle.conv1d(rnd(x), w.astype(np.float32),
                        None if b is None else b.astype(np.float32), x_prev=rnd(xp),
                        silu=bool(case % 5))
    assert_close(host(out), ref, io, f"conv1d (B {nb} L {L} D {D} K {K})")


@pytest.mark.parametrize("case", range(CASES))
def test_random_ssd(case):
    rng = np.random.default_rng(1100 + case)
    io = ("f32", "bf16")[case % 2] if case % 4 else "bf16"
    nb, L = int(rng.integers(1, 3)), int(rng.integers(1, 400))
    G = int(rng.choice([1, 2]))
    H = G * int(rng.integers(1, 4))
    P = int(rng.choice([1, 3, 16, 64]))
    N = int(rng.choice([1, 5, 16, 64, 128]))
    if case % 4 == 0:
        P, N = 64, 128            # the tensor-core kernel's shape
    chunk = int(rng.choice([0, 32, 64, 128, 256]))
    gate, h0 = bool(case % 2), bool((case // 2) % 2)
    p = W.ssd_problem(nb, L, H, P, G, N, chunk=chunk, io=io, seed=1200 + case, gate=gate, h0=h0)
    iot = io_dtype(io)
    tc = ssm.ssd_uses_tensor_cores(dev(p.x, iot), dev(p.delta, iot), dev(p.A), dev(p.B, iot),
                                   dev(p.C, iot), z=dev(p.z, iot))
    ay, ah = ssd_tc_allowance(p) if tc else (None, None)
    y, hf = run_ssd(p)
    yr, hr = oracle.ssd(**p.oracle_args())
    assert_close(y, yr, io, f"ssd y (B {nb} L {L} H {H} P {P} G {G} N {N} chunk {chunk})",
                 allow=ay)
    assert_close(hf, hr, io, "ssd h_final", allow=ah)


@pytest.mark.parametrize("case", range(CASES))
def test_random_decode_steps(case):
    rng = np.random.default_rng(1300 + case)
    io = ("f32", "bf16")[case % 2]
    nb, D = int(rng.integers(1, 9)), int(rng.integers(1, 200))
    N = int(rng.choice([1, 4, 6, 8, 16, 32, 40, 64]))
    p = W.decode_problem(nb, D, N, 4, io=io, seed=1400 + case, gate=bool(case % 3))
    iot = io_dtype(io)
    state = dev(p.state0)
    ref = p.state0.astype(np.float64).copy()
    for s in range(4):
        tok = p.tokens(s)
        y = ssm.step_decode(state, dev(tok["x"], iot), dev(tok["delta"], iot), dev(p.A),
                            dev(tok["B"], iot), dev(tok["C"], iot), D=dev(p.D),
                            z=dev(tok["z"], iot), delta_bias=dev(p.bias))
        yr = oracle.decode_step(ref, tok["x"], tok["delta"], p.A, tok["B"], tok["C"], Dv=p.D,
                                z=tok["z"], bias=p.bias, softplus=True)
        torch.cuda.synchronize()
        assert_close(host(y), yr, io, f"decode y step {s} (B {nb} D {D} N {N})")
    assert_close(host(state), ref, io, "decode state")


@pytest.mark.parametrize("case", range(CASES))
def test_random_ssd_decode_steps(case):
    rng = np.random.default_rng(1500 + case)
    io = ("f32", "bf16")[case % 2]
    nb = int(rng.integers(1, 6))
    G = int(rng.choice([1, 2]))
    H = G * int(rng.integers(1, 5))
    P = int(rng.choice([1, 3, 16, 64]))
    N = int(rng.choice([5, 8, 16, 40, 64, 128, 200]))
    p = W.ssd_problem(nb, 3, H, P, G, N, io=io, seed=1600 + case, gate=bool(case % 3), h0=True)
    iot = io_dtype(io)
    state = dev(p.h0)
    ref = p.h0.astype(np.float64).copy()
    for s in range(3):
        y = ssm.ssd_step_decode(state, dev(p.x[:, s], iot), dev(p.delta[:, s], iot), dev(p.A),
                                dev(p.B[:, s], iot), dev(p.C[:, s], iot), D=dev(p.D),
                                z=None if p.z is None else dev(p.z[:, s], iot),
                                delta_bias=dev(p.bias))
        yr = oracle.ssd_decode_step(ref, p.x[:, s], p.delta[:, s], p.A, p.B[:, s], p.C[:, s],
                                    Dv=p.D, z=None if p.z is None else p.z[:, s], bias=p.bias)
        torch.cuda.synchronize()
        assert_close(host(y), yr, io, f"ssd decode y step {s} (B {nb} H {H} P {P} G {G} N {N})")
    assert_close(host(state), ref, io, "ssd decode state")
