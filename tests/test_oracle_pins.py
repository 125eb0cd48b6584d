"""Pins of the fp64 oracle to facts fixed by the pages and by mathematics.

None of these re-types the oracle's loop: each compares it with a different
route to the same number (a materialised matrix, a convolution, an FFT, a
closed form, an asymptotic, or an invariant), so that a dropped term, a wrong
sign or index or a transposed operand in the oracle fails at least one.
"""
import math

import numpy as np
import pytest

import oracle
from selective_state_space_132_b300 import workloads as W


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _small_scan(seed, nb=2, L=9, D=3, N=4, softplus=True, h0=False, gate=True, A="random"):
    p = W.scan_problem(nb, L, D, N, io="f32", seed=seed, gate=gate, h0=h0, softplus=softplus,
                       A=A)
    return p


# ---------------------------------------------------------------- softplus / silu facts
def test_softplus_identities():
    # softplus(0) = ln 2; softplus(v) - softplus(-v) = v; softplus(v) -> v, -> e^v
    assert oracle.softplus(0.0) == pytest.approx(math.log(2.0), rel=1e-15, abs=0)
    for v in (-30.0, -3.5, -0.25, 0.7, 4.0, 40.0):
        assert oracle.softplus(v) - oracle.softplus(-v) == pytest.approx(v, rel=1e-14, abs=1e-14)
    assert oracle.softplus(800.0) == 800.0           # no overflow
    assert oracle.softplus(-50.0) == pytest.approx(math.exp(-50.0), rel=1e-12)


def test_bias_recipe_inverts_softplus():
    # the delta-bias recipe draws u ~ U[1e-3, 1e-1] and stores inv_softplus(u)
    b = W._bias(_rng(3), 64)
    back = np.array([oracle.softplus(float(v)) for v in b])
    assert np.all(back >= 1e-3 * (1 - 1e-6)) and np.all(back <= 1e-1 * (1 + 1e-6))


# ---------------------------------------------------------------- semiseparable matrix
def _semiseparable_y(p, d, b):
    """y for channel d, batch b by materialising M_ts = C_t^T (prod_{r=s+1}^t Abar_r) B_s dl_s
    (Mamba-2 page, "1-세미분리 행렬") and the h0 term C_t^T (prod_{r=0}^t Abar_r) h0, with every
    product taken factor by factor."""
    L, N = p.seqlen, p.dstate
    raw = p.delta[b, :, d].astype(np.float64) + (p.bias[d] if p.bias is not None else 0.0)
    dl = np.array([oracle.softplus(v) for v in raw]) if p.softplus else raw
    Abar = np.exp(dl[:, None] * p.A[d][None, :].astype(np.float64))       # (L, N)
    Bm = p.B[b].astype(np.float64)
    Cm = p.C[b].astype(np.float64)
    x = p.x[b, :, d].astype(np.float64)
    M = np.zeros((L, L))
    for t in range(L):
        for s in range(t + 1):
            prod = np.ones(N)
            for r in range(s + 1, t + 1):
                prod = prod * Abar[r]
            M[t, s] = np.sum(Cm[t] * prod * Bm[s]) * dl[s]
    y = M @ x
    if p.h0 is not None:
        for t in range(L):
            prod = np.ones(N)
            for r in range(0, t + 1):
                prod = prod * Abar[r]
            y[t] += np.sum(Cm[t] * prod * p.h0[b, d].astype(np.float64))
    if p.D is not None:
        y = y + p.D[d] * x
    return y


@pytest.mark.parametrize("seed,softplus,h0", [(1, True, False), (2, False, True), (3, True, True)])
def test_scan_equals_semiseparable_matrix(seed, softplus, h0):
    p = _small_scan(seed, nb=2, L=11, D=3, N=5, softplus=softplus, h0=h0, gate=False)
    if not softplus:
        p.delta = np.abs(p.delta)  # keep the step positive without softplus
        p.bias = None
    y, _ = oracle.scan(**p.oracle_args())
    for b in range(p.batch):
        for d in range(p.dim):
            ref = _semiseparable_y(p, d, b)
            np.testing.assert_allclose(y[b, :, d], ref, rtol=1e-12, atol=1e-13)


def test_gate_multiplies_by_silu():
    p = _small_scan(4, gate=True)
    y_g, h_g = oracle.scan(**p.oracle_args())
    args = p.oracle_args()
    args["z"] = None
    y_u, h_u = oracle.scan(**args)
    ratio = y_g / y_u
    z = p.z.astype(np.float64)
    # silu(z) = z*sigmoid(z): silu(z) - silu(-z) = z, and ratio tends to z for large z
    expected = z / (1.0 + np.exp(-z))
    np.testing.assert_allclose(ratio, expected, rtol=1e-11)
    np.testing.assert_array_equal(h_g, h_u)  # the gate never touches the state


# ---------------------------------------------------------------- LTI convolution kernel
def test_lti_case_is_causal_convolution():
    """Constant dl, B, C over time: y = Kbar * x with Kbar_k = sum_n C_n Abar_n^k dl B_n
    (tildalice review, "SSM의 이중 연산 모드"), checked with numpy.convolve and numpy.fft."""
    rng = _rng(11)
    L, D, N = 64, 2, 6
    x = rng.standard_normal((1, L, D))
    dl = np.array([0.07, 0.31])
    delta = np.broadcast_to(dl, (1, L, D)).copy()
    A = -rng.uniform(0.5, 4.0, size=(D, N))
    Bc = rng.standard_normal(N)
    Cc = rng.standard_normal(N)
    Bm = np.broadcast_to(Bc, (1, L, N)).copy()
    Cm = np.broadcast_to(Cc, (1, L, N)).copy()
    Dv = rng.standard_normal(D)
    y, _ = oracle.scan(x, delta, A, Bm, Cm, Dv=Dv, softplus=False)
    for d in range(D):
        k = np.arange(L)
        Abar = np.exp(dl[d] * A[d])
        K = np.array([np.sum(Cc * Abar ** kk * dl[d] * Bc) for kk in k])
        direct = np.convolve(x[0, :, d], K)[:L] + Dv[d] * x[0, :, d]
        nfft = 2 * L
        viafft = np.fft.irfft(np.fft.rfft(x[0, :, d], nfft) * np.fft.rfft(K, nfft), nfft)[:L]
        viafft = viafft + Dv[d] * x[0, :, d]
        np.testing.assert_allclose(y[0, :, d], direct, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(y[0, :, d], viafft, rtol=1e-9, atol=1e-11)


def test_lssl_window_three_kernel():
    """Window-3 example of the LSSL convolution ("Convolution for LTI-SSM" in the
    yongggg review): y_3 = K_3 . [x_3, x_2, x_1] with K_3 = [C Abar^2 Bbar, C Abar Bbar, C Bbar]."""
    rng = _rng(12)
    N = 3
    A = -rng.uniform(0.5, 2.0, size=(1, N))
    dl = 0.2
    Bc, Cc = rng.standard_normal(N), rng.standard_normal(N)
    x = rng.standard_normal((1, 3, 1))
    y, _ = oracle.scan(x, np.full((1, 3, 1), dl), A, np.tile(Bc, (1, 3, 1)),
                       np.tile(Cc, (1, 3, 1)), softplus=False)
    Abar, Bbar = np.exp(dl * A[0]), dl * Bc
    K3 = np.array([np.sum(Cc * Abar ** 2 * Bbar), np.sum(Cc * Abar * Bbar), np.sum(Cc * Bbar)])
    assert y[0, 2, 0] == pytest.approx(float(K3 @ x[0, :, 0]), rel=1e-13)


# ---------------------------------------------------------------- limits and closed forms
def test_zero_step_keeps_state_and_passes_skip():
    """dl = 0 exactly: Abar = I and Bbar = 0, so h stays h0 and y = (C.h0 + D x) silu(z)."""
    p = _small_scan(5, h0=True, gate=True)
    p.delta[:] = 0.0
    p.bias = None
    p.softplus = False
    y, hf = oracle.scan(**p.oracle_args())
    np.testing.assert_array_equal(hf, p.h0.astype(np.float64))
    z = p.z.astype(np.float64)
    ch0 = np.einsum("bln,bdn->bld", p.C.astype(np.float64), p.h0.astype(np.float64))
    Dx = p.D.astype(np.float64)[None, None, :] * p.x.astype(np.float64)
    expected = (ch0 + Dx) * (z / (1 + np.exp(-z)))
    np.testing.assert_allclose(y, expected, rtol=1e-12, atol=1e-14)
    # and with h0 = 0 the output is only the skip term
    args = p.oracle_args()
    args["h0"] = None
    y0, hf0 = oracle.scan(**args)
    np.testing.assert_allclose(y0, Dx * (z / (1 + np.exp(-z))),
                               rtol=1e-12, atol=1e-14)
    assert not np.any(hf0)


def test_large_step_forgets():
    """dl -> infinity with A < 0: Abar -> 0, so h_t = dl B_t x_t and
    y_t = dl (C_t . B_t) x_t + D x_t (tildalice review, "Δ의 직관적 이해")."""
    p = _small_scan(6, h0=True, gate=False, A="random")
    p.delta[:] = 60.0  # softplus(60 + bias) ~ 60 + bias, exp(-30) negligible at rtol 1e-9
    y, hf = oracle.scan(**p.oracle_args())
    dl = np.array([oracle.softplus(60.0 + float(b)) for b in p.bias])
    cb = np.einsum("bln,bln->bl", p.C.astype(np.float64), p.B.astype(np.float64))
    x = p.x.astype(np.float64)
    expected = dl[None, None, :] * cb[:, :, None] * x + p.D.astype(np.float64)[None, None, :] * x
    np.testing.assert_allclose(y, expected, rtol=1e-9, atol=1e-12)
    expected_h = dl[None, :, None] * p.B[:, -1, None, :].astype(np.float64) * x[:, -1, :, None]
    np.testing.assert_allclose(hf, expected_h, rtol=1e-9)


def test_constant_input_geometric_series():
    """Constant x, dl, B, C and h0 = 0: h_t = dl B x (1 - a^{t+1}) / (1 - a), a = exp(dl A)."""
    L, N = 40, 5
    A = -np.array([[0.3, 1.0, 2.0, 5.0, 9.0]])
    dl, xv = 0.05, 1.7
    Bc = np.array([0.5, -1.0, 2.0, 0.25, -0.75])
    Cc = np.array([1.0, 0.5, -0.5, 2.0, 1.5])
    Dv = np.array([0.3])
    y, hf = oracle.scan(np.full((1, L, 1), xv), np.full((1, L, 1), dl), A,
                        np.tile(Bc, (1, L, 1)), np.tile(Cc, (1, L, 1)), Dv=Dv, softplus=False)
    a = np.exp(dl * A[0])
    t = np.arange(L)[:, None]
    h = dl * Bc * xv * (1 - a ** (t + 1)) / (1 - a)
    np.testing.assert_allclose(y[0, :, 0], h @ Cc + Dv[0] * xv, rtol=1e-12)
    np.testing.assert_allclose(hf[0, 0], h[-1], rtol=1e-12)


def test_free_decay_of_initial_state():
    """x = 0: h_t,n = exp(A_n * sum_{r<=t} dl_r) h0_n, a sum instead of a product."""
    p = _small_scan(7, h0=True, gate=False, L=25)
    p.x[:] = 0.0
    y, hf = oracle.scan(**p.oracle_args())
    raw = p.delta.astype(np.float64) + p.bias[None, None, :]
    dl = np.vectorize(oracle.softplus)(raw)
    S = np.cumsum(dl, axis=1)                                   # (B, L, D)
    h = np.exp(S[..., None] * p.A[None, None].astype(np.float64)) * p.h0[:, None]
    np.testing.assert_allclose(hf, h[:, -1], rtol=1e-12)
    np.testing.assert_allclose(y, np.einsum("bln,bldn->bld", p.C.astype(np.float64), h),
                               rtol=1e-10, atol=1e-14)


# ---------------------------------------------------------------- invariants
def test_causality_bit_exact():
    p = _small_scan(8, L=20)
    y1, _ = oracle.scan(**p.oracle_args())
    p.x[:, 13, :] += 1.0
    y2, _ = oracle.scan(**p.oracle_args())
    np.testing.assert_array_equal(y1[:, :13], y2[:, :13])
    assert np.all(y1[:, 13] != y2[:, 13])


def test_linearity_in_input_and_initial_state():
    p = _small_scan(9, h0=True)
    q = _small_scan(10, h0=True)
    args_p, args_q = p.oracle_args(), p.oracle_args()
    args_q["x"], args_q["h0"] = q.x, q.h0
    yp, hp = oracle.scan(**args_p)
    yq, hq = oracle.scan(**args_q)
    args_c = p.oracle_args()
    args_c["x"] = 2.0 * p.x.astype(np.float64) - 0.5 * q.x
    args_c["h0"] = 2.0 * p.h0.astype(np.float64) - 0.5 * q.h0
    yc, hc = oracle.scan(**args_c)
    np.testing.assert_allclose(yc, 2.0 * yp - 0.5 * yq, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(hc, 2.0 * hp - 0.5 * hq, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("cut", [1, 17, 38])
def test_split_sequence_state_passing(cut):
    p = _small_scan(13, L=39, h0=True)
    y, hf = oracle.scan(**p.oracle_args())
    a1 = p.oracle_args()
    for k in ("x", "delta", "z"):
        a1[k] = getattr(p, k)[:, :cut]
    for k, src in (("Bm", p.B), ("Cm", p.C)):
        a1[k] = src[:, :cut]
    y1, h1 = oracle.scan(**a1)
    a2 = p.oracle_args()
    for k in ("x", "delta", "z"):
        a2[k] = getattr(p, k)[:, cut:]
    for k, src in (("Bm", p.B), ("Cm", p.C)):
        a2[k] = src[:, cut:]
    a2["h0"] = h1
    y2, h2 = oracle.scan(**a2)
    np.testing.assert_allclose(np.concatenate([y1, y2], axis=1), y, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(h2, hf, rtol=1e-13, atol=1e-15)


def test_decode_steps_equal_scan():
    p = _small_scan(14, L=17, h0=True)
    y, hf = oracle.scan(**p.oracle_args())
    state = p.h0.astype(np.float64).copy()
    for t in range(p.seqlen):
        yt = oracle.decode_step(state, p.x[:, t], p.delta[:, t], p.A, p.B[:, t], p.C[:, t],
                                Dv=p.D, z=p.z[:, t], bias=p.bias, softplus=True)
        np.testing.assert_array_equal(yt, y[:, t])
    np.testing.assert_array_equal(state, hf)


def test_channels_and_batches_independent():
    p = _small_scan(15, nb=3, D=5)
    y, hf = oracle.scan(**p.oracle_args())
    perm = np.array([3, 0, 4, 1, 2])
    args = p.oracle_args()
    for k in ("x", "delta", "z"):
        args[k] = getattr(p, k)[:, :, perm]
    args["A"] = p.A[perm]
    args["Dv"], args["bias"] = p.D[perm], p.bias[perm]
    yp, hp = oracle.scan(**args)
    np.testing.assert_array_equal(yp, y[:, :, perm])
    np.testing.assert_array_equal(hp, hf[:, perm])


# ---------------------------------------------------------------- SSD (multi-head scalar A)
def _ssd_small(seed, nb=2, L=23, H=4, P=3, G=2, N=5, gate=True, h0=True):
    return W.ssd_problem(nb, L, H, P, G, N, chunk=8, io="f32", seed=seed, gate=gate, h0=h0)


def test_ssd_equals_scan_with_broadcast_decay():
    """Each SSD head is an S6 scan over its P channels with A[d, n] = A_h and the
    head's step shared by its channels (Mamba-2 page, "멀티-헤드 구조")."""
    p = _ssd_small(21)
    y, hf = oracle.ssd(**p.oracle_args())
    hpg = p.heads // p.ngroups
    for h in range(p.heads):
        g = h // hpg
        x = p.x[:, :, h, :]
        delta = np.repeat(p.delta[:, :, h:h + 1], p.headdim, axis=2)
        A = np.full((p.headdim, p.dstate), p.A[h])
        ys, hs = oracle.scan(x, delta, A, p.B[:, :, g], p.C[:, :, g],
                             Dv=np.full(p.headdim, p.D[h]), z=p.z[:, :, h, :],
                             bias=np.full(p.headdim, p.bias[h]), softplus=True,
                             h0=p.h0[:, h])
        np.testing.assert_allclose(y[:, :, h, :], ys, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(hf[:, h], hs, rtol=1e-13, atol=1e-15)


def _chunked_dual(p, Q):
    """SSD by chunks (Mamba-2 page, "SSD 타일링 알고리즘" and "SSM-Attention 동치성"):
    inside a chunk Y = (L o C B^T) (dl x) with L_ts = exp(Acum_t - Acum_s) [s <= t];
    between chunks the state is passed as S <- exp(Acum_end) S + sum_s
    exp(Acum_end - Acum_s) dl_s x_s B_s^T, and read by Y += exp(Acum_t) C_t S^T."""
    nb, L, H, P = p.x.shape
    G, N = p.ngroups, p.dstate
    hpg = H // G
    raw = p.delta.astype(np.float64) + p.bias[None, None, :]
    dl = np.vectorize(oracle.softplus)(raw)                    # (B, L, H)
    y = np.zeros((nb, L, H, P))
    hf = np.zeros((nb, H, P, N))
    for b in range(nb):
        for h in range(H):
            g = h // hpg
            S = p.h0[b, h].astype(np.float64).copy() if p.h0 is not None else np.zeros((P, N))
            for c0 in range(0, L, Q):
                c1 = min(L, c0 + Q)
                a = dl[b, c0:c1, h] * p.A[h]
                Acum = np.cumsum(a)
                Cc = p.C[b, c0:c1, g].astype(np.float64)
                Bc = p.B[b, c0:c1, g].astype(np.float64)
                X = p.x[b, c0:c1, h].astype(np.float64)
                seg = Acum[:, None] - Acum[None, :]
                Lmask = np.where(np.tril(np.ones_like(seg)) > 0, np.exp(np.minimum(seg, 0)), 0.0)
                Yd = (Lmask * (Cc @ Bc.T)) @ (dl[b, c0:c1, h][:, None] * X)
                Yo = np.exp(Acum)[:, None] * (Cc @ S.T)
                yc = Yd + Yo + p.D[h] * X
                if p.z is not None:
                    zc = p.z[b, c0:c1, h].astype(np.float64)
                    yc = yc * (zc / (1 + np.exp(-zc)))
                y[b, c0:c1, h] = yc
                w = np.exp(Acum[-1] - Acum) * dl[b, c0:c1, h]
                S = np.exp(Acum[-1]) * S + (w[:, None] * X).T @ Bc
            hf[b, h] = S
    return y, hf


@pytest.mark.parametrize("Q", [1, 4, 8, 23, 64])
def test_ssd_equals_chunked_dual_form(Q):
    p = _ssd_small(22)
    y, hf = oracle.ssd(**p.oracle_args())
    yc, hc = _chunked_dual(p, Q)
    np.testing.assert_allclose(y, yc, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(hf, hc, rtol=1e-10, atol=1e-12)


def test_oracle_runs_threaded_identically():
    p = _small_scan(30, nb=3, D=7, L=33)
    y1, h1 = oracle.scan(**p.oracle_args(), threads=1)
    y4, h4 = oracle.scan(**p.oracle_args(), threads=4)
    np.testing.assert_array_equal(y1, y4)
    np.testing.assert_array_equal(h1, h4)


# ---------------------------------------------------------------- multi-head decode step
def test_ssd_decode_steps_equal_ssd_scan():
    """L single-token steps of the multi-head recurrence equal the (pinned) SSD oracle
    over the same L tokens, outputs and final state, with groups and a gate."""
    p = _ssd_small(11, nb=2, L=13, H=4, P=3, G=2, N=5, gate=True, h0=True)
    y_ref, h_ref = oracle.ssd(**p.oracle_args())
    state = p.h0.astype(np.float64).copy()
    ys = []
    for t in range(p.seqlen):
        ys.append(oracle.ssd_decode_step(state, p.x[:, t], p.delta[:, t], p.A, p.B[:, t],
                                         p.C[:, t], Dv=p.D, z=p.z[:, t], bias=p.bias,
                                         softplus=p.softplus))
    np.testing.assert_allclose(np.stack(ys, axis=1), y_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(state, h_ref, rtol=1e-12, atol=1e-12)


def test_ssd_decode_zero_step_keeps_state():
    """dl = 0 exactly (raw 0, no bias, no softplus): the state is unchanged and
    y = S C + D x (no gate)."""
    rng = _rng(12)
    nb, H, P, G, N = 2, 4, 3, 2, 5
    state = rng.standard_normal((nb, H, P, N))
    s0 = state.copy()
    x = rng.standard_normal((nb, H, P))
    Bm = rng.standard_normal((nb, G, N))
    Cm = rng.standard_normal((nb, G, N))
    A = -rng.uniform(1, 16, H)
    Dv = rng.standard_normal(H)
    y = oracle.ssd_decode_step(state, x, np.zeros((nb, H)), A, Bm, Cm, Dv=Dv, softplus=False)
    np.testing.assert_array_equal(state, s0)
    g = np.arange(H) // (H // G)
    expect = np.einsum("bhpn,bhn->bhp", s0, Cm[:, g]) + Dv[None, :, None] * x
    np.testing.assert_allclose(y, expect, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- zero-order hold
def _rk4_continuous(p, d, b, substeps=400):
    """Integrate the continuous SSM h' = A h + B x (tildalice "연속 시간 SSM") through each
    step's interval of length dl_t with x, B held constant (the hold that the zero-order
    discretisation assumes), classic RK4, and read y_t = C_t h + D x_t at the end."""
    raw = p.delta[b, :, d].astype(np.float64) + (p.bias[d] if p.bias is not None else 0.0)
    dl = np.array([oracle.softplus(v) for v in raw]) if p.softplus else raw
    A = p.A[d].astype(np.float64)
    h = np.zeros(p.dstate) if p.h0 is None else p.h0[b, d].astype(np.float64).copy()
    ys = []
    for t in range(p.seqlen):
        u = p.B[b, t].astype(np.float64) * float(p.x[b, t, d])
        f = lambda hh: A * hh + u
        k = dl[t] / substeps
        for _ in range(substeps):
            k1 = f(h); k2 = f(h + 0.5 * k * k1); k3 = f(h + 0.5 * k * k2); k4 = f(h + k * k3)
            h = h + k / 6.0 * (k1 + 2 * k2 + 2 * k3 + k4)
        ys.append(float(np.dot(p.C[b, t].astype(np.float64), h)) +
                  (float(p.D[d]) if p.D is not None else 0.0) * float(p.x[b, t, d]))
    return np.array(ys), h


def test_zoh_scan_equals_integrated_ode():
    p = W.scan_problem(1, 12, 2, 4, io="f32", seed=31, gate=False, h0=True, A="random")
    p.zoh = True
    y, hf = oracle.scan(**p.oracle_args())
    for d in range(p.dim):
        y_ode, h_ode = _rk4_continuous(p, d, 0)
        np.testing.assert_allclose(y[0, :, d], y_ode, rtol=1e-9, atol=1e-9)
        np.testing.assert_allclose(hf[0, d], h_ode, rtol=1e-9, atol=1e-9)


def test_zoh_limits():
    # A = 0: the hold coefficient (e^{dl a} - 1) / a tends to dl, so ZOH equals Euler
    p = W.scan_problem(2, 9, 3, 4, io="f32", seed=32, h0=True)
    p.A = np.zeros_like(p.A)
    ye, he = oracle.scan(**p.oracle_args())
    p.zoh = True
    yz, hz = oracle.scan(**p.oracle_args())
    np.testing.assert_array_equal(yz, ye)
    np.testing.assert_array_equal(hz, he)
    # small steps: ZOH - Euler shrinks like dl^2 (B̄ differs by dl^2 a / 2 + ...)
    diffs = []
    for eps in (1e-2, 1e-3):
        q = W.scan_problem(2, 9, 3, 4, io="f32", seed=33, softplus=False, use_bias=False,
                           gate=False, A="random")
        q.delta = np.abs(q.delta) * np.float32(eps)
        ye, _ = oracle.scan(**q.oracle_args())
        q.zoh = True
        yz, _ = oracle.scan(**q.oracle_args())
        diffs.append(np.abs(yz - ye).max() / np.abs(ye).max())
    assert diffs[1] < diffs[0] * 0.02   # one decade of dl -> about two decades of error


# ---------------------------------------------------------------- causal conv1d + SiLU
def test_conv1d_equals_numpy_convolution():
    """The causal depthwise convolution equals numpy.convolve per channel (a textbook
    routine; the kernel reversed, since the layer correlates), then SiLU."""
    rng = _rng(21)
    nb, L, D, K = 2, 17, 5, 4
    x = rng.standard_normal((nb, L, D))
    w = rng.standard_normal((D, K))
    bias = rng.standard_normal(D)
    out = oracle.conv1d(x, w, bias)
    for b in range(nb):
        for d in range(D):
            pre = np.convolve(x[b, :, d], w[d, ::-1])[:L] + bias[d]
            np.testing.assert_allclose(out[b, :, d], pre / (1 + np.exp(-pre)), rtol=1e-13,
                                       atol=1e-13)


def test_conv1d_impulse_and_carried_window():
    rng = _rng(22)
    D, K = 3, 4
    w = rng.standard_normal((D, K))
    # a unit impulse at t = 2 reads the kernel back, last tap first (no bias, no SiLU)
    x = np.zeros((1, 9, D))
    x[0, 2, :] = 1.0
    out = oracle.conv1d(x, w, silu=False)
    for k in range(K):
        np.testing.assert_allclose(out[0, 2 + k], w[:, K - 1 - k], rtol=0, atol=0)
    # splitting a sequence and carrying the last K-1 inputs equals one call
    x = rng.standard_normal((2, 20, D))
    full = oracle.conv1d(x, w, silu=True)
    first = oracle.conv1d(x[:, :11], w, silu=True)
    second = oracle.conv1d(x[:, 11:], w, x_prev=x[:, 11 - (K - 1):11], silu=True)
    np.testing.assert_allclose(np.concatenate([first, second], 1), full, rtol=1e-14, atol=1e-14)


# ---------------------------------------------------------------- backward (adjoint) pins
_GRAD_INPUTS = ("x", "delta", "A", "B", "C", "D", "z", "bias", "h0")


def _bwd_problem(seed, zoh, nb=2, L=7, D=3, N=4):
    rng = _rng(seed)
    p = dict(x=rng.standard_normal((nb, L, D)), delta=0.5 * rng.standard_normal((nb, L, D)),
             A=-rng.uniform(0.5, 4.0, (D, N)), B=rng.standard_normal((nb, L, N)),
             C=rng.standard_normal((nb, L, N)), D=rng.standard_normal(D),
             z=rng.standard_normal((nb, L, D)), bias=rng.uniform(-1.0, 0.5, D),
             h0=rng.standard_normal((nb, D, N)))
    if zoh:
        p["A"][0, 1] = 0.0              # the A -> 0 limit of the zero-order hold
        p["A"][1, 2] = -1e-4            # and its neighbourhood (series branch)
    gy = rng.standard_normal((nb, L, D))
    ghf = rng.standard_normal((nb, D, N))
    return p, gy, ghf


def _loss(p, gy, ghf, zoh):
    y, hf = oracle.scan(p["x"], p["delta"], p["A"], p["B"], p["C"], Dv=p["D"], z=p["z"],
                        bias=p["bias"], softplus=True, h0=p["h0"], zoh=zoh, threads=1)
    return float(np.sum(gy * y) + np.sum(ghf * hf))


def _bwd(p, gy, ghf, zoh):
    g = oracle.scan_bwd(gy, p["x"], p["delta"], p["A"], p["B"], p["C"], Dv=p["D"], z=p["z"],
                        bias=p["bias"], softplus=True, h0=p["h0"], gh_final=ghf, zoh=zoh)
    return dict(x=g["gx"], delta=g["gdelta"], A=g["gA"], B=g["gB"], C=g["gC"], D=g["gD"],
                z=g["gz"], bias=g["gbias"], h0=g["gh0"])


@pytest.mark.parametrize("zoh", [False, True])
def test_backward_equals_central_differences(zoh):
    """Every gradient the adjoint returns equals the central difference of the forward
    oracle's scalar loss <gy, y> + <gh_final, h_final>, element by element."""
    p, gy, ghf = _bwd_problem(61 + zoh, zoh)
    g = _bwd(p, gy, ghf, zoh)
    eps = 1e-6
    for name in _GRAD_INPUTS:
        a = p[name]
        fd = np.empty_like(a)
        for i in np.ndindex(a.shape):
            keep = a[i]
            a[i] = keep + eps
            up = _loss(p, gy, ghf, zoh)
            a[i] = keep - eps
            dn = _loss(p, gy, ghf, zoh)
            a[i] = keep
            fd[i] = (up - dn) / (2 * eps)
        scale = max(1.0, float(np.max(np.abs(fd))))
        assert np.max(np.abs(g[name] - fd)) < 2e-7 * scale, name


def _torch_scan_loss(t, gy, ghf, zoh):
    """A plain PyTorch fp64 restatement of the forward recurrence (own loop, no oracle
    code), differentiated by autograd."""
    import torch
    x, dr, A, Bm, Cm, Dv, z, bias, h0 = (t[k] for k in _GRAD_INPUTS)
    dl = torch.nn.functional.softplus(dr + bias)                       # (B,L,D)
    h = h0
    loss = 0.0
    for s in range(x.shape[1]):
        e = dl[:, s, :, None] * A[None]                                # (B,D,N)
        if zoh:
            # coef = dl * phi(e), phi(e) = (e^e - 1)/e, smooth through e = 0 (Taylor
            # polynomial there) so that autograd sees the derivative at A = 0 too
            small = e.abs() < 1e-3
            e_safe = torch.where(small, torch.ones_like(e), e)
            phi = torch.where(small, 1 + e / 2 + e * e / 6 + e * e * e / 24,
                              torch.expm1(e_safe) / e_safe)
            coef = dl[:, s, :, None] * phi
        else:
            coef = dl[:, s, :, None]
        h = torch.exp(e) * h + coef * Bm[:, s, None, :] * x[:, s, :, None]
        yr = (h * Cm[:, s, None, :]).sum(-1) + Dv * x[:, s]
        y = yr * torch.nn.functional.silu(z[:, s])
        loss = loss + (y * gy[:, s]).sum()
    return loss + (h * ghf).sum()


@pytest.mark.parametrize("zoh", [False, True])
def test_backward_equals_autograd_of_an_independent_loop(zoh):
    import torch
    p, gy, ghf = _bwd_problem(71 + zoh, zoh, nb=3, L=40, D=6, N=8)
    t = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in p.items()}
    _torch_scan_loss(t, torch.tensor(gy), torch.tensor(ghf), zoh).backward()
    g = _bwd(p, gy, ghf, zoh)
    for name in _GRAD_INPUTS:
        ref = t[name].grad.numpy()
        assert oracle.rel_l2(g[name], ref) < 1e-12, name


def test_backward_without_optional_inputs():
    """No gate, no D, no bias, no h0, no softplus, no final-state gradient: gx then
    equals the transposed semiseparable matrix applied to gy."""
    rng = _rng(81)
    nb, L, D, N = 1, 12, 2, 3
    x = rng.standard_normal((nb, L, D))
    dl = rng.uniform(0.05, 0.6, (nb, L, D))
    A = -rng.uniform(0.5, 3.0, (D, N))
    Bm, Cm = rng.standard_normal((nb, L, N)), rng.standard_normal((nb, L, N))
    gy = rng.standard_normal((nb, L, D))
    g = oracle.scan_bwd(gy, x, dl, A, Bm, Cm, softplus=False)
    for d in range(D):
        M = np.zeros((L, L))
        for t_ in range(L):
            for s in range(t_ + 1):
                decay = np.exp(A[d] * dl[0, s + 1:t_ + 1, d].sum())
                M[t_, s] = np.sum(Cm[0, t_] * decay * Bm[0, s]) * dl[0, s, d]
        np.testing.assert_allclose(g["gx"][0, :, d], M.T @ gy[0, :, d], rtol=1e-12, atol=1e-12)
    # gradients of the absent D and bias (taken at zero): sum gy x and sum gdelta
    np.testing.assert_allclose(g["gD"], (gy * x).sum(axis=(0, 1)), rtol=1e-12)
    np.testing.assert_allclose(g["gbias"], g["gdelta"].sum(axis=(0, 1)), rtol=1e-12)
    # with no final-state gradient, gh0 = sum_t (prod_{r<=t} Abar_r) C_t gy_t
    for d in range(D):
        acc = np.zeros(N)
        for t_ in range(L):
            acc += np.exp(A[d] * dl[0, :t_ + 1, d].sum()) * Cm[0, t_] * gy[0, t_, d]
        np.testing.assert_allclose(g["gh0"][0, d], acc, rtol=1e-12)
