"""GPU parity of ssm_ssd_chunk_fwd (Mamba-2 SSD form) against the fp64 oracle."""
import numpy as np
import pytest

import oracle
from selective_state_space_132_b300 import workloads as W

import selective_state_space_132_b300 as ssm

from _parity import Parity, assert_close, dev, io_dtype, run_scan, run_ssd, ssd_tc_allowance

pytestmark = pytest.mark.gpu


def _check(p, chunk=None):
    """y is compared with the (b, h, p) channels as rows (each over time), so a wrong
    chunk hand-over in one chain shows in its rows; h_final by (b, h, p).  The
    tensor-core kernel gets the allowance of its bf16 operands."""
    ay, ah = ssd_tc_allowance(p) if _uses_tc(p) else (None, None)
    y, hf = run_ssd(p, chunk)
    yr, hr = oracle.ssd(**p.oracle_args())
    assert np.all(np.isfinite(y))
    assert_close(y, yr, p.io, "y", row_axes=(0, 2, 3), allow=ay)
    assert_close(hf, hr, p.io, "h_final", allow=ah)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("P,N,G,H", [(64, 128, 1, 4), (64, 64, 2, 4), (16, 16, 1, 3),
                                     (32, 128, 4, 8), (8, 5, 1, 2)])
def test_shapes(io, P, N, G, H):
    p = W.ssd_problem(2, 300, H, P, G, N, chunk=64, io=io, seed=60 + P + N, h0=True)
    _check(p)


def _uses_tc(p):
    io = io_dtype(p.io)
    return ssm.ssd_uses_tensor_cores(dev(p.x, io), dev(p.delta, io), dev(p.A), dev(p.B, io),
                                     dev(p.C, io), z=dev(p.z, io))


@pytest.mark.parametrize("L,nb,H,G,gate,h0", [(1, 1, 2, 1, False, False),
                                              (77, 2, 3, 1, True, True),
                                              (128, 1, 2, 2, False, True),
                                              (129, 3, 4, 2, False, False),
                                              (700, 2, 6, 3, True, True)])
def test_tensor_core_path(L, nb, H, G, gate, h0):
    """The tcgen05 chunked kernel (bf16, P = 64, N = 128): short, exact-tile, ragged and
    multi-tile sequences, several batches and groups, with and without gate and h0."""
    p = W.ssd_problem(nb, L, H, 64, G, 128, chunk=128, io="bf16", seed=80 + L + H, gate=gate,
                      h0=h0)
    assert _uses_tc(p)
    _check(p)


def test_tensor_core_chains_split_between_blocks():
    """More (batch, head) chains than resident blocks: the persistent grid cuts chains
    between blocks and hands the state over through the workspace."""
    p = W.ssd_problem(1, 300, 320, 64, 1, 128, chunk=128, io="bf16", seed=91, h0=True)
    assert _uses_tc(p)
    _check(p)


def test_tensor_core_path_is_not_taken_for_other_shapes():
    assert not _uses_tc(W.ssd_problem(1, 64, 2, 32, 1, 128, io="bf16", seed=1))
    assert not _uses_tc(W.ssd_problem(1, 64, 2, 64, 1, 64, io="bf16", seed=1))
    assert not _uses_tc(W.ssd_problem(1, 64, 2, 64, 1, 128, io="f32", seed=1))


@pytest.mark.parametrize("chunk", [32, 64, 128, 256])
def test_chunk_sizes(chunk):
    p = W.ssd_problem(1, 520, 4, 64, 1, 128, chunk=chunk, io="bf16", seed=70, gate=True)
    _check(p, chunk)


def test_gate_and_no_skip():
    p = W.ssd_problem(2, 257, 4, 64, 1, 64, chunk=256, io="bf16", seed=71, gate=True,
                      use_D=False, h0=True)
    _check(p)


def test_ssd_equals_scan_with_head_broadcast():
    """An SSD head is an S6 scan over its P channels with a shared decay: run both on
    the GPU and compare."""
    p = W.ssd_problem(1, 200, 2, 16, 1, 16, chunk=64, io="f32", seed=72)
    y, _ = run_ssd(p)
    for h in range(p.heads):
        s = W.scan_problem(1, 200, 16, 16, io="f32", seed=0, gate=False)
        s.x = np.ascontiguousarray(p.x[:, :, h, :])
        s.delta = np.ascontiguousarray(np.repeat(p.delta[:, :, h:h + 1], 16, axis=2))
        s.A = np.full((16, 16), p.A[h], np.float32)
        s.B, s.C = np.ascontiguousarray(p.B[:, :, 0]), np.ascontiguousarray(p.C[:, :, 0])
        s.D = np.full(16, p.D[h], np.float32)
        s.bias = np.full(16, p.bias[h], np.float32)
        ys, _ = run_scan(s)
        assert oracle.rel_l2(y[:, :, h, :], ys) < 2e-6


@pytest.mark.slow
def test_mamba2_full_size():
    """Reference workload: batch 4, L 8192, 80 heads x 64, N 128, one group, chunk 256,
    bf16, run in full on the GPU and compared with the oracle on every output and every
    final state, one batch row at a time (each an independent oracle call)."""
    p = W.config_problem(3)
    assert _uses_tc(p)
    y, hf = run_ssd(p)
    H, P = p.heads, p.headdim
    py = Parity("bf16", "y (Mamba-2 SSD)", p.batch * H * P)
    ph = Parity("bf16", "h_final (Mamba-2 SSD)", p.batch * H * P)
    for b in range(p.batch):
        args = p.oracle_args()
        args["x"], args["delta"] = p.x[b:b + 1], p.delta[b:b + 1]
        args["Bm"], args["Cm"] = p.B[b:b + 1], p.C[b:b + 1]
        yr, hr = oracle.ssd(**args)
        ay, ah = ssd_tc_allowance(p, batch=b)
        rows = slice(b * H * P, (b + 1) * H * P)
        # rows (b, h, p) over time
        py.add(y[b].reshape(p.seqlen, H * P).T, yr[0].reshape(p.seqlen, H * P).T, rows=rows,
               allow=ay[0].reshape(p.seqlen, H * P).T)
        ph.add(hf[b].reshape(H * P, -1), hr[0].reshape(H * P, -1), rows=rows,
               allow=ah[0].reshape(H * P, -1))
        del yr, hr, ay, ah
    py.check()
    ph.check()
