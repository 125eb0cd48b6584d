"""GPU parity of ssm_ssd_step_decode (multi-head scalar-A decode step) against the fp64
oracle, with the state carried across calls."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_132_b300 as ssm
from selective_state_space_132_b300 import workloads as W

from _parity import assert_close, dev, host, io_dtype, run_ssd

pytestmark = pytest.mark.gpu


def _run(p, steps):
    """`steps` decode calls over the first tokens of an SSD problem, against the oracle;
    returns the GPU outputs (B, steps, H, P) and final state."""
    io = io_dtype(p.io)
    state = dev(p.h0) if p.h0 is not None else torch.zeros(
        (p.batch, p.heads, p.headdim, p.dstate), dtype=torch.float32, device="cuda")
    ref = (p.h0.astype(np.float64).copy() if p.h0 is not None
           else np.zeros((p.batch, p.heads, p.headdim, p.dstate)))
    ys, yrs = [], []
    A, Dv, bias = dev(p.A), dev(p.D), dev(p.bias)
    for t in range(steps):
        z = None if p.z is None else p.z[:, t]
        y = ssm.ssd_step_decode(state, dev(p.x[:, t], io), dev(p.delta[:, t], io), A,
                                dev(p.B[:, t], io), dev(p.C[:, t], io), D=Dv,
                                z=dev(z, io), delta_bias=bias)
        ys.append(host(y))
        yrs.append(oracle.ssd_decode_step(ref, p.x[:, t], p.delta[:, t], p.A, p.B[:, t],
                                          p.C[:, t], Dv=p.D, z=z, bias=p.bias))
    torch.cuda.synchronize()
    assert_close(np.stack(ys, 1), np.stack(yrs, 1), p.io, "y over all steps")
    assert_close(host(state), ref, p.io, "state")
    return np.stack(ys, 1), host(state)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("P,N,G,H,gate", [(64, 128, 1, 4, False), (16, 16, 2, 4, True),
                                          (8, 5, 1, 3, True), (32, 200, 2, 2, False),
                                          (64, 64, 4, 8, True)])
def test_ssd_decode_shapes(io, P, N, G, H, gate):
    p = W.ssd_problem(3, 9, H, P, G, N, io=io, seed=120 + P + N, gate=gate, h0=True)
    _run(p, 9)


def test_ssd_decode_equals_chunked_form():
    """L decode calls on the GPU equal one ssm_ssd_chunk_fwd (tensor-core kernel) over
    the same L tokens."""
    p = W.ssd_problem(2, 150, 4, 64, 1, 128, chunk=128, io="bf16", seed=130, h0=True)
    y_dec, h_dec = _run(p, p.seqlen)
    y_chk, h_chk = run_ssd(p, 128)
    assert oracle.rel_l2(y_dec, y_chk) < 3e-3 and oracle.rel_l2(h_dec, h_chk) < 3e-3


def test_ssd_decode_mamba2_batch64_shape():
    """Batch 64, 80 heads x 64, N 128, one group: three steps in place, checked in full."""
    p = W.ssd_problem(64, 3, 80, 64, 1, 128, io="bf16", seed=131, h0=True)
    _run(p, 3)
