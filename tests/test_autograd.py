"""selective_scan: torch autograd through the library's forward and backward kernels,
against the fp64 oracle's adjoint."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_132_b300 as ssm
from selective_state_space_132_b300 import workloads as W

from _parity import assert_close, dev, host, io_dtype

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("zoh", [False, True])
def test_autograd_matches_oracle_adjoint(io, zoh):
    p = W.scan_problem(2, 70, 40, 16, io=io, seed=60, h0=True)
    t = io_dtype(io)
    leaves = {k: dev(v, t if k in ("x", "delta", "B", "C", "z") else torch.float32).requires_grad_()
              for k, v in (("x", p.x), ("delta", p.delta), ("A", p.A), ("B", p.B), ("C", p.C),
                           ("D", p.D), ("z", p.z), ("bias", p.bias), ("h0", p.h0))}
    y, hf = ssm.selective_scan(leaves["x"], leaves["delta"], leaves["A"], leaves["B"],
                               leaves["C"], D=leaves["D"], z=leaves["z"],
                               delta_bias=leaves["bias"], h0=leaves["h0"],
                               discretization="zoh" if zoh else "euler")
    rng = np.random.default_rng(61)
    gy = dev(rng.standard_normal(y.shape), t)
    ghf = dev(rng.standard_normal(hf.shape))
    ((y.float() * gy.float()).sum() + (hf * ghf).sum()).backward()
    ref = oracle.scan_bwd(host(gy), p.x, p.delta, p.A, p.B, p.C, Dv=p.D, z=p.z, bias=p.bias,
                          h0=p.h0, gh_final=host(ghf), zoh=zoh)
    for leaf, theirs in (("x", "gx"), ("delta", "gdelta"), ("A", "gA"), ("B", "gB"),
                         ("C", "gC"), ("D", "gD"), ("z", "gz"), ("bias", "gbias"),
                         ("h0", "gh0")):
        g = leaves[leaf].grad
        assert g is not None and g.dtype == leaves[leaf].dtype, leaf
        assert_close(host(g), ref[theirs], io, f"grad {leaf}")


def test_autograd_long_sequence_split_over_time():
    """A sequence the forward kernel splits over time chunks on its own (its chunk
    summaries carry the state), run end to end through autograd."""
    p = W.scan_problem(1, 8192, 64, 16, io="f32", seed=62, h0=True)
    assert ssm.scan_plan(1, 8192, 64, 16, torch.float32)[1] > 1
    x, delta = dev(p.x).requires_grad_(), dev(p.delta).requires_grad_()
    A, h0 = dev(p.A).requires_grad_(), dev(p.h0).requires_grad_()
    y, hf = ssm.selective_scan(x, delta, A, dev(p.B), dev(p.C), D=dev(p.D), z=dev(p.z),
                               delta_bias=dev(p.bias), h0=h0)
    yr, hr = oracle.scan(**p.oracle_args())
    assert_close(host(y), yr, "f32", "y", row_axes=(0, 2))
    rng = np.random.default_rng(63)
    gy = dev(rng.standard_normal(y.shape))
    (y * gy).sum().backward()
    ref = oracle.scan_bwd(host(gy), p.x, p.delta, p.A, p.B, p.C, Dv=p.D, z=p.z, bias=p.bias,
                          h0=p.h0)
    for leaf, theirs in ((x, "gx"), (delta, "gdelta"), (A, "gA"), (h0, "gh0")):
        assert_close(host(leaf.grad), ref[theirs], "f32", f"grad {theirs}")


def test_autograd_only_requested_gradients():
    """Inputs that need no gradient get None; the requested ones are still right."""
    p = W.scan_problem(2, 40, 24, 16, io="f32", seed=64, h0=True)
    x = dev(p.x).requires_grad_()
    B = dev(p.B).requires_grad_()
    A, D, z, bias, h0 = dev(p.A), dev(p.D), dev(p.z), dev(p.bias), dev(p.h0)
    delta = dev(p.delta)
    y, _ = ssm.selective_scan(x, delta, A, B, dev(p.C), D=D, z=z, delta_bias=bias, h0=h0)
    gy = dev(np.random.default_rng(65).standard_normal(y.shape))
    (y * gy).sum().backward()
    assert A.grad is None and delta.grad is None and h0.grad is None and D.grad is None
    ref = oracle.scan_bwd(host(gy), p.x, p.delta, p.A, p.B, p.C, Dv=p.D, z=p.z, bias=p.bias,
                          h0=p.h0)
    assert_close(host(x.grad), ref["gx"], "f32", "grad x")
    assert_close(host(B.grad), ref["gB"], "f32", "grad B")
