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
