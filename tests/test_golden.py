"""The fixtures under tests/golden/ (written by tests/golden/make_golden.py from the
oracle): the oracle still reproduces them (a change of its arithmetic must be
deliberate), and the CUDA entry points match them at the fp32 tolerance."""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        d = json.load(f)
    return d, {k: np.asarray(v, np.float64) for k, v in d["inputs"].items()}


def test_oracle_reproduces_scan_fixture():
    d, p = _load("scan_small.json")
    y, hf = oracle.scan(p["x"], p["delta"], p["A"], p["B"], p["C"], Dv=p["D"], z=p["z"],
                        bias=p["bias"], softplus=True, threads=1)
    np.testing.assert_allclose(y, d["y"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(hf, d["h_final"], rtol=1e-14, atol=1e-15)
    g = oracle.scan_bwd(p["dy"], p["x"], p["delta"], p["A"], p["B"], p["C"], Dv=p["D"],
                        z=p["z"], bias=p["bias"], softplus=True)
    for k, v in d["grads"].items():
        np.testing.assert_allclose(g[k], v, rtol=1e-13, atol=1e-14, err_msg=k)


def test_oracle_reproduces_conv1d_fixture():
    d, p = _load("conv1d_small.json")
    out = oracle.conv1d(p["x"], p["w"], p["bias"], silu=True)
    np.testing.assert_allclose(out, d["out"], rtol=1e-14, atol=1e-15)


@pytest.mark.gpu
def test_cuda_matches_fixtures():
    import torch
    import selective_state_space_132_b300 as ssm

    def t(a):
        return torch.tensor(np.asarray(a, np.float32), device="cuda")

    d, p = _load("scan_small.json")
    y, hf = ssm.scan_fwd(t(p["x"]), t(p["delta"]), t(p["A"]), t(p["B"]), t(p["C"]), D=t(p["D"]),
                         z=t(p["z"]), delta_bias=t(p["bias"]))
    g = ssm.scan_bwd(t(p["dy"]), t(p["x"]), t(p["delta"]), t(p["A"]), t(p["B"]), t(p["C"]),
                     D=t(p["D"]), z=t(p["z"]), delta_bias=t(p["bias"]))
    torch.cuda.synchronize()
    assert oracle.rel_l2(y.double().cpu().numpy(), d["y"]) <= 1e-5
    assert oracle.rel_l2(hf.double().cpu().numpy(), d["h_final"]) <= 1e-5
    for mine, theirs in (("dx", "gx"), ("ddelta", "gdelta"), ("dA", "gA"), ("dB", "gB"),
                         ("dC", "gC"), ("dD", "gD"), ("ddelta_bias", "gbias"), ("dz", "gz"),
                         ("dh0", "gh0")):
        got = g[mine].double().cpu().numpy()
        assert oracle.rel_l2(got, d["grads"][theirs]) <= 1e-5, mine
    d, p = _load("conv1d_small.json")
    out = ssm.conv1d(t(p["x"]), t(p["w"]), t(p["bias"]))
    torch.cuda.synchronize()
    assert oracle.rel_l2(out.double().cpu().numpy(), d["out"]) <= 1e-5
