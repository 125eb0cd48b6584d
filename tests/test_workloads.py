"""The seeded input recipes: deterministic, correctly shaped and bf16-exact."""
import numpy as np
import torch

from selective_state_space_132_b300 import workloads as W


def test_round_bf16_matches_torch_rne():
    rng = np.random.Generator(np.random.PCG64(0))
    a = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 3,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 65504.0, 1e-30],
                                 np.float32)])
    ours = W.round_bf16(a)
    ref = torch.from_numpy(a).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(ours.view(np.uint32), ref.view(np.uint32))


def test_problems_are_deterministic_and_shaped():
    p1 = W.config_problem(1, batch=2, seqlen=40, dim=24)
    p2 = W.config_problem(1, batch=2, seqlen=40, dim=24)
    for k in ("x", "delta", "B", "C", "z", "D", "bias", "A"):
        np.testing.assert_array_equal(getattr(p1, k), getattr(p2, k))
    assert p1.x.shape == (2, 40, 24) and p1.B.shape == (2, 40, 16) and p1.A.shape == (24, 16)
    np.testing.assert_array_equal(W.round_bf16(p1.x), p1.x)
    assert np.all(p1.A == -np.arange(1, 17, dtype=np.float32)[None, :])
    s = W.config_problem(3, batch=1, seqlen=64, heads=4)
    assert s.x.shape == (1, 64, 4, 64) and s.B.shape == (1, 64, 1, 128) and s.z is None
    assert np.all((s.A <= -1.0) & (s.A >= -16.0))
    d = W.config_problem(4, batch=3, dim=40, steps=2)
    t0, t0b = d.tokens(0), d.tokens(0)
    np.testing.assert_array_equal(t0["x"], t0b["x"])
    assert not np.array_equal(t0["x"], d.tokens(1)["x"])
    assert d.state0.shape == (3, 40, 16)


def test_config_zero_is_fp32():
    p = W.config_problem(0)
    assert p.io == "f32" and p.x.shape == (1, 64, 16) and p.A.shape == (16, 4)
    assert p.z is not None and p.h0 is None
