"""The entry points can be captured in CUDA graphs: no host synchronisation and no
allocation outside PyTorch's (graph-aware) allocator on the call path.  A captured call
replays to the bit-identical result of a direct call."""
import numpy as np
import pytest
import torch

import selective_state_space_132_b300 as ssm
from selective_state_space_132_b300 import workloads as W

from _parity import dev

pytestmark = pytest.mark.gpu


def _capture(fn):
    """Warm up fn on a side stream (allocations, one-time lookups), capture it, replay."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = fn()
    g.replay()
    torch.cuda.synchronize()
    return g, out


@pytest.mark.parametrize("tc", [0, 64])
def test_scan_in_a_graph(tc):
    p = W.scan_problem(2, 300, 96, 16, io="bf16", seed=21, h0=True)
    t = torch.bfloat16
    a = (dev(p.x, t), dev(p.delta, t), dev(p.A), dev(p.B, t), dev(p.C, t))
    kw = dict(D=dev(p.D), z=dev(p.z, t), delta_bias=dev(p.bias), h0=dev(p.h0), time_chunk=tc)
    y_ref, h_ref = ssm.scan_fwd(*a, **kw)
    g, (y, h) = _capture(lambda: ssm.scan_fwd(*a, **kw))
    assert torch.equal(y, y_ref) and torch.equal(h, h_ref)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, y_ref)


def test_ssd_in_a_graph():
    p = W.ssd_problem(1, 300, 3, 64, 1, 128, chunk=128, io="bf16", seed=22)
    t = torch.bfloat16
    a = (dev(p.x, t), dev(p.delta, t), dev(p.A), dev(p.B, t), dev(p.C, t))
    kw = dict(D=dev(p.D), delta_bias=dev(p.bias), chunk_size=128)
    y_ref, h_ref = ssm.ssd_chunk_fwd(*a, **kw)
    g, (y, h) = _capture(lambda: ssm.ssd_chunk_fwd(*a, **kw))
    assert torch.equal(y, y_ref) and torch.equal(h, h_ref)


def test_decode_steps_in_a_graph():
    """Eight decode steps captured as one graph advance the state exactly like eight
    direct calls."""
    p = W.decode_problem(4, 256, 16, 8, io="bf16", seed=23)
    t = torch.bfloat16
    toks = [{k: dev(v, t) for k, v in p.tokens(s).items()} for s in range(8)]
    A, Dv, bias = dev(p.A), dev(p.D), dev(p.bias)

    def steps(state):
        return [ssm.step_decode(state, k["x"], k["delta"], A, k["B"], k["C"], D=Dv, z=k["z"],
                                delta_bias=bias) for k in toks]
    ref_state = dev(p.state0)
    ys_ref = steps(ref_state)
    state = dev(p.state0)
    warm = dev(p.state0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        steps(warm)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ys = steps(state)
    state.copy_(dev(p.state0))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(state, ref_state)
    assert all(torch.equal(a, b) for a, b in zip(ys, ys_ref))


def test_conv1d_and_backward_in_a_graph():
    rng = np.random.default_rng(24)
    t = torch.bfloat16
    x = dev(rng.standard_normal((2, 256, 128)), t)
    w = dev(rng.standard_normal((128, 4)))
    out_ref = ssm.conv1d(x, w)
    g, out = _capture(lambda: ssm.conv1d(x, w))
    assert torch.equal(out, out_ref)

    p = W.scan_problem(2, 100, 64, 16, io="f32", seed=25, h0=True)
    a = (dev(p.x), dev(p.delta), dev(p.A), dev(p.B), dev(p.C))
    dy = dev(rng.standard_normal((2, 100, 64)))
    kw = dict(D=dev(p.D), z=dev(p.z), delta_bias=dev(p.bias), h0=dev(p.h0))
    ref = ssm.scan_bwd(dy, *a, **kw)
    g2, got = _capture(lambda: ssm.scan_bwd(dy, *a, **kw))
    for k in ("dx", "ddelta", "dz", "dh0"):
        assert torch.equal(got[k], ref[k]), k
    for k in ("dA", "dB", "dC", "dD", "ddelta_bias"):
        assert torch.allclose(got[k], ref[k], rtol=1e-5, atol=1e-6), k
