"""Independent calls on different streams, in flight together, give the results they
give alone: the library keeps no state between calls (each call owns its workspace)."""
import numpy as np
import pytest
import torch

import selective_state_space_132_b300 as ssm
from selective_state_space_132_b300 import workloads as W

from _parity import dev

pytestmark = pytest.mark.gpu


def test_calls_on_concurrent_streams_match_sequential():
    t = torch.bfloat16
    scans = []
    for i in range(3):
        p = W.scan_problem(2, 400, 128, 16, io="bf16", seed=30 + i, h0=True)
        scans.append(((dev(p.x, t), dev(p.delta, t), dev(p.A), dev(p.B, t), dev(p.C, t)),
                      dict(D=dev(p.D), z=dev(p.z, t), delta_bias=dev(p.bias), h0=dev(p.h0),
                           time_chunk=(0, 64, 128)[i])))
    q = W.ssd_problem(1, 300, 3, 64, 1, 128, chunk=128, io="bf16", seed=33)
    ssd_args = ((dev(q.x, t), dev(q.delta, t), dev(q.A), dev(q.B, t), dev(q.C, t)),
                dict(D=dev(q.D), delta_bias=dev(q.bias), chunk_size=128))
    rng = np.random.default_rng(34)
    cx, cw = dev(rng.standard_normal((2, 512, 256)), t), dev(rng.standard_normal((256, 4)))
    bp = W.scan_problem(1, 120, 64, 16, io="f32", seed=35)
    bwd_args = ((dev(rng.standard_normal((1, 120, 64))), dev(bp.x), dev(bp.delta), dev(bp.A),
                 dev(bp.B), dev(bp.C)), dict(D=dev(bp.D), z=dev(bp.z), delta_bias=dev(bp.bias)))

    def run_all(streams):
        out = []
        for i, (a, kw) in enumerate(scans):
            with torch.cuda.stream(streams[i % len(streams)]):
                out.append(ssm.scan_fwd(*a, **kw))
        with torch.cuda.stream(streams[3 % len(streams)]):
            out.append(ssm.ssd_chunk_fwd(*ssd_args[0], **ssd_args[1]))
        with torch.cuda.stream(streams[4 % len(streams)]):
            out.append((ssm.conv1d(cx, cw),))
        with torch.cuda.stream(streams[5 % len(streams)]):
            g = ssm.scan_bwd(*bwd_args[0], **bwd_args[1])
            out.append((g["dx"], g["ddelta"], g["dz"], g["dh0"]))
        return out

    seq = run_all([torch.cuda.current_stream()])
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(6)]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    conc = run_all(streams)
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(zip(seq, conc)):
        for u, v in zip(a, b):
            assert torch.equal(u, v), f"call {i}"
