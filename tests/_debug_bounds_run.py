"""Runs every GPU entry point once on ragged shapes, on both kernel paths of each, with
the library named by SSM_LIBRARY (the debug-bounds build), and prints one JSON line per
call: the device status word after the call and the rel-L2 error against the oracle.
Called by tests/test_debug_bounds.py in a subprocess (one library per process)."""
import json
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import oracle  # noqa: E402
import selective_state_space_132_b300 as ssm  # noqa: E402
from selective_state_space_132_b300 import workloads as W  # noqa: E402

from _parity import dev, host, io_dtype  # noqa: E402


def ws(nbytes):
    return torch.empty(max(256, nbytes), dtype=torch.uint8, device="cuda")


def report(name, workspace, err):
    torch.cuda.synchronize()
    print(json.dumps({"call": name, "status": ssm.read_device_status(workspace),
                      "rel_l2": float(err)}), flush=True)


def main():
    assert ssm.library_path().endswith("libssm_debug.so"), ssm.library_path()
    # S6 scan: TMA kernel (whole, split over time, with checkpoints) and general kernel
    for io, D, N, tc, ck in [("bf16", 64, 16, 0, False), ("bf16", 64, 16, 64, True),
                             ("f32", 45, 5, 96, True), ("bf16", 96, 64, 0, False)]:
        p = W.scan_problem(2, 300, D, N, io=io, seed=900 + D + N, h0=True)
        t = io_dtype(io)
        a = (dev(p.x, t), dev(p.delta, t), dev(p.A), dev(p.B, t), dev(p.C, t))
        kw = dict(D=dev(p.D), z=dev(p.z, t), delta_bias=dev(p.bias), h0=dev(p.h0),
                  time_chunk=tc)
        w = ws(ssm.scan_workspace_size(2, 300, D, N, t, tc))
        out = ssm.scan_fwd(*a, workspace=w, checkpoints=True if ck else None, **kw)
        yr, hr = oracle.scan(**p.oracle_args())
        report(f"scan {io} D{D} N{N} chunk{tc} ckpt{ck}", w, oracle.rel_l2(host(out[0]), yr))
        # backward, from its own checkpoints and from the forward's
        gy = dev(np.random.default_rng(1).standard_normal((2, 300, D)), t)
        wb = ws(ssm.scan_bwd_workspace_size(2, 300, D, N, t))
        g = ssm.scan_bwd(gy, *a, D=kw["D"], z=kw["z"], delta_bias=kw["delta_bias"],
                         h0=kw["h0"], workspace=wb, checkpoints=out[2] if ck else None)
        report(f"scan_bwd {io} D{D} N{N} ckpt{ck}", wb,
               0.0 if np.all(np.isfinite(host(g["dx"]))) else 1.0)
    # SSD: tensor-core kernel (ragged, several chains split between blocks) and sequential
    for P, N, H in [(64, 128, 5), (16, 64, 3)]:
        p = W.ssd_problem(2, 300, H, P, 1, N, chunk=128, io="bf16", seed=950 + P, h0=True)
        t = torch.bfloat16
        w = ws(ssm.ssd_workspace_size(dev(p.x, t), dev(p.delta, t), dev(p.A), dev(p.B, t),
                                      dev(p.C, t), 128))
        y, _ = ssm.ssd_chunk_fwd(dev(p.x, t), dev(p.delta, t), dev(p.A), dev(p.B, t),
                                 dev(p.C, t), D=dev(p.D), delta_bias=dev(p.bias), h0=dev(p.h0),
                                 chunk_size=128, workspace=w)
        yr, _ = oracle.ssd(**p.oracle_args())
        report(f"ssd P{P} N{N} H{H}", w, oracle.rel_l2(host(y), yr))
    # decode step: bulk-copy kernel (N 16) and general kernel (N 5)
    for N in (16, 5):
        p = W.decode_problem(8, 200, N, 1, io="bf16", seed=970 + N)
        tok = p.tokens(0)
        t = torch.bfloat16
        state = dev(p.state0)
        w = ws(256)
        y = ssm.step_decode(state, dev(tok["x"], t), dev(tok["delta"], t), dev(p.A),
                            dev(tok["B"], t), dev(tok["C"], t), D=dev(p.D), z=dev(tok["z"], t),
                            delta_bias=dev(p.bias), workspace=w)
        ref = oracle.decode_step(np.ascontiguousarray(p.state0, np.float64), tok["x"],
                                 tok["delta"], p.A, tok["B"], tok["C"], Dv=p.D, z=tok["z"],
                                 bias=p.bias)
        report(f"decode N{N}", w, oracle.rel_l2(host(y), ref))
    # conv1d: TMA kernel (D 128) and general kernel (D 20)
    for D in (128, 20):
        rng = np.random.default_rng(980 + D)
        x = rng.standard_normal((2, 300, D)).astype(np.float32)
        wt = (0.5 * rng.standard_normal((D, 4))).astype(np.float32)
        xb = dev(x, torch.bfloat16)
        w = ws(256)
        out = ssm.conv1d(xb, dev(wt), workspace=w)
        ref = oracle.conv1d(host(xb), wt)
        report(f"conv1d D{D}", w, oracle.rel_l2(host(out), ref))


if __name__ == "__main__":
    main()
