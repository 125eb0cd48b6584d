"""Helpers shared by the GPU parity tests: move seeded problems to the device,
run the library through its C ABI binding, and compare with the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import selective_state_space_132_b300 as ssm

# tolerances (relative L2 over the whole tensor): fp32 I/O 1e-5, bf16 I/O 3e-3
TOL = {"f32": 1e-5, "bf16": 3e-3}


def io_dtype(io: str):
    return torch.bfloat16 if io == "bf16" else torch.float32


def dev(a, dtype=torch.float32, device="cuda"):
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device=device,
                                                                          dtype=dtype)


def host(t):
    return None if t is None else t.detach().float().cpu().numpy().astype(np.float64)


def run_scan(p, time_chunk=0, h_final=True, stream=None):
    io = io_dtype(p.io)
    y, hf = ssm.scan_fwd(dev(p.x, io), dev(p.delta, io), dev(p.A), dev(p.B, io), dev(p.C, io),
                         D=dev(p.D), z=dev(p.z, io), delta_bias=dev(p.bias),
                         delta_softplus=p.softplus, h0=dev(p.h0), return_final_state=h_final,
                         time_chunk=time_chunk, stream=stream,
                         discretization="zoh" if p.zoh else "euler")
    torch.cuda.synchronize()
    return host(y), host(hf)


def run_ssd(p, chunk=None):
    io = io_dtype(p.io)
    y, hf = ssm.ssd_chunk_fwd(dev(p.x, io), dev(p.delta, io), dev(p.A), dev(p.B, io),
                              dev(p.C, io), D=dev(p.D), z=dev(p.z, io), delta_bias=dev(p.bias),
                              delta_softplus=p.softplus, h0=dev(p.h0),
                              chunk_size=chunk if chunk is not None else p.chunk)
    torch.cuda.synchronize()
    return host(y), host(hf)


def bf16_rounding_floor(ref) -> float:
    """rel-L2 between the oracle's values and the same values rounded to bf16 (RNE):
    the error any correctly rounded bf16 output has."""
    r = torch.from_numpy(np.asarray(ref, np.float64)).to(torch.float32).to(torch.bfloat16)
    return oracle.rel_l2(r.double().numpy(), ref)


def assert_close(got, ref, io, what):
    """rel-L2 of got against the unrounded fp64 oracle within the tolerance of the I/O
    type.  For bf16 the bound is never below what rounding the oracle itself to bf16
    costs (plus 5e-4): on tiny tensors dominated by one value that floor alone can
    exceed 3e-3, and no correct bf16 result could meet the plain bound there."""
    err = oracle.rel_l2(got, ref)
    tol = TOL[io]
    if io == "bf16":
        tol = max(tol, bf16_rounding_floor(ref) + 5e-4)
    assert err <= tol, f"{what}: rel-L2 {err:.3e} > {tol:.1e}"
    return err
