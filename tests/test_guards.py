"""Out-of-bounds writes and run-to-run races, without a sanitizer: every output lives
inside a larger buffer whose guard regions hold a sentinel that must survive the call,
and repeated calls on the same inputs must give bit-identical results (the sums that
the scan backward accumulates with atomics may differ in the last bits only)."""
import ctypes

import numpy as np
import pytest
import torch

import selective_state_space_132_b300 as ssm
from selective_state_space_132_b300 import binding as bd
from selective_state_space_132_b300 import workloads as W

from _parity import dev, io_dtype

pytestmark = pytest.mark.gpu

GUARD = 4096          # elements on each side (keeps 16-byte alignment for every dtype)
SENTINEL = 1024.0     # exact in bf16 and fp32


class Guarded:
    def __init__(self, shape, dtype):
        n = int(np.prod(shape))
        self.base = torch.full((GUARD + n + GUARD,), SENTINEL, dtype=dtype, device="cuda")
        self.t = self.base[GUARD:GUARD + n].view(shape)

    def intact(self):
        torch.cuda.synchronize()
        return bool((self.base[:GUARD] == SENTINEL).all() and (self.base[-GUARD:] == SENTINEL).all())


def _scan_inputs(io, D, N, L=77, nb=3, seed=5):
    p = W.scan_problem(nb, L, D, N, io=io, seed=seed, h0=True)
    t = io_dtype(io)
    return p, dict(x=dev(p.x, t), delta=dev(p.delta, t), A=dev(p.A), B=dev(p.B, t),
                   C=dev(p.C, t), D=dev(p.D), z=dev(p.z, t), delta_bias=dev(p.bias),
                   h0=dev(p.h0))


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("D,N,tc", [(45, 16, 0), (64, 16, 0), (64, 16, 32), (96, 5, 0)])
def test_scan_writes_stay_inside_and_repeat(io, D, N, tc):
    p, a = _scan_inputs(io, D, N)
    t = io_dtype(io)
    y = Guarded((p.batch, p.seqlen, D), t)
    hf = Guarded((p.batch, D, N), torch.float32)
    ssm.scan_fwd(a["x"], a["delta"], a["A"], a["B"], a["C"], D=a["D"], z=a["z"],
                 delta_bias=a["delta_bias"], h0=a["h0"], y=y.t, h_final=hf.t, time_chunk=tc)
    assert y.intact() and hf.intact()
    y1, h1 = y.t.clone(), hf.t.clone()
    ssm.scan_fwd(a["x"], a["delta"], a["A"], a["B"], a["C"], D=a["D"], z=a["z"],
                 delta_bias=a["delta_bias"], h0=a["h0"], y=y.t, h_final=hf.t, time_chunk=tc)
    torch.cuda.synchronize()
    assert torch.equal(y.t, y1) and torch.equal(hf.t, h1)


@pytest.mark.parametrize("P,N,H,L", [(64, 128, 3, 300), (16, 64, 4, 130)])
def test_ssd_writes_stay_inside_and_repeat(P, N, H, L):
    p = W.ssd_problem(2, L, H, P, 1, N, chunk=128, io="bf16", seed=6, h0=True)
    t = torch.bfloat16
    y = Guarded((2, L, H, P), t)
    hf = Guarded((2, H, P, N), torch.float32)
    args = (dev(p.x, t), dev(p.delta, t), dev(p.A), dev(p.B, t), dev(p.C, t))
    kw = dict(D=dev(p.D), delta_bias=dev(p.bias), h0=dev(p.h0), chunk_size=128)
    ssm.ssd_chunk_fwd(*args, y=y.t, h_final=hf.t, **kw)
    assert y.intact() and hf.intact()
    y1, h1 = y.t.clone(), hf.t.clone()
    ssm.ssd_chunk_fwd(*args, y=y.t, h_final=hf.t, **kw)
    torch.cuda.synchronize()
    assert torch.equal(y.t, y1) and torch.equal(hf.t, h1)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("D,K", [(64, 4), (40, 3), (37, 4)])
def test_conv1d_writes_stay_inside_and_repeat(io, D, K):
    rng = np.random.default_rng(7)
    t = io_dtype(io)
    x = dev(rng.standard_normal((2, 200, D)), t)
    w = dev(rng.standard_normal((D, K)))
    out = Guarded((2, 200, D), t)
    ssm.conv1d(x, w, out=out.t)
    assert out.intact()
    o1 = out.t.clone()
    ssm.conv1d(x, w, out=out.t)
    torch.cuda.synchronize()
    assert torch.equal(out.t, o1)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("D,N", [(37, 16), (64, 16), (20, 64)])
def test_decode_writes_stay_inside(io, D, N):
    p = W.decode_problem(5, D, N, 1, io=io, seed=8)
    t = io_dtype(io)
    state = Guarded((5, D, N), torch.float32)
    state.t.copy_(dev(p.state0))
    y = Guarded((5, D), t)
    tok = p.tokens(0)
    ssm.step_decode(state.t, dev(tok["x"], t), dev(tok["delta"], t), dev(p.A), dev(tok["B"], t),
                    dev(tok["C"], t), D=dev(p.D), z=dev(tok["z"], t), delta_bias=dev(p.bias),
                    y=y.t)
    assert state.intact() and y.intact()


@pytest.mark.parametrize("N", [16, 128, 200])
def test_ssd_decode_writes_stay_inside(N):
    p = W.ssd_problem(3, 1, 4, 64, 2, N, io="bf16", seed=9, h0=True)
    t = torch.bfloat16
    state = Guarded((3, 4, 64, N), torch.float32)
    state.t.copy_(dev(p.h0))
    y = Guarded((3, 4, 64), t)
    ssm.ssd_step_decode(state.t, dev(p.x[:, 0], t), dev(p.delta[:, 0], t), dev(p.A),
                        dev(p.B[:, 0], t), dev(p.C[:, 0], t), D=dev(p.D), delta_bias=dev(p.bias),
                        y=y.t)
    assert state.intact() and y.intact()


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("D,N", [(45, 16), (64, 32), (20, 5)])
def test_scan_bwd_writes_stay_inside_and_repeat(io, D, N):
    p, a = _scan_inputs(io, D, N, L=60, nb=2, seed=10)
    t = io_dtype(io)
    nb, L = p.batch, p.seqlen
    dy = dev(np.random.default_rng(3).standard_normal((nb, L, D)), t)
    g = dict(dx=Guarded((nb, L, D), t), ddelta=Guarded((nb, L, D), t), dz=Guarded((nb, L, D), t),
             dA=Guarded((D, N), torch.float32), dB=Guarded((nb, L, N), torch.float32),
             dC=Guarded((nb, L, N), torch.float32), dD=Guarded((D,), torch.float32),
             ddelta_bias=Guarded((D,), torch.float32), dh0=Guarded((nb, D, N), torch.float32))
    lib = ssm.load_library()

    def run():
        args = bd.ScanBwdArgs(nb, L, D, N, 1 if io == "bf16" else 0, 1, 0, 0,
                              a["x"].data_ptr(), a["delta"].data_ptr(), a["B"].data_ptr(),
                              a["C"].data_ptr(), a["z"].data_ptr(), a["A"].data_ptr(),
                              a["D"].data_ptr(), a["delta_bias"].data_ptr(), a["h0"].data_ptr(),
                              dy.data_ptr(), None, *(g[k].t.data_ptr() for k in (
                                  "dx", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias",
                                  "dh0")), None, 0)
        need = ctypes.c_size_t(0)
        assert lib.ssm_scan_bwd_workspace_size(ctypes.byref(args), ctypes.byref(need)) == 0
        ws = torch.empty(need.value, dtype=torch.uint8, device="cuda")
        args.workspace, args.workspace_bytes = ws.data_ptr(), need.value
        assert lib.ssm_scan_bwd(ctypes.byref(args), None) == 0
        torch.cuda.synchronize()

    run()
    assert all(v.intact() for v in g.values())
    first = {k: v.t.clone() for k, v in g.items()}
    run()
    for k in ("dx", "ddelta", "dz", "dh0"):          # written once per element
        assert torch.equal(g[k].t, first[k]), k
    for k in ("dA", "dB", "dC", "dD", "ddelta_bias"):  # summed with fp32 atomics
        assert torch.allclose(g[k].t, first[k], rtol=1e-5, atol=1e-6), k


@pytest.mark.parametrize("io,D,N,tc", [("bf16", 64, 16, 0), ("bf16", 64, 16, 32),
                                       ("f32", 45, 5, 0), ("bf16", 32, 64, 0)])
def test_scan_checkpoints_stay_inside_and_repeat(io, D, N, tc):
    """ssm_scan_fwd_ckpt writes the checkpoints inside their buffer (ragged last
    checkpoint interval: L = 77), the same on every call, and ssm_scan_bwd_ckpt reads
    them without writing outside its outputs."""
    p, a = _scan_inputs(io, D, N)
    t = io_dtype(io)
    shape = ssm.scan_ckpt_shape(p.batch, p.seqlen, D, N)
    ck = Guarded(shape, torch.float32)
    y = Guarded((p.batch, p.seqlen, D), t)

    def fwd():
        ssm.scan_fwd(a["x"], a["delta"], a["A"], a["B"], a["C"], D=a["D"], z=a["z"],
                     delta_bias=a["delta_bias"], h0=a["h0"], y=y.t, time_chunk=tc,
                     checkpoints=ck.t)
        torch.cuda.synchronize()
    fwd()
    assert ck.intact() and y.intact()
    first = ck.t.clone()
    fwd()
    assert torch.equal(ck.t, first)
    dy = dev(np.random.default_rng(4).standard_normal((p.batch, p.seqlen, D)), t)
    dx = Guarded((p.batch, p.seqlen, D), t)
    g = ssm.scan_bwd(dy, a["x"], a["delta"], a["A"], a["B"], a["C"], D=a["D"], z=a["z"],
                     delta_bias=a["delta_bias"], h0=a["h0"], checkpoints=ck.t)
    dx.t.copy_(g["dx"])
    torch.cuda.synchronize()
    assert ck.intact() and torch.equal(ck.t, first)
