"""fp64 CPU oracle for the selective-SSM scan, the SSD (scalar-A multi-head)
form and the decode step.

TEST INFRASTRUCTURE ONLY: the test-suite, the smoke check and the benchmark's
CPU-baseline leg may import this package; the product path never does.  The
arithmetic lives in ``ssm_oracle.c`` (plain C, double precision, sequential in
time); this module compiles it with gcc, loads it with ctypes and marshals numpy
arrays.  It shares nothing with the CUDA library.

Every function upcasts its inputs to float64 (bf16- or fp32-valued inputs are
exactly representable) and returns float64 arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libssm_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``ssm_oracle.c`` into ``libssm_oracle.so`` (gcc, OpenMP, -O2,
    no fast-math) unless an up-to-date build exists."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    dp = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.c_int64
    lib.oracle_scan_f64.restype = ctypes.c_int
    lib.oracle_scan_f64.argtypes = [i64, i64, i64, i64] + [dp] * 8 + [ctypes.c_int, ctypes.c_int,
                                                                    dp, dp, dp, ctypes.c_int]
    lib.oracle_ssd_f64.restype = ctypes.c_int
    lib.oracle_ssd_f64.argtypes = [i64] * 6 + [dp] * 8 + [ctypes.c_int, dp, dp, dp, ctypes.c_int]
    lib.oracle_decode_f64.restype = ctypes.c_int
    lib.oracle_decode_f64.argtypes = [i64, i64, i64, dp] + [dp] * 8 + [ctypes.c_int, ctypes.c_int,
                                                                    dp, ctypes.c_int]
    lib.oracle_ssd_decode_f64.restype = ctypes.c_int
    lib.oracle_ssd_decode_f64.argtypes = [i64] * 5 + [dp] * 9 + [ctypes.c_int, dp, ctypes.c_int]
    lib.oracle_conv1d_f64.restype = ctypes.c_int
    lib.oracle_conv1d_f64.argtypes = [i64] * 4 + [dp] * 4 + [ctypes.c_int, dp, ctypes.c_int]
    lib.oracle_scan_bwd_f64.restype = ctypes.c_int
    lib.oracle_scan_bwd_f64.argtypes = ([i64] * 4 + [dp] * 8 + [ctypes.c_int, ctypes.c_int]
                                        + [dp] * 12 + [ctypes.c_int])
    lib.oracle_softplus_f64.restype = ctypes.c_double
    lib.oracle_softplus_f64.argtypes = [ctypes.c_double]
    lib.oracle_max_threads.restype = ctypes.c_int
    _lib = lib
    return lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def softplus(v: float) -> float:
    return float(_load().oracle_softplus_f64(float(v)))


def scan(x, delta, A, Bm, Cm, Dv=None, z=None, bias=None, softplus: bool = True,
         h0=None, threads: Optional[int] = None, zoh: bool = False):
    """Sequential S6 scan.  x, delta, z: (B,L,D); Bm, Cm: (B,L,N); A: (D,N);
    Dv, bias: (D,); h0: (B,D,N).  zoh selects the zero-order-hold input coefficient
    (exp(dl A) - 1) / A instead of dl.  Returns (y (B,L,D), h_final (B,D,N))."""
    lib = _load()
    x, delta, A, Bm, Cm = map(_f64, (x, delta, A, Bm, Cm))
    Dv, z, bias, h0 = map(_f64, (Dv, z, bias, h0))
    nb, L, D = x.shape
    N = A.shape[1]
    assert delta.shape == x.shape and A.shape == (D, N)
    assert Bm.shape == (nb, L, N) and Cm.shape == (nb, L, N)
    y = np.empty((nb, L, D), np.float64)
    hf = np.empty((nb, D, N), np.float64)
    rc = lib.oracle_scan_f64(nb, L, D, N, _ptr(x), _ptr(delta), _ptr(A), _ptr(Bm), _ptr(Cm),
                             _ptr(Dv), _ptr(z), _ptr(bias), int(bool(softplus)), int(bool(zoh)),
                             _ptr(h0), _ptr(y), _ptr(hf), threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_scan_f64 failed: {rc}")
    return y, hf


def scan_bwd(gy, x, delta, A, Bm, Cm, Dv=None, z=None, bias=None, softplus: bool = True,
             h0=None, gh_final=None, zoh: bool = False, threads: Optional[int] = None):
    """Gradients of scan() for the upstream gradient gy (B,L,D) (and gh_final (B,D,N)
    of the final state, zero when None).  Returns a dict with gx, gdelta (B,L,D);
    gA (D,N); gB, gC (B,L,N); gD, gbias (D,); gz (B,L,D) when z is given; gh0 (B,D,N)."""
    lib = _load()
    x, delta, A, Bm, Cm = (_f64(a) for a in (x, delta, A, Bm, Cm))
    Dv, z, bias, h0, gy, gh_final = (_f64(a) for a in (Dv, z, bias, h0, gy, gh_final))
    nb, L, D = x.shape
    N = A.shape[1]
    out = dict(gx=np.empty((nb, L, D)), gdelta=np.empty((nb, L, D)), gA=np.empty((D, N)),
               gB=np.empty((nb, L, N)), gC=np.empty((nb, L, N)), gD=np.empty(D),
               gbias=np.empty(D), gh0=np.empty((nb, D, N)))
    if z is not None:
        out["gz"] = np.empty((nb, L, D))
    rc = lib.oracle_scan_bwd_f64(nb, L, D, N, _ptr(x), _ptr(delta), _ptr(A), _ptr(Bm), _ptr(Cm),
                                 _ptr(Dv), _ptr(z), _ptr(bias), int(bool(softplus)),
                                 int(bool(zoh)), _ptr(h0), _ptr(gy), _ptr(gh_final),
                                 _ptr(out["gx"]), _ptr(out["gdelta"]), _ptr(out["gA"]),
                                 _ptr(out["gB"]), _ptr(out["gC"]), _ptr(out["gD"]),
                                 _ptr(out.get("gz")), _ptr(out["gbias"]), _ptr(out["gh0"]),
                                 threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_scan_bwd_f64 failed: {rc}")
    return out


def ssd(x, delta, A, Bm, Cm, Dv=None, z=None, bias=None, softplus: bool = True,
        h0=None, threads: Optional[int] = None):
    """Sequential multi-head scalar-A SSM.  x, z: (B,L,H,P); delta: (B,L,H);
    A, Dv, bias: (H,); Bm, Cm: (B,L,G,N); h0: (B,H,P,N).
    Returns (y (B,L,H,P), h_final (B,H,P,N))."""
    lib = _load()
    x, delta, A, Bm, Cm = map(_f64, (x, delta, A, Bm, Cm))
    Dv, z, bias, h0 = map(_f64, (Dv, z, bias, h0))
    nb, L, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    assert delta.shape == (nb, L, H) and A.shape == (H,)
    assert Bm.shape == (nb, L, G, N) and Cm.shape == Bm.shape and H % G == 0
    y = np.empty((nb, L, H, P), np.float64)
    hf = np.empty((nb, H, P, N), np.float64)
    rc = lib.oracle_ssd_f64(nb, L, H, P, G, N, _ptr(x), _ptr(delta), _ptr(A), _ptr(Bm),
                            _ptr(Cm), _ptr(Dv), _ptr(z), _ptr(bias), int(bool(softplus)),
                            _ptr(h0), _ptr(y), _ptr(hf), threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_ssd_f64 failed: {rc}")
    return y, hf


def decode_step(state, x, delta, A, Bm, Cm, Dv=None, z=None, bias=None,
                softplus: bool = True, threads: Optional[int] = None, zoh: bool = False):
    """One recurrent step.  state: (B,D,N) float64, UPDATED IN PLACE (it must
    already be a C-contiguous float64 array); x, delta, z: (B,D); Bm, Cm: (B,N);
    A: (D,N); Dv, bias: (D,).  Returns y (B,D)."""
    lib = _load()
    if not (isinstance(state, np.ndarray) and state.dtype == np.float64
            and state.flags.c_contiguous):
        raise TypeError("state must be a C-contiguous float64 numpy array")
    x, delta, A, Bm, Cm = map(_f64, (x, delta, A, Bm, Cm))
    Dv, z, bias = map(_f64, (Dv, z, bias))
    nb, D, N = state.shape
    assert x.shape == (nb, D) and A.shape == (D, N) and Bm.shape == (nb, N)
    y = np.empty((nb, D), np.float64)
    rc = lib.oracle_decode_f64(nb, D, N, _ptr(state), _ptr(x), _ptr(delta), _ptr(A), _ptr(Bm),
                               _ptr(Cm), _ptr(Dv), _ptr(z), _ptr(bias), int(bool(softplus)),
                               int(bool(zoh)), _ptr(y), threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_decode_f64 failed: {rc}")
    return y


def ssd_decode_step(state, x, delta, A, Bm, Cm, Dv=None, z=None, bias=None,
                    softplus: bool = True, threads: Optional[int] = None):
    """One token of the multi-head scalar-A recurrence.  state: (B,H,P,N) float64,
    UPDATED IN PLACE; x, z: (B,H,P); delta: (B,H); Bm, Cm: (B,G,N); A, Dv, bias: (H,).
    Returns y (B,H,P)."""
    lib = _load()
    if not (isinstance(state, np.ndarray) and state.dtype == np.float64
            and state.flags.c_contiguous):
        raise TypeError("state must be a C-contiguous float64 numpy array")
    x, delta, A, Bm, Cm = map(_f64, (x, delta, A, Bm, Cm))
    Dv, z, bias = map(_f64, (Dv, z, bias))
    nb, H, P, N = state.shape
    G = Bm.shape[1]
    assert x.shape == (nb, H, P) and delta.shape == (nb, H) and A.shape == (H,)
    assert Bm.shape == (nb, G, N) and Cm.shape == Bm.shape and H % G == 0
    y = np.empty((nb, H, P), np.float64)
    rc = lib.oracle_ssd_decode_f64(nb, H, P, G, N, _ptr(state), _ptr(x), _ptr(delta), _ptr(A),
                                   _ptr(Bm), _ptr(Cm), _ptr(Dv), _ptr(z), _ptr(bias),
                                   int(bool(softplus)), _ptr(y), threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_ssd_decode_f64 failed: {rc}")
    return y


def conv1d(x, w, bias=None, x_prev=None, silu: bool = True, threads: Optional[int] = None):
    """Causal depthwise convolution along time (kernel K, K-1 steps of left padding, or
    the carried-in x_prev (B, K-1, D)), then SiLU.  x: (B,L,D); w: (D,K); bias: (D,).
    Returns (B,L,D)."""
    lib = _load()
    x, w = _f64(x), _f64(w)
    bias, x_prev = _f64(bias), _f64(x_prev)
    nb, L, D = x.shape
    K = w.shape[1]
    assert w.shape == (D, K)
    if x_prev is not None:
        assert x_prev.shape == (nb, K - 1, D)
    out = np.empty((nb, L, D), np.float64)
    rc = lib.oracle_conv1d_f64(nb, L, D, K, _ptr(x), _ptr(w), _ptr(bias), _ptr(x_prev),
                               int(bool(silu)), _ptr(out), threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_conv1d_f64 failed: {rc}")
    return out


def rel_l2(a, b) -> float:
    """||a - b||_2 / ||b||_2 over the flattened arrays, in float64."""
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    den = float(np.linalg.norm(b))
    num = float(np.linalg.norm(a - b))
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return num / den
