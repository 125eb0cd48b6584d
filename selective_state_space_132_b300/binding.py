"""ctypes binding of libssm.so (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# SSM_LIBRARY names another build of the same library (e.g. one compiled with different
# tile switches); by default the in-tree build next to this file is loaded.
_LIB_PATH = os.environ.get("SSM_LIBRARY") or os.path.join(_HERE, "libssm.so")
_lib = None

SSM_F32, SSM_BF16 = 0, 1
_STATUS = {0: "SSM_OK", 1: "SSM_ERR_INVALID_ARG", 2: "SSM_ERR_UNSUPPORTED",
           3: "SSM_ERR_ALIGNMENT", 4: "SSM_ERR_WORKSPACE", 5: "SSM_ERR_CUDA",
           6: "SSM_ERR_TIMEOUT", 7: "SSM_ERR_BOUNDS"}

EXPORTED = ["ssm_scan_workspace_size", "ssm_scan_plan", "ssm_scan_fwd", "ssm_scan_fwd_noalloc",
            "ssm_scan_bwd_workspace_size", "ssm_scan_bwd",
            "ssm_scan_ckpt_size", "ssm_scan_fwd_ckpt", "ssm_scan_bwd_ckpt",
            "ssm_ssd_workspace_size", "ssm_ssd_chunk_fwd", "ssm_ssd_plan", "ssm_step_decode",
            "ssm_ssd_step_decode", "ssm_conv1d", "ssm_status_string", "ssm_version",
            "ssm_check_bounded_wait", "ssm_check_scan_lookback",
            "ssm_read_device_status"]

_i64, _i32, _vp, _fp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p


class ScanArgs(ctypes.Structure):
    _fields_ = [("batch", _i64), ("seqlen", _i64), ("dim", _i64), ("dstate", _i64),
                ("time_chunk", _i64), ("io_dtype", _i32), ("delta_softplus", _i32),
                ("x", _vp), ("delta", _vp), ("B", _vp), ("C", _vp), ("z", _vp),
                ("A", _fp), ("D", _fp), ("delta_bias", _fp), ("h0", _fp),
                ("y", _vp), ("h_final", _fp), ("workspace", _vp),
                ("workspace_bytes", ctypes.c_size_t), ("discretization", _i32),
                ("reserved", _i32)]


class SSDArgs(ctypes.Structure):
    _fields_ = [("batch", _i64), ("seqlen", _i64), ("nheads", _i64), ("headdim", _i64),
                ("ngroups", _i64), ("dstate", _i64), ("chunk_size", _i64),
                ("io_dtype", _i32), ("delta_softplus", _i32),
                ("x", _vp), ("delta", _vp), ("B", _vp), ("C", _vp), ("z", _vp),
                ("A", _fp), ("D", _fp), ("delta_bias", _fp), ("h0", _fp),
                ("y", _vp), ("h_final", _fp), ("workspace", _vp),
                ("workspace_bytes", ctypes.c_size_t)]


class DecodeArgs(ctypes.Structure):
    _fields_ = [("batch", _i64), ("dim", _i64), ("dstate", _i64),
                ("io_dtype", _i32), ("delta_softplus", _i32), ("state", _fp),
                ("x", _vp), ("delta", _vp), ("B", _vp), ("C", _vp), ("z", _vp),
                ("A", _fp), ("D", _fp), ("delta_bias", _fp), ("y", _vp),
                ("discretization", _i32), ("reserved", _i32),
                ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t)]


class ScanBwdArgs(ctypes.Structure):
    _fields_ = [("batch", _i64), ("seqlen", _i64), ("dim", _i64), ("dstate", _i64),
                ("io_dtype", _i32), ("delta_softplus", _i32), ("discretization", _i32),
                ("reserved", _i32), ("x", _vp), ("delta", _vp), ("B", _vp), ("C", _vp),
                ("z", _vp), ("A", _fp), ("D", _fp), ("delta_bias", _fp), ("h0", _fp),
                ("dy", _vp), ("dh_final", _fp), ("dx", _vp), ("ddelta", _vp), ("dz", _vp),
                ("dA", _fp), ("dB", _fp), ("dC", _fp), ("dD", _fp), ("ddelta_bias", _fp),
                ("dh0", _fp), ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t)]


class Conv1dArgs(ctypes.Structure):
    _fields_ = [("batch", _i64), ("seqlen", _i64), ("dim", _i64), ("width", _i64),
                ("io_dtype", _i32), ("silu", _i32), ("x", _vp), ("x_prev", _vp),
                ("weight", _fp), ("bias", _fp), ("out", _vp), ("workspace", _vp),
                ("workspace_bytes", ctypes.c_size_t)]


DISCRETIZATIONS = {"euler": 0, "zoh": 1}


def _disc(name: str) -> int:
    if name not in DISCRETIZATIONS:
        raise ValueError(f"discretization must be one of {sorted(DISCRETIZATIONS)}")
    return DISCRETIZATIONS[name]


class SSDDecodeArgs(ctypes.Structure):
    _fields_ = [("batch", _i64), ("nheads", _i64), ("headdim", _i64), ("ngroups", _i64),
                ("dstate", _i64), ("io_dtype", _i32), ("delta_softplus", _i32),
                ("state", _fp), ("x", _vp), ("delta", _vp), ("B", _vp), ("C", _vp), ("z", _vp),
                ("A", _fp), ("D", _fp), ("delta_bias", _fp), ("y", _vp)]


class SSMError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _STATUS.get(status, str(status))
        try:
            msg += ": " + load_library().ssm_status_string(status).decode()
        except Exception:
            pass
        super().__init__(f"{where} failed with {msg}")


def library_path() -> str:
    return _LIB_PATH


def build_library(force: bool = False) -> str:
    from .build import build
    return build(force=force)


def load_library():
    """Load libssm.so from the package directory (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                           "`python -m selective_state_space_132_b300.build`")
    lib = ctypes.CDLL(_LIB_PATH)
    lib.ssm_scan_workspace_size.argtypes = [ctypes.POINTER(ScanArgs),
                                            ctypes.POINTER(ctypes.c_size_t)]
    lib.ssm_scan_fwd.argtypes = [ctypes.POINTER(ScanArgs), _vp]
    lib.ssm_scan_fwd_noalloc.argtypes = [ctypes.POINTER(ScanArgs), _vp]
    lib.ssm_scan_plan.argtypes = [ctypes.POINTER(ScanArgs), ctypes.POINTER(ctypes.c_int64),
                                  ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
    lib.ssm_ssd_workspace_size.argtypes = [ctypes.POINTER(SSDArgs),
                                           ctypes.POINTER(ctypes.c_size_t)]
    lib.ssm_ssd_chunk_fwd.argtypes = [ctypes.POINTER(SSDArgs), _vp]
    lib.ssm_ssd_plan.argtypes = [ctypes.POINTER(SSDArgs), ctypes.POINTER(ctypes.c_int32)]
    lib.ssm_step_decode.argtypes = [ctypes.POINTER(DecodeArgs), _vp]
    lib.ssm_ssd_step_decode.argtypes = [ctypes.POINTER(SSDDecodeArgs), _vp]
    lib.ssm_ssd_step_decode.restype = ctypes.c_int
    lib.ssm_scan_bwd_workspace_size.argtypes = [ctypes.POINTER(ScanBwdArgs),
                                                ctypes.POINTER(ctypes.c_size_t)]
    lib.ssm_scan_bwd_workspace_size.restype = ctypes.c_int
    lib.ssm_scan_bwd.argtypes = [ctypes.POINTER(ScanBwdArgs), _vp]
    lib.ssm_scan_bwd.restype = ctypes.c_int
    lib.ssm_scan_ckpt_size.argtypes = [ctypes.POINTER(ScanArgs), ctypes.POINTER(ctypes.c_int64),
                                       ctypes.POINTER(ctypes.c_size_t)]
    lib.ssm_scan_ckpt_size.restype = ctypes.c_int
    lib.ssm_scan_fwd_ckpt.argtypes = [ctypes.POINTER(ScanArgs), _vp, ctypes.c_size_t, _vp]
    lib.ssm_scan_fwd_ckpt.restype = ctypes.c_int
    lib.ssm_scan_bwd_ckpt.argtypes = [ctypes.POINTER(ScanBwdArgs), _vp, ctypes.c_size_t, _vp]
    lib.ssm_scan_bwd_ckpt.restype = ctypes.c_int
    lib.ssm_conv1d.argtypes = [ctypes.POINTER(Conv1dArgs), _vp]
    lib.ssm_conv1d.restype = ctypes.c_int
    lib.ssm_read_device_status.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_int)]
    lib.ssm_check_bounded_wait.argtypes = [_vp, ctypes.c_int64, _vp]
    lib.ssm_check_bounded_wait.restype = ctypes.c_int
    lib.ssm_check_scan_lookback.argtypes = [ctypes.POINTER(ScanArgs), ctypes.c_int64, _vp]
    lib.ssm_check_scan_lookback.restype = ctypes.c_int
    for fn in ("ssm_scan_workspace_size", "ssm_scan_plan", "ssm_scan_fwd", "ssm_scan_fwd_noalloc",
               "ssm_ssd_workspace_size", "ssm_ssd_chunk_fwd", "ssm_ssd_plan", "ssm_step_decode",
               "ssm_read_device_status"):
        getattr(lib, fn).restype = ctypes.c_int
    lib.ssm_status_string.argtypes = [ctypes.c_int]
    lib.ssm_status_string.restype = ctypes.c_char_p
    lib.ssm_version.restype = ctypes.c_int
    _lib = lib
    return lib


def version() -> int:
    return int(load_library().ssm_version())


# ---------------------------------------------------------------- helpers
def _io_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SSM_BF16
    if t.dtype == torch.float32:
        return SSM_F32
    raise TypeError(f"I/O tensors must be bfloat16 or float32, got {t.dtype}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _check(t: Optional[torch.Tensor], name: str, shape, dtype, device):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream(stream, device=None) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _launch(fn, args, stream, device, where: str):
    """Call a compute entry point with the tensors' device current (the library
    launches on the current device) and, by default, that device's current stream."""
    with torch.cuda.device(device):
        _raise(fn(ctypes.byref(args), _stream(stream, device)), where)


def _raise(rc: int, where: str):
    if rc != 0:
        raise SSMError(rc, where)


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor]):
    if nbytes == 0:
        return None, 0
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError(f"workspace of {workspace.numel()} bytes < {nbytes} needed")
    return workspace, workspace.numel() * workspace.element_size()


# ---------------------------------------------------------------- scan
def _scan_args(x, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, y, h_final,
               time_chunk, discretization: str = "euler") -> ScanArgs:
    nb, L, Dm = x.shape
    N = A.shape[1]
    dev, io = x.device, x.dtype
    _io_code(x)
    _check(delta, "delta", (nb, L, Dm), io, dev)
    _check(A, "A", (Dm, N), torch.float32, dev)
    _check(B, "B", (nb, L, N), io, dev)
    _check(C, "C", (nb, L, N), io, dev)
    _check(D, "D", (Dm,), torch.float32, dev)
    _check(z, "z", (nb, L, Dm), io, dev)
    _check(delta_bias, "delta_bias", (Dm,), torch.float32, dev)
    _check(h0, "h0", (nb, Dm, N), torch.float32, dev)
    _check(y, "y", (nb, L, Dm), io, dev)
    _check(h_final, "h_final", (nb, Dm, N), torch.float32, dev)
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    a = ScanArgs(nb, L, Dm, N, int(time_chunk), _io_code(x), int(bool(delta_softplus)),
                 _ptr(x), _ptr(delta), _ptr(B), _ptr(C), _ptr(z), _ptr(A), _ptr(D),
                 _ptr(delta_bias), _ptr(h0), _ptr(y), _ptr(h_final), None, 0)
    a.discretization = _disc(discretization)
    return a


def scan_workspace_size(batch: int, seqlen: int, dim: int, dstate: int,
                        io_dtype=torch.bfloat16, time_chunk: int = 0) -> int:
    a = ScanArgs(batch, seqlen, dim, dstate, int(time_chunk),
                 SSM_BF16 if io_dtype == torch.bfloat16 else SSM_F32, 1,
                 None, None, None, None, None, None, None, None, None, None, None, None, 0)
    out = ctypes.c_size_t(0)
    _raise(load_library().ssm_scan_workspace_size(ctypes.byref(a), ctypes.byref(out)),
           "ssm_scan_workspace_size")
    return int(out.value)


def scan_plan(batch: int, seqlen: int, dim: int, dstate: int, io_dtype=torch.bfloat16,
              time_chunk: int = 0):
    """(steps per time chunk, number of chunks, kernel launches per call)."""
    a = ScanArgs(batch, seqlen, dim, dstate, int(time_chunk),
                 SSM_BF16 if io_dtype == torch.bfloat16 else SSM_F32, 1,
                 None, None, None, None, None, None, None, None, None, None, None, None, 0)
    cl, k, n = ctypes.c_int64(0), ctypes.c_int32(0), ctypes.c_int32(0)
    _raise(load_library().ssm_scan_plan(ctypes.byref(a), ctypes.byref(cl), ctypes.byref(k),
                                        ctypes.byref(n)), "ssm_scan_plan")
    return int(cl.value), int(k.value), int(n.value)


def scan_launches_per_call(batch, seqlen, dim, dstate, io_dtype=torch.bfloat16,
                           time_chunk: int = 0) -> int:
    return scan_plan(batch, seqlen, dim, dstate, io_dtype, time_chunk)[2]


def scan_fwd(x: torch.Tensor, delta: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
             C: torch.Tensor, D: Optional[torch.Tensor] = None, z: Optional[torch.Tensor] = None,
             delta_bias: Optional[torch.Tensor] = None, delta_softplus: bool = True,
             h0: Optional[torch.Tensor] = None, return_final_state: bool = True,
             y: Optional[torch.Tensor] = None, h_final: Optional[torch.Tensor] = None,
             workspace: Optional[torch.Tensor] = None, time_chunk: int = 0,
             stream=None, discretization: str = "euler",
             checkpoints=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Selective scan.  x, delta, z: (B, L, D); A: (D, N) fp32; B, C: (B, L, N);
    D, delta_bias: (D,) fp32; h0: (B, D, N) fp32; discretization "euler" (B̄ = dl B)
    or "zoh" (zero-order hold).  Returns (y, h_final).
    checkpoints: an fp32 tensor of scan_ckpt_shape(...) (or True, to allocate one) that
    also receives the states scan_bwd rebuilds the sequence from (ssm_scan_fwd_ckpt);
    the return value is then (y, h_final, checkpoints)."""
    lib = load_library()
    nb, L, Dm = x.shape
    N = A.shape[1]
    if y is None:
        y = torch.empty_like(x)
    if h_final is None and return_final_state:
        h_final = torch.empty((nb, Dm, N), dtype=torch.float32, device=x.device)
    args = _scan_args(x, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, y, h_final,
                      time_chunk, discretization)
    need = ctypes.c_size_t(0)
    _raise(lib.ssm_scan_workspace_size(ctypes.byref(args), ctypes.byref(need)),
           "ssm_scan_workspace_size")
    ws, nbytes = _workspace(int(need.value), x.device, workspace)
    args.workspace, args.workspace_bytes = _ptr(ws), nbytes
    if checkpoints is None or checkpoints is False:
        _launch(lib.ssm_scan_fwd, args, stream, x.device, "ssm_scan_fwd")
        return y, h_final
    shape = scan_ckpt_shape(nb, L, Dm, N)
    if checkpoints is True:
        checkpoints = torch.empty(shape, dtype=torch.float32, device=x.device)
    _check(checkpoints, "checkpoints", shape, torch.float32, x.device)
    fn = lib.ssm_scan_fwd_ckpt
    with torch.cuda.device(x.device):
        rc = fn(ctypes.byref(args), _ptr(checkpoints), checkpoints.numel() * 4,
                _stream(stream, x.device))
    _raise(rc, "ssm_scan_fwd_ckpt")
    return y, h_final, checkpoints


def scan_ckpt_steps(dstate: int) -> int:
    """Steps between the state checkpoints the backward pass rebuilds the sequence from."""
    args = ScanArgs()
    args.batch, args.seqlen, args.dim, args.dstate = 1, 1, 1, dstate
    steps, nbytes = ctypes.c_int64(0), ctypes.c_size_t(0)
    _raise(load_library().ssm_scan_ckpt_size(ctypes.byref(args), ctypes.byref(steps),
                                             ctypes.byref(nbytes)), "ssm_scan_ckpt_size")
    return int(steps.value)


def scan_ckpt_shape(batch: int, seqlen: int, dim: int, dstate: int) -> Tuple[int, int, int, int]:
    """(B, ceil(L / T), D, N): the fp32 checkpoint tensor of ssm_scan_fwd_ckpt."""
    T = scan_ckpt_steps(dstate)
    return (batch, (seqlen + T - 1) // T, dim, dstate)


def scan_bwd(dy: torch.Tensor, x: torch.Tensor, delta: torch.Tensor, A: torch.Tensor,
             B: torch.Tensor, C: torch.Tensor, D: Optional[torch.Tensor] = None,
             z: Optional[torch.Tensor] = None, delta_bias: Optional[torch.Tensor] = None,
             delta_softplus: bool = True, h0: Optional[torch.Tensor] = None,
             dh_final: Optional[torch.Tensor] = None, discretization: str = "euler",
             workspace: Optional[torch.Tensor] = None, stream=None,
             checkpoints: Optional[torch.Tensor] = None) -> dict:
    """Gradients of scan_fwd with the same inputs, for the gradient dy (B, L, D) of y and
    dh_final (B, D, N) fp32 of the final state (zero when None).  The hidden states
    are recomputed, not stored: from checkpoints the kernel computes itself, or from
    `checkpoints` written by scan_fwd(..., checkpoints=...) on the same inputs
    (ssm_scan_bwd_ckpt).  Returns a dict: dx, ddelta (B, L, D) in x's dtype;
    dz (when z is given); dA (D, N), dB, dC (B, L, N), dD, ddelta_bias (D,), dh0
    (B, D, N), all fp32."""
    lib = load_library()
    nb, L, Dm = x.shape
    N = A.shape[1]
    dev, io = x.device, x.dtype
    _scan_args(x, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, None, None, 0,
               discretization)                                  # shape and dtype checks
    _check(dy, "dy", (nb, L, Dm), io, dev)
    _check(dh_final, "dh_final", (nb, Dm, N), torch.float32, dev)
    f32 = dict(dtype=torch.float32, device=dev)
    g = dict(dx=torch.empty_like(x), ddelta=torch.empty_like(x),
             dz=torch.empty_like(x) if z is not None else None,
             dA=torch.empty((Dm, N), **f32), dB=torch.empty((nb, L, N), **f32),
             dC=torch.empty((nb, L, N), **f32), dD=torch.empty((Dm,), **f32),
             ddelta_bias=torch.empty((Dm,), **f32), dh0=torch.empty((nb, Dm, N), **f32))
    args = ScanBwdArgs(nb, L, Dm, N, _io_code(x), int(bool(delta_softplus)), _disc(discretization),
                       0, _ptr(x), _ptr(delta), _ptr(B), _ptr(C), _ptr(z), _ptr(A), _ptr(D),
                       _ptr(delta_bias), _ptr(h0), _ptr(dy), _ptr(dh_final), _ptr(g["dx"]),
                       _ptr(g["ddelta"]), _ptr(g["dz"]), _ptr(g["dA"]), _ptr(g["dB"]),
                       _ptr(g["dC"]), _ptr(g["dD"]), _ptr(g["ddelta_bias"]), _ptr(g["dh0"]),
                       None, 0)
    if checkpoints is not None:
        _check(checkpoints, "checkpoints", scan_ckpt_shape(nb, L, Dm, N), torch.float32, dev)
        # the workspace holds only the status word
        ws, nbytes = _workspace(256, dev, workspace)
        args.workspace, args.workspace_bytes = _ptr(ws), nbytes
        with torch.cuda.device(dev):
            rc = lib.ssm_scan_bwd_ckpt(ctypes.byref(args), _ptr(checkpoints),
                                       checkpoints.numel() * 4, _stream(stream, dev))
        _raise(rc, "ssm_scan_bwd_ckpt")
    else:
        need = ctypes.c_size_t(0)
        _raise(lib.ssm_scan_bwd_workspace_size(ctypes.byref(args), ctypes.byref(need)),
               "ssm_scan_bwd_workspace_size")
        ws, nbytes = _workspace(int(need.value), dev, workspace)
        args.workspace, args.workspace_bytes = _ptr(ws), nbytes
        _launch(lib.ssm_scan_bwd, args, stream, x.device, "ssm_scan_bwd")
    if z is None:
        del g["dz"]
    return g


def scan_bwd_workspace_size(batch: int, seqlen: int, dim: int, dstate: int,
                            io_dtype=torch.bfloat16) -> int:
    args = ScanBwdArgs(batch, seqlen, dim, dstate, 1 if io_dtype == torch.bfloat16 else 0, 1, 0, 0)
    out = ctypes.c_size_t(0)
    _raise(load_library().ssm_scan_bwd_workspace_size(ctypes.byref(args), ctypes.byref(out)),
           "ssm_scan_bwd_workspace_size")
    return int(out.value)


NOALLOC_SCRATCH_BYTES = 4 << 20


def scan_fwd_noalloc(x, delta, A, B, C, D=None, z=None, delta_bias=None,
                     delta_softplus: bool = True, h0=None, y=None, h_final=None,
                     time_chunk: int = 0, stream=None, discretization: str = "euler"):
    """ssm_scan_fwd_noalloc: the scan with the library's fixed scratch buffer instead
    of a workspace, for callers that must not allocate device memory per call.
    Outputs y and h_final must be passed in (nothing is allocated here either)."""
    if y is None:
        raise ValueError("scan_fwd_noalloc allocates nothing: pass y (and h_final if wanted)")
    args = _scan_args(x, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, y, h_final,
                      time_chunk, discretization)
    _launch(load_library().ssm_scan_fwd_noalloc, args, stream, x.device, "ssm_scan_fwd_noalloc")
    return y, h_final


# ---------------------------------------------------------------- SSD
def _ssd_args(x, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, y, h_final,
              chunk_size) -> SSDArgs:
    nb, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    dev, io = x.device, x.dtype
    _io_code(x)
    _check(delta, "delta", (nb, L, H), io, dev)
    _check(A, "A", (H,), torch.float32, dev)
    _check(B, "B", (nb, L, G, N), io, dev)
    _check(C, "C", (nb, L, G, N), io, dev)
    _check(D, "D", (H,), torch.float32, dev)
    _check(z, "z", (nb, L, H, P), io, dev)
    _check(delta_bias, "delta_bias", (H,), torch.float32, dev)
    _check(h0, "h0", (nb, H, P, N), torch.float32, dev)
    _check(y, "y", (nb, L, H, P), io, dev)
    _check(h_final, "h_final", (nb, H, P, N), torch.float32, dev)
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    return SSDArgs(nb, L, H, P, G, N, int(chunk_size), _io_code(x), int(bool(delta_softplus)),
                   _ptr(x), _ptr(delta), _ptr(B), _ptr(C), _ptr(z), _ptr(A), _ptr(D),
                   _ptr(delta_bias), _ptr(h0), _ptr(y), _ptr(h_final), None, 0)


def ssd_workspace_size(x, delta, A, B, C, chunk_size: int = 256) -> int:
    args = _ssd_args(x, delta, A, B, C, None, None, None, True, None, None, None, chunk_size)
    out = ctypes.c_size_t(0)
    _raise(load_library().ssm_ssd_workspace_size(ctypes.byref(args), ctypes.byref(out)),
           "ssm_ssd_workspace_size")
    return int(out.value)


def ssd_uses_tensor_cores(x, delta, A, B, C, z=None, y=None, chunk_size: int = 0) -> bool:
    """Whether ssd_chunk_fwd takes the tcgen05 chunked kernel for these tensors."""
    if y is None:
        y = torch.empty_like(x)
    args = _ssd_args(x, delta, A, B, C, None, z, None, True, None, y, None, chunk_size)
    out = ctypes.c_int32(0)
    _raise(load_library().ssm_ssd_plan(ctypes.byref(args), ctypes.byref(out)), "ssm_ssd_plan")
    return bool(out.value)


def ssd_chunk_fwd(x: torch.Tensor, delta: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                  C: torch.Tensor, D: Optional[torch.Tensor] = None,
                  z: Optional[torch.Tensor] = None, delta_bias: Optional[torch.Tensor] = None,
                  delta_softplus: bool = True, h0: Optional[torch.Tensor] = None,
                  chunk_size: int = 256, return_final_state: bool = True,
                  y: Optional[torch.Tensor] = None, h_final: Optional[torch.Tensor] = None,
                  workspace: Optional[torch.Tensor] = None,
                  stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Multi-head scalar-A SSM (Mamba-2 SSD).  x, z: (B, L, H, P); delta: (B, L, H);
    A, D, delta_bias: (H,) fp32; B, C: (B, L, G, N); h0: (B, H, P, N) fp32."""
    lib = load_library()
    nb, L, H, P = x.shape
    N = B.shape[3]
    if y is None:
        y = torch.empty_like(x)
    if h_final is None and return_final_state:
        h_final = torch.empty((nb, H, P, N), dtype=torch.float32, device=x.device)
    args = _ssd_args(x, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, y, h_final,
                     chunk_size)
    need = ctypes.c_size_t(0)
    _raise(lib.ssm_ssd_workspace_size(ctypes.byref(args), ctypes.byref(need)),
           "ssm_ssd_workspace_size")
    ws, nbytes = _workspace(int(need.value), x.device, workspace)
    args.workspace, args.workspace_bytes = _ptr(ws), nbytes
    _launch(lib.ssm_ssd_chunk_fwd, args, stream, x.device, "ssm_ssd_chunk_fwd")
    return y, h_final


def read_device_status(workspace: torch.Tensor, stream=None) -> int:
    out = ctypes.c_int(0)
    with torch.cuda.device(workspace.device):
        _raise(load_library().ssm_read_device_status(_ptr(workspace),
                                                     _stream(stream, workspace.device),
                                                     ctypes.byref(out)),
               "ssm_read_device_status")
    return int(out.value)


# ---------------------------------------------------------------- decode
def step_decode(state: torch.Tensor, x: torch.Tensor, delta: torch.Tensor, A: torch.Tensor,
                B: torch.Tensor, C: torch.Tensor, D: Optional[torch.Tensor] = None,
                z: Optional[torch.Tensor] = None, delta_bias: Optional[torch.Tensor] = None,
                delta_softplus: bool = True, y: Optional[torch.Tensor] = None,
                stream=None, discretization: str = "euler",
                workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One recurrent step; ``state`` (B, D, N) fp32 is updated in place.
    x, delta, z: (B, D); B, C: (B, N); A: (D, N) fp32; D, delta_bias: (D,) fp32.
    workspace: optional 256-byte uint8 tensor that receives the device status word
    (read it with read_device_status)."""
    lib = load_library()
    nb, Dm, N = state.shape
    dev, io = x.device, x.dtype
    _io_code(x)
    _check(state, "state", (nb, Dm, N), torch.float32, dev)
    _check(x, "x", (nb, Dm), io, dev)
    _check(delta, "delta", (nb, Dm), io, dev)
    _check(A, "A", (Dm, N), torch.float32, dev)
    _check(B, "B", (nb, N), io, dev)
    _check(C, "C", (nb, N), io, dev)
    _check(D, "D", (Dm,), torch.float32, dev)
    _check(z, "z", (nb, Dm), io, dev)
    _check(delta_bias, "delta_bias", (Dm,), torch.float32, dev)
    if y is None:
        y = torch.empty_like(x)
    _check(y, "y", (nb, Dm), io, dev)
    args = DecodeArgs(nb, Dm, N, _io_code(x), int(bool(delta_softplus)), _ptr(state), _ptr(x),
                      _ptr(delta), _ptr(B), _ptr(C), _ptr(z), _ptr(A), _ptr(D),
                      _ptr(delta_bias), _ptr(y))
    args.discretization = _disc(discretization)
    if workspace is not None:
        args.workspace = _ptr(workspace)
        args.workspace_bytes = workspace.numel() * workspace.element_size()
    _launch(lib.ssm_step_decode, args, stream, x.device, "ssm_step_decode")
    return y


# ---------------------------------------------------------------- multi-head decode
def ssd_step_decode(state: torch.Tensor, x: torch.Tensor, delta: torch.Tensor, A: torch.Tensor,
                    B: torch.Tensor, C: torch.Tensor, D: Optional[torch.Tensor] = None,
                    z: Optional[torch.Tensor] = None, delta_bias: Optional[torch.Tensor] = None,
                    delta_softplus: bool = True, y: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
    """One token of the multi-head scalar-A recurrence; ``state`` (B, H, P, N) fp32 is
    updated in place.  x, z: (B, H, P); delta: (B, H); B, C: (B, G, N); A, D,
    delta_bias: (H,) fp32."""
    lib = load_library()
    nb, H, P, N = state.shape
    G = B.shape[1]
    dev, io = x.device, x.dtype
    _io_code(x)
    _check(state, "state", (nb, H, P, N), torch.float32, dev)
    _check(x, "x", (nb, H, P), io, dev)
    _check(delta, "delta", (nb, H), io, dev)
    _check(A, "A", (H,), torch.float32, dev)
    _check(B, "B", (nb, G, N), io, dev)
    _check(C, "C", (nb, G, N), io, dev)
    _check(D, "D", (H,), torch.float32, dev)
    _check(z, "z", (nb, H, P), io, dev)
    _check(delta_bias, "delta_bias", (H,), torch.float32, dev)
    if y is None:
        y = torch.empty_like(x)
    _check(y, "y", (nb, H, P), io, dev)
    args = SSDDecodeArgs(nb, H, P, G, N, _io_code(x), int(bool(delta_softplus)), _ptr(state),
                         _ptr(x), _ptr(delta), _ptr(B), _ptr(C), _ptr(z), _ptr(A), _ptr(D),
                         _ptr(delta_bias), _ptr(y))
    _launch(lib.ssm_ssd_step_decode, args, stream, x.device, "ssm_ssd_step_decode")
    return y


# ---------------------------------------------------------------- causal conv1d + SiLU
def conv1d(x: torch.Tensor, weight: torch.Tensor, bias: Optional[torch.Tensor] = None,
           x_prev: Optional[torch.Tensor] = None, silu: bool = True,
           out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
           stream=None) -> torch.Tensor:
    """Causal depthwise convolution along time, then SiLU.  x: (B, L, D); weight: (D, K)
    fp32; bias: (D,) fp32; x_prev: (B, K-1, D), the inputs just before x (zeros when
    None); workspace: optional 256-byte device status word (read_device_status).
    Returns (B, L, D) in x's dtype."""
    lib = load_library()
    nb, L, Dm = x.shape
    K = weight.shape[1]
    dev, io = x.device, x.dtype
    _io_code(x)
    _check(x, "x", (nb, L, Dm), io, dev)
    _check(weight, "weight", (Dm, K), torch.float32, dev)
    _check(bias, "bias", (Dm,), torch.float32, dev)
    _check(x_prev, "x_prev", (nb, K - 1, Dm), io, dev)
    if out is None:
        out = torch.empty_like(x)
    _check(out, "out", (nb, L, Dm), io, dev)
    args = Conv1dArgs(nb, L, Dm, K, _io_code(x), int(bool(silu)), _ptr(x), _ptr(x_prev),
                      _ptr(weight), _ptr(bias), _ptr(out), _ptr(workspace),
                      0 if workspace is None else workspace.numel() * workspace.element_size())
    _launch(lib.ssm_conv1d, args, stream, x.device, "ssm_conv1d")
    return out


# ---------------------------------------------------------------- autograd
class SelectiveScanFn(torch.autograd.Function):
    """scan_fwd with its gradients from scan_bwd.  The hidden states are recomputed in
    the backward pass from the inputs; with checkpoint_states the forward pass also keeps
    the state every few steps (scan_fwd(..., checkpoints=True)) and the backward pass
    starts from those instead of rebuilding them."""

    @staticmethod
    def forward(ctx, x, delta, A, B, C, D, z, delta_bias, h0, delta_softplus, discretization,
                checkpoint_states=False):
        out = scan_fwd(x, delta, A, B, C, D=D, z=z, delta_bias=delta_bias,
                       delta_softplus=delta_softplus, h0=h0, discretization=discretization,
                       checkpoints=True if checkpoint_states else None)
        y, h_final = out[0], out[1]
        ck = out[2] if checkpoint_states else None
        ctx.save_for_backward(x, delta, A, B, C, D, z, delta_bias, h0, ck)
        ctx.delta_softplus, ctx.discretization = delta_softplus, discretization
        return y, h_final

    @staticmethod
    def backward(ctx, dy, dh_final):
        x, delta, A, B, C, D, z, delta_bias, h0, ck = ctx.saved_tensors
        need = ctx.needs_input_grad
        if not any(need[:9]):
            return (None,) * 12
        g = scan_bwd(dy.contiguous().to(x.dtype), x, delta, A, B, C, D=D, z=z,
                     delta_bias=delta_bias, delta_softplus=ctx.delta_softplus, h0=h0,
                     dh_final=None if dh_final is None else dh_final.contiguous().float(),
                     discretization=ctx.discretization, checkpoints=ck)

        def out(i, grad, like):
            # only the inputs autograd asked for get a gradient
            return grad.to(like.dtype) if (need[i] and like is not None) else None
        return (out(0, g["dx"], x), out(1, g["ddelta"], delta), out(2, g["dA"], A),
                out(3, g["dB"], B), out(4, g["dC"], C), out(5, g["dD"], D),
                out(6, g.get("dz"), z), out(7, g["ddelta_bias"], delta_bias),
                out(8, g["dh0"], h0), None, None, None)


def selective_scan(x: torch.Tensor, delta: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                   C: torch.Tensor, D: Optional[torch.Tensor] = None,
                   z: Optional[torch.Tensor] = None, delta_bias: Optional[torch.Tensor] = None,
                   h0: Optional[torch.Tensor] = None, delta_softplus: bool = True,
                   discretization: str = "euler",
                   checkpoint_states: bool = False) -> Tuple[torch.Tensor, torch.Tensor]:
    """Differentiable selective scan: (y, h_final) = scan_fwd(...), with every input's
    gradient from the library's backward kernel.  Shapes and dtypes as scan_fwd; the
    gradients of B and C (fp32 sums over channels) are returned in B's and C's dtype.
    checkpoint_states keeps scan_ckpt_shape(...) fp32 of states from the forward to the
    backward pass (about D N / T floats per token, T = scan_ckpt_steps(N)) and spares
    the backward its own forward pass over the sequence."""
    return SelectiveScanFn.apply(x, delta, A, B, C, D, z, delta_bias, h0, delta_softplus,
                                 discretization, checkpoint_states)
