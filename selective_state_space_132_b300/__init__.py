"""B300-native selective state-space (S6) scan, SSD chunk form and decode step.

The compute lives in ``libssm.so`` (hand-written CUDA for sm_103a, C ABI in
``include/ssm.h``).  This module is a thin ctypes binding: it checks tensor
dtypes and shapes, allocates outputs and workspaces with PyTorch, and passes raw
device pointers and the current CUDA stream.  Every step of the computation runs
in the library's kernels; if the library is missing, the calls raise.

    y, h_final = scan_fwd(x, delta, A, B, C, D=..., z=..., delta_bias=...)
    y, h_final = ssd_chunk_fwd(x, delta, A, B, C, D=..., chunk_size=256)
    y          = step_decode(state, x, delta, A, B, C, D=..., z=...)  # state in place
    y          = ssd_step_decode(state, x, delta, A, B, C, D=...)      # state in place
    out        = conv1d(x, weight, bias)                               # causal conv + SiLU
    grads      = scan_bwd(dy, x, delta, A, B, C, D=..., z=...)         # recomputed states
    y, h_final = selective_scan(x, delta, A, B, C, D=..., z=...)      # autograd-ready
"""
from __future__ import annotations

from .binding import (SSMError, build_library, conv1d, library_path, load_library,
                      read_device_status, scan_bwd, scan_bwd_workspace_size, scan_ckpt_shape,
                      scan_ckpt_steps, scan_fwd, selective_scan,
                      scan_fwd_noalloc, scan_launches_per_call, scan_plan, scan_workspace_size,
                      ssd_chunk_fwd, ssd_step_decode, ssd_uses_tensor_cores, ssd_workspace_size,
                      step_decode, version)

__all__ = ["SSMError", "build_library", "conv1d", "library_path", "load_library",
           "read_device_status", "scan_bwd", "scan_bwd_workspace_size", "scan_ckpt_shape",
           "scan_ckpt_steps", "scan_fwd", "selective_scan",
           "scan_fwd_noalloc", "scan_launches_per_call", "scan_plan", "scan_workspace_size",
           "ssd_chunk_fwd", "ssd_step_decode", "ssd_uses_tensor_cores", "ssd_workspace_size",
           "step_decode", "version"]
