"""Helpers shared by the GPU parity tests: move seeded problems to the device,
run the library through its C ABI binding, and compare with the fp64 oracle.

A comparison (``Parity``) applies three bounds, each written here:

1. Whole tensor: rel-L2 = ||got - ref|| / ||ref|| <= 1e-5 for fp32 I/O and <= 3e-3 for
   bf16 I/O.  For bf16 the bound is the larger of 3e-3 and the error that rounding the
   oracle's own values to bf16 (round to nearest even) has: where that floor exceeds
   3e-3 (tiny tensors dominated by a few values) no bf16 result can meet 3e-3.
2. Per row: the rel-L2 of every row (a channel over time, a (batch, head) chain, ...)
   <= 1e-4 (fp32) or max(3e-3, 2 x the row's own bf16 rounding floor).  A correct bf16
   row errs by its rounding (about the floor) plus the fp32 arithmetic before it (far
   smaller), so twice the floor bounds it; a wrong carry into one channel or one wrong
   hand-over in a long chain moves one row by far more while barely moving bound 1.
3. Per element: |got - ref| <= rtol |ref| + atol rms(ref), rtol = 2^-8 (half a bf16
   ulp is at most 2^-8 of the value) or 1e-5 (fp32), atol = 1e-2 (bf16) or 1e-4 (fp32)
   times the root mean square of the reference.  The absolute part covers cancellation
   in y = C.h + D x and the gate's hardware tanh (absolute error about 2.4e-4 |z| on
   the sigmoid); a wrong tile or a stale value errs by the size of the values
   themselves, a hundred times more.

The SSD tensor-core kernel rounds three operands to bf16 before its fp32-accumulated
products: the masked matrix M, the carried state S_in and the decay-weighted inputs Xw
(each rounding at most 2^-9 of the value).  For a sum of products whose operands carry
relative error e, the error is at most e times the sum of the absolute values of the
terms, so its outputs get a per-element allowance of 3 x 2^-9 x |terms| (and 2 x 2^-9
for the final state), where |terms| is the oracle run on the absolute values of the
inputs (every product and decay then adds up without cancellation).  Bounds 2 and 3
add that allowance; bound 1 stays the plain 3e-3.

Pieces of a large result can be added one at a time (a channel block, a batch row, a
decode step), so full-size workloads are compared on every output without holding the
whole float64 tensor.  With SSM_PARITY_REPORT set to a file path, every comparison
appends one JSON line with its figures there, including the diagnostic error against
the oracle rounded to bf16.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle
import selective_state_space_132_b300 as ssm
from selective_state_space_132_b300 import workloads as W

# tolerances (relative L2 over the whole tensor): fp32 I/O 1e-5, bf16 I/O 3e-3
TOL = {"f32": 1e-5, "bf16": 3e-3}
ROW_TOL = {"f32": 1e-4, "bf16": 3e-3}
RTOL = {"f32": 1e-5, "bf16": 2.0 ** -8}
ATOL = {"f32": 1e-4, "bf16": 1e-2}


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


def _bf16(a):
    """Values rounded to bf16 (round to nearest even), as float64.  Values beyond the
    float32 range stay as they are (they only occur in a failing comparison)."""
    a = np.asarray(a, np.float64)
    f = a.astype(np.float32)
    ok = np.isfinite(f)
    out = a.copy()
    out[ok] = W.round_bf16(np.where(ok, f, 0.0).astype(np.float32))[ok]
    return out


def bf16_rounding_floor(ref) -> float:
    """rel-L2 between the oracle's values and the same values rounded to bf16 (RNE):
    the error any correctly rounded bf16 output has."""
    ref = np.asarray(ref, np.float64)
    return oracle.rel_l2(_bf16(ref), ref)


class Parity:
    """Accumulates the comparison of a GPU result with the oracle over one or more
    pieces, then checks the three bounds of this module.  Each piece is given as a
    2-D pair (rows, elements) with the global rows it holds: a slice, an index array,
    or None for all rows in order."""

    def __init__(self, io: str, what: str, nrows: int):
        self.io, self.what, self.nrows = io, what, nrows
        self.num = np.zeros(nrows)       # per row: sum (got - ref)^2
        self.den = np.zeros(nrows)       # per row: sum ref^2
        self.flo = np.zeros(nrows)       # per row: sum (bf16(ref) - ref)^2
        self.cnt = np.zeros(nrows)       # per row: elements
        self.alw = np.zeros(nrows)       # per row: sum of squared element allowances
        self.diag = 0.0                  # sum (got - bf16(ref))^2
        self.count = 0
        self.excess = -np.inf            # max over elements of |got - ref| - rtol |ref|
        self.excess_at = None
        self.finite = True

    def add(self, got, ref, rows=None, allow=None):
        """allow: optional per-element extra absolute tolerance (same shape)."""
        got = np.asarray(got, np.float64)
        ref = np.asarray(ref, np.float64)
        assert got.shape == ref.shape and got.ndim == 2, (got.shape, ref.shape)
        allow = None if allow is None else np.asarray(allow, np.float64)
        assert allow is None or allow.shape == got.shape
        if rows is None:
            rows = slice(0, got.shape[0])
        if isinstance(rows, slice):
            def acc(buf, v):
                buf[rows] += v
            first = rows.start or 0
            row_id = lambda i: first + i  # noqa: E731
        else:
            rows = np.asarray(rows)

            def acc(buf, v):
                np.add.at(buf, rows, v)
            row_id = lambda i: int(rows[i])  # noqa: E731
        self.finite &= bool(np.all(np.isfinite(got)))
        diff = got - ref
        acc(self.num, np.sum(diff * diff, axis=1))
        acc(self.den, np.sum(ref * ref, axis=1))
        acc(self.cnt, np.full(got.shape[0], float(got.shape[1])))
        if allow is not None:
            acc(self.alw, np.sum(allow * allow, axis=1))
        if self.io == "bf16":
            rb = _bf16(ref)
            acc(self.flo, np.sum((rb - ref) ** 2, axis=1))
            self.diag += float(np.sum((got - rb) ** 2))
        self.count += got.size
        if got.size:
            ex = np.abs(diff) - RTOL[self.io] * np.abs(ref)
            if allow is not None:
                ex = ex - allow
            k = int(np.argmax(ex))
            if ex.flat[k] > self.excess:
                self.excess = float(ex.flat[k])
                self.excess_at = (row_id(k // got.shape[1]), k % got.shape[1])
        return self

    def check(self):
        io = self.io
        num, den = float(self.num.sum()), float(self.den.sum())
        err = 0.0 if num == 0.0 else (np.sqrt(num / den) if den > 0 else np.inf)
        floor = np.sqrt(float(self.flo.sum()) / den) if den > 0 else 0.0
        tol = max(TOL[io], floor) if io == "bf16" else TOL[io]
        rms = np.sqrt(den / self.count) if self.count else 0.0
        # a row whose values are a thousand times below the tensor's rms (or zero) is
        # measured against that level instead, and left to the element bound
        den_row = np.maximum(self.den, (1e-3 * rms) ** 2 * self.cnt)
        with np.errstate(divide="ignore", invalid="ignore"):
            row_err = np.where(den_row > 0, np.sqrt(self.num / den_row),
                               np.where(self.num > 0, np.inf, 0.0))
            row_floor = np.where(den_row > 0, np.sqrt(self.flo / den_row), 0.0)
        row_tol = (np.maximum(ROW_TOL[io], 2.0 * row_floor) if io == "bf16"
                   else np.full(self.nrows, ROW_TOL[io]))
        with np.errstate(divide="ignore", invalid="ignore"):
            row_tol = row_tol + np.where(den_row > 0, np.sqrt(self.alw / den_row), 0.0)
        # a rel-L2 over fewer than 8 values is a per-element ratio; the element bound
        # covers those rows (a one-value row of a sum with cancellation is no signal)
        row_err = np.where(self.cnt >= 8, row_err, 0.0)
        worst = int(np.argmax(row_err / row_tol)) if self.nrows else 0
        atol = ATOL[io] * rms
        report = dict(what=self.what, io=io, elements=self.count, rel_l2=err, tol=tol,
                      bf16_floor=floor if io == "bf16" else None,
                      rel_l2_vs_bf16_oracle=(np.sqrt(self.diag / den) if io == "bf16" and den > 0
                                             else None),
                      rows=self.nrows, worst_row=worst,
                      worst_row_rel_l2=float(row_err[worst]) if self.nrows else 0.0,
                      worst_row_tol=float(row_tol[worst]) if self.nrows else 0.0,
                      max_elem_excess_over_atol=(self.excess / atol if atol > 0 else
                                                 (0.0 if self.excess <= 0 else np.inf)),
                      worst_elem=self.excess_at)
        path = os.environ.get("SSM_PARITY_REPORT")
        if path:
            with open(path, "a") as f:
                f.write(json.dumps(report, default=float) + "\n")
        assert self.finite, f"{self.what}: non-finite values"
        assert err <= tol, f"{self.what}: rel-L2 {err:.3e} > {tol:.1e}"
        assert self.nrows == 0 or row_err[worst] <= row_tol[worst], (
            f"{self.what}: row {worst} rel-L2 {row_err[worst]:.3e} > {row_tol[worst]:.1e}")
        assert self.count == 0 or self.excess <= atol, (
            f"{self.what}: element {self.excess_at} off by {self.excess:.3e} beyond "
            f"rtol |ref| (atol {atol:.3e})")
        return report


def assert_close(got, ref, io, what, row_axes=None, allow=None):
    """Compare a whole result with the oracle under the three bounds.  Rows are the
    index tuples over ``row_axes`` (default: every axis but the last), elements the
    rest.  Returns the whole-tensor rel-L2."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if got.ndim == 0:
        got, ref = got.reshape(1, 1), ref.reshape(1, 1)
    if row_axes is None:
        row_axes = tuple(range(got.ndim - 1)) if got.ndim > 1 else ()
    rest = tuple(a for a in range(got.ndim) if a not in row_axes)
    order = tuple(row_axes) + rest
    nrows = int(np.prod([got.shape[a] for a in row_axes])) if row_axes else 1
    g2 = np.transpose(got, order).reshape(nrows, -1)
    r2 = np.transpose(ref, order).reshape(nrows, -1)
    a2 = None
    if allow is not None:
        a2 = np.transpose(np.broadcast_to(np.asarray(allow, np.float64), got.shape),
                          order).reshape(nrows, -1)
    return Parity(io, what, nrows).add(g2, r2, allow=a2).check()["rel_l2"]


def ssd_tc_allowance(p, batch=None):
    """Per-element allowances (y, h_final) of the SSD tensor-core kernel's bf16
    operands for problem p (optionally one batch row): 3 x 2^-9 x |terms| for y and
    2 x 2^-9 x |terms| for the final state, |terms| from the oracle on |inputs|."""
    sl = slice(None) if batch is None else slice(batch, batch + 1)
    ab = lambda a: None if a is None else np.abs(a[sl])  # noqa: E731
    y_abs, h_abs = oracle.ssd(ab(p.x), p.delta[sl], p.A, ab(p.B), ab(p.C),
                              Dv=None if p.D is None else np.abs(p.D), z=None, bias=p.bias,
                              softplus=p.softplus, h0=ab(p.h0))
    if p.z is not None:
        z = p.z[sl].astype(np.float64)
        y_abs = y_abs * np.abs(z / (1.0 + np.exp(-z)))
    return 3.0 * 2.0 ** -9 * y_abs, 2.0 * 2.0 ** -9 * h_abs
