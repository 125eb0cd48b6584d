"""Seeded synthetic inputs for the scan, SSD and decode workloads.

This module is shared by the tests, the benchmark and the smoke check on BOTH
sides of every comparison (the CUDA library and the fp64 oracle), so it holds
no arithmetic of the method itself: only random draws, the parameter recipes
of the five reference workloads, and round-to-nearest-even to bf16.

Recipes (Mamba review on tildalice.io, sections "Selection Mechanism" and
"초기화 전략"; Mamba-2 page, sections "멀티-헤드 구조" and "학습"):
  * A[d, n] = -(n + 1)  (the S4D-real A = -exp(A_log), A_log = log(1..N));
  * raw step Δraw ~ N(0, 0.5^2) (0.5 read as the standard deviation);
  * Δ bias = inv_softplus(u) = log(expm1(u)), u ~ U[1e-3, 1e-1], per channel;
  * B, C ~ N(0, 1) with shape (batch, L, N): shared across channels;
  * x, z ~ N(0, 1); D ~ N(0, 1);
  * SSD: A_h = -U[1, 16] per head, Δraw per (t, head), one shared B/C group.

Draw order per problem, from ``numpy.random.Generator(PCG64(seed))``:
x, Δraw, bias-uniform, B, C, z, D, A (SSD only), initial state.  Values are
drawn in float32 (uniforms in float64) and rounded to bf16 (round to nearest
even) where the I/O dtype is bf16, so both sides see the same numbers.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, Optional

import numpy as np

# Reference workloads by index: the S6 scan in fp32 (tiny), the 130M-layer
# shape, the long-context DNA shape, the Mamba-2 SSD shape and decode.
SCAN_FP32_TINY = dict(kind="scan", batch=1, seqlen=64, dim=16, dstate=4, io="f32", gate=True)
SCAN_MAMBA130M = dict(kind="scan", batch=8, seqlen=2048, dim=1536, dstate=16, io="bf16",
                      gate=True)
SCAN_LONG_DNA = dict(kind="scan", batch=1, seqlen=131072, dim=2048, dstate=16, io="bf16",
                     gate=True)
SSD_MAMBA2 = dict(kind="ssd", batch=4, seqlen=8192, heads=80, headdim=64, ngroups=1,
                  dstate=128, chunk=256, io="bf16", gate=False)
DECODE_B256 = dict(kind="decode", batch=256, dim=5120, dstate=16, steps=1000, io="bf16",
                   gate=True)

CONFIGS = [SCAN_FP32_TINY, SCAN_MAMBA130M, SCAN_LONG_DNA, SSD_MAMBA2, DECODE_B256]
CONFIG_NAMES = ["scan_f32_B1_D16_L64_N4", "scan_bf16_B8_D1536_L2048_N16",
                "scan_bf16_B1_D2048_L131072_N16", "ssd_bf16_B4_L8192_H80_P64_N128_G1_Q256",
                "decode_bf16_B256_D5120_N16_x1000"]


def config_seed(index: int) -> int:
    return 1000 + index


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32
    arrays holding exactly-representable bf16 values.  Inputs must be finite."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def _io(a: np.ndarray, io: str) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    return round_bf16(a) if io == "bf16" else a


def _normal(rng, shape, std=1.0):
    out = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out


def _bias(rng, count):
    u = rng.uniform(1e-3, 1e-1, size=count)  # float64
    return np.log(np.expm1(u)).astype(np.float32)


@dataclass
class ScanProblem:
    batch: int
    seqlen: int
    dim: int
    dstate: int
    io: str
    x: np.ndarray
    delta: np.ndarray
    A: np.ndarray
    B: np.ndarray
    C: np.ndarray
    D: Optional[np.ndarray]
    z: Optional[np.ndarray]
    bias: Optional[np.ndarray]
    softplus: bool
    h0: Optional[np.ndarray]
    zoh: bool = False  # zero-order-hold input coefficient instead of dl

    @property
    def updates(self) -> int:
        return self.batch * self.seqlen * self.dim * self.dstate

    def oracle_args(self) -> Dict[str, object]:
        return dict(x=self.x, delta=self.delta, A=self.A, Bm=self.B, Cm=self.C, Dv=self.D,
                    z=self.z, bias=self.bias, softplus=self.softplus, h0=self.h0, zoh=self.zoh)


def scan_problem(batch: int, seqlen: int, dim: int, dstate: int, io: str = "bf16",
                 seed: int = 0, gate: bool = True, use_D: bool = True, use_bias: bool = True,
                 softplus: bool = True, h0: bool = False, A: str = "s4d") -> ScanProblem:
    """Synthetic S6 scan inputs with the reference recipe.  ``A`` is "s4d"
    (A[d,n] = -(n+1)) or "random" (A[d,n] = -U[0.5, 16], for tests that need
    an unstructured A; drawn after the initial state)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    shp = (batch, seqlen, dim)
    x = _io(_normal(rng, shp), io)
    delta = _io(_normal(rng, shp, 0.5), io)
    bias = _bias(rng, dim)
    Bm = _io(_normal(rng, (batch, seqlen, dstate)), io)
    Cm = _io(_normal(rng, (batch, seqlen, dstate)), io)
    z = _io(_normal(rng, shp), io)
    Dv = _normal(rng, (dim,))
    hz = _normal(rng, (batch, dim, dstate)) if h0 else None
    if A == "s4d":
        Am = -np.tile(np.arange(1, dstate + 1, dtype=np.float32), (dim, 1))
    elif A == "random":
        Am = -rng.uniform(0.5, 16.0, size=(dim, dstate)).astype(np.float32)
    else:
        raise ValueError(A)
    return ScanProblem(batch, seqlen, dim, dstate, io, x, delta, np.ascontiguousarray(Am),
                       Bm, Cm, Dv if use_D else None, z if gate else None,
                       bias if use_bias else None, softplus, hz)


@dataclass
class SSDProblem:
    batch: int
    seqlen: int
    heads: int
    headdim: int
    ngroups: int
    dstate: int
    chunk: int
    io: str
    x: np.ndarray
    delta: np.ndarray
    A: np.ndarray
    B: np.ndarray
    C: np.ndarray
    D: Optional[np.ndarray]
    z: Optional[np.ndarray]
    bias: Optional[np.ndarray]
    softplus: bool
    h0: Optional[np.ndarray]

    @property
    def updates(self) -> int:
        return self.batch * self.seqlen * self.heads * self.headdim * self.dstate

    def oracle_args(self) -> Dict[str, object]:
        return dict(x=self.x, delta=self.delta, A=self.A, Bm=self.B, Cm=self.C, Dv=self.D,
                    z=self.z, bias=self.bias, softplus=self.softplus, h0=self.h0)


def ssd_problem(batch: int, seqlen: int, heads: int, headdim: int, ngroups: int, dstate: int,
                chunk: int = 256, io: str = "bf16", seed: int = 0, gate: bool = False,
                use_D: bool = True, use_bias: bool = True, softplus: bool = True,
                h0: bool = False) -> SSDProblem:
    rng = np.random.Generator(np.random.PCG64(seed))
    x = _io(_normal(rng, (batch, seqlen, heads, headdim)), io)
    delta = _io(_normal(rng, (batch, seqlen, heads), 0.5), io)
    bias = _bias(rng, heads)
    Bm = _io(_normal(rng, (batch, seqlen, ngroups, dstate)), io)
    Cm = _io(_normal(rng, (batch, seqlen, ngroups, dstate)), io)
    z = _io(_normal(rng, (batch, seqlen, heads, headdim)), io) if gate else None
    Dv = _normal(rng, (heads,))
    A = (-rng.uniform(1.0, 16.0, size=heads)).astype(np.float32)
    hz = _normal(rng, (batch, heads, headdim, dstate)) if h0 else None
    return SSDProblem(batch, seqlen, heads, headdim, ngroups, dstate, chunk, io, x, delta, A,
                      Bm, Cm, Dv if use_D else None, z, bias if use_bias else None, softplus,
                      hz)


@dataclass
class DecodeProblem:
    batch: int
    dim: int
    dstate: int
    steps: int
    io: str
    seed: int
    state0: np.ndarray
    A: np.ndarray
    D: np.ndarray
    bias: np.ndarray
    softplus: bool = True
    gate: bool = True
    _cache: dict = field(default_factory=dict, repr=False)

    @property
    def updates_per_step(self) -> int:
        return self.batch * self.dim * self.dstate

    def tokens(self, step: int) -> Dict[str, np.ndarray]:
        """Token inputs of one step, from their own seed (seed, step), so any
        step can be regenerated on its own: x, delta, z (B,D); B, C (B,N)."""
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([self.seed, step])))
        shp = (self.batch, self.dim)
        x = _io(_normal(rng, shp), self.io)
        delta = _io(_normal(rng, shp, 0.5), self.io)
        Bm = _io(_normal(rng, (self.batch, self.dstate)), self.io)
        Cm = _io(_normal(rng, (self.batch, self.dstate)), self.io)
        z = _io(_normal(rng, shp), self.io)
        return dict(x=x, delta=delta, B=Bm, C=Cm, z=z if self.gate else None)


def decode_problem(batch: int, dim: int, dstate: int, steps: int, io: str = "bf16",
                   seed: int = 0, gate: bool = True) -> DecodeProblem:
    rng = np.random.Generator(np.random.PCG64(seed))
    bias = _bias(rng, dim)
    Dv = _normal(rng, (dim,))
    state0 = _normal(rng, (batch, dim, dstate))
    A = -np.tile(np.arange(1, dstate + 1, dtype=np.float32), (dim, 1))
    return DecodeProblem(batch, dim, dstate, steps, io, seed, state0, np.ascontiguousarray(A),
                         Dv, bias, True, gate)


def config_problem(index: int, **overrides):
    """The problem of a reference workload (optionally with smaller sizes
    given as overrides, e.g. ``seqlen=300``), seeded with 1000 + index."""
    cfg = dict(CONFIGS[index])
    cfg.update(overrides)
    seed = config_seed(index)
    kind = cfg.pop("kind")
    if kind == "scan":
        return scan_problem(cfg["batch"], cfg["seqlen"], cfg["dim"], cfg["dstate"], cfg["io"],
                            seed=seed, gate=cfg["gate"])
    if kind == "ssd":
        return ssd_problem(cfg["batch"], cfg["seqlen"], cfg["heads"], cfg["headdim"],
                           cfg["ngroups"], cfg["dstate"], cfg["chunk"], cfg["io"], seed=seed,
                           gate=cfg["gate"])
    if kind == "decode":
        return decode_problem(cfg["batch"], cfg["dim"], cfg["dstate"], cfg["steps"], cfg["io"],
                              seed=seed, gate=cfg["gate"])
    raise ValueError(kind)
