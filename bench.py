"""Benchmark of the selective-scan hot path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-extras] [--no-cpu]

One step = one forward pass of the S6 scan (softplus step, exp decay, state
recurrence, C readout, D skip, SiLU gate, and the carry between time chunks) over
one batch of the long-context workload (batch 1, d_inner 2048, L 131072, N 16, bf16
I/O, fp32 state: the largest scan configuration, 2.15 GB of inputs and outputs),
inputs already resident in HBM, L2 flushed before every step (a 256 MB write, then a
256 MB read so that the lines left in L2 are clean).  `--workload` selects the
130M-layer shape instead (batch 8, d_inner 1536, L 2048, N 16).  The metric is
state updates per second (B*L*D*N / time).  Rank 0 prints one JSON
line.  Under torchrun (N > 1) every rank runs its own independent batch (the
chains of the scan are independent: no data-path collective), so scaling is
weak and `value` is the updates of all ranks over the slowest rank's time.

`--impl reference` times the fp64 CPU oracle on the host cores instead, on a
bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from selective_state_space_132_b300 import workloads as W  # noqa: E402

HBM_FALLBACK_GBS = 6400.0
BF16_FALLBACK_TFLOPS = 1800.0
L2_FLUSH_BYTES = 256 << 20

# ncu DRAM traffic (bytes, read + written) of one scan call (the summary pass and the
# output pass when the plan splits the sequence), keyed by the sha256 prefix of the
# kernel's sources at the time of the capture and by workload; an entry whose key no
# longer matches the sources is ignored (traffic reported as null).
PROFILED_TRAFFIC = {
    "88390bb0d78ad0a6": {
        # scan_tma_lb_kernel (summary and output passes in one launch), mean of 5 calls:
        # 2,969.3 MB read + 525.3 MB written (the launch list of the bench line's command)
        "scan_bf16_B1_D2048_L131072_N16": 3494627532,
    },
}

# ncu occupancy of the binding resources of one scan launch, keyed like PROFILED_TRAFFIC:
# dispatch_busy = (warp instructions + MUFU and packed-fp32 warp instructions, which take
# two dispatch cycles) / (SM cycles x 4 sub-partitions x SMs); shared_wavefronts_of_peak =
# l1tex__data_pipe_lsu_wavefronts_mem_shared.avg.pct_of_peak_sustained_elapsed, one
# captured launch per workload
PROFILED_OCCUPANCY = {
    "88390bb0d78ad0a6": {
        "scan_bf16_B1_D2048_L131072_N16": {"dispatch_busy": 0.935, "shared_wavefronts_of_peak": 0.731,
                                           "issue_active": 0.668},
        "scan_bf16_B8_D1536_L2048_N16": {"dispatch_busy": 0.685, "shared_wavefronts_of_peak": 0.588,
                                         "issue_active": 0.501},
    },
}

WORKLOADS = {
    "scan_bf16_B8_D1536_L2048_N16": 1,
    "scan_bf16_B1_D2048_L131072_N16": 2,
    "ssd_bf16_B4_L8192_H80_P64_N128_G1_Q256": 3,
    "decode_bf16_B256_D5120_N16_x1000": 4,
}
SCAN_SOURCES = ["scan_tma.cu", "scan_fwd.cu", "common.cuh", "ptx.cuh", "tma_host.cuh"]


# ------------------------------------------------------------------ small helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(
            d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return HBM_FALLBACK_GBS, BF16_FALLBACK_TFLOPS, 1400.0, "fallback"


def kernel_source_hash(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "selective_state_space_132_b300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# Per-SM issue rates measured on B300 with a throughput microbenchmark (lanes per clock)
MUFU_EX2_PER_CLK = 29.7
FFMA_PER_CLK = 113.0


def scan_ceilings(p, algo_bytes, hbm_gbs, device):
    """Lower bounds on one scan step from each unit, at the SM clock of the part:
    MUFU (one exp per state update, plus softplus (2) and SiLU (1) per (t, d)), fp32
    (four operations per update: dl*A, dl*x*B, the state FMA, the C readout FMA) and
    HBM (the algorithmic bytes at the measured copy bandwidth)."""
    import torch
    props = torch.cuda.get_device_properties(device)
    sms = props.multi_processor_count
    clk = 2032e6                      # maximum SM clock of the part (Hz)
    units = p.updates
    rows = p.batch * p.seqlen * p.dim
    mufu = (units + 3 * rows) / (sms * MUFU_EX2_PER_CLK * clk)
    fp32 = 4 * units / (sms * FFMA_PER_CLK * clk)
    # instruction dispatch: per update at least 4 fp32 operations (one cycle per warp
    # instruction each) and one ex2 (two cycles), 32 lanes per SM sub-partition
    dispatch = 6 * units / 32 / (sms * 4 * clk)
    hbm = algo_bytes / (hbm_gbs * 1e9)
    return {"mufu_us": mufu * 1e6, "fp32_us": fp32 * 1e6, "dispatch_us": dispatch * 1e6,
            "hbm_us": hbm * 1e6, "sms": sms,
            "basis": "per-SM rates measured on B300: ex2 29.7 lanes/clk, FFMA 113/clk; "
                     "ex2 and fp32x2 take two dispatch cycles per warp instruction, FFMA one "
                     "(recurrence-core probe: 103.5 cycles per 16-state warp step at four "
                     "warps per sub-partition); 2032 MHz"}


# Instruction dispatch per state update: one ex2 (two dispatch cycles of a sub-partition
# per warp instruction, measured) and four fp32 operations (one each: dl*A, dl*x*B, the
# state FMA, the C readout), i.e. six lane slots of the 32 a sub-partition dispatches
# per cycle.
DISPATCH_SLOTS_PER_UPDATE = 6


def scan_dispatch_peak(device, clk=2032e6):
    """State updates/s at which instruction dispatch alone binds the scan: every SM
    sub-partition (four per SM) dispatches one warp instruction (32 lane slots) per
    cycle at the part's maximum SM clock."""
    import torch
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    return sms * 4 * 32 * clk / DISPATCH_SLOTS_PER_UPDATE


def scan_bytes(nb, L, D, N, e, gate=True, h0=False):
    """Algorithmic bytes of one scan: x, delta (, z), y in the I/O dtype, B and C,
    A, D and the bias in fp32, the final state (and h0) in fp32; no h_t."""
    tok = nb * L * D * e
    return (tok * (4 if gate else 3) + 2 * nb * L * N * e + D * N * 4 + 2 * D * 4
            + nb * D * N * 4 * (2 if h0 else 1))


def ssd_bytes(nb, L, H, P, G, N, e):
    return (2 * nb * L * H * P * e + nb * L * H * e + 2 * nb * L * G * N * e + 3 * H * 4
            + nb * H * P * N * 4)


def decode_bytes_per_step(nb, D, N, e):
    return 2 * nb * D * N * 4 + 4 * nb * D * e + 2 * nb * N * e + D * N * 4 + 2 * D * 4


def ssd_flops(nb, L, H, P, G, N, Q):
    """Dense tensor-core FLOPs of the chunked dual form: C B^T once per (b, chunk,
    group), the causal half of (L o C B^T) X, the chunk states and C S^T."""
    nc = (L + Q - 1) // Q
    per_chunk_head = Q * Q * P + 2 * Q * P * N + 2 * Q * P * N
    return nb * nc * (2 * Q * Q * N * G + H * per_chunk_head)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms in a thread."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        inside = [s for (t, s) in self.samples if t0 <= t <= t1]
        rows = inside or [s for (_, s) in self.samples]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [q.strip() for q in r.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "reasons": sorted(reasons), "samples": len(rows),
                "samples_in_timed_region": len(inside)}


# ------------------------------------------------------------------ distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    """Largest value over all ranks (the slowest rank's time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda") if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: float, seconds_max: float, world: int) -> float:
    """Whole-job throughput: every rank processed units_per_rank in at most seconds_max."""
    return units_per_rank * world / seconds_max


# ------------------------------------------------------------------ our arm
def bench_config(workload, p, world):
    """The `config` object of the JSON line, the same in both arms."""
    return {"workload": workload, "batch": p.batch, "seqlen": p.seqlen, "d_inner": p.dim,
            "d_state": p.dstate, "io": p.io, "state": "fp32", "gate": True,
            "l2": "flushed before every step (256 MB write, then 256 MB read); the inputs "
                  f"({scan_bytes(p.batch, p.seqlen, p.dim, p.dstate, 2 if p.io == 'bf16' else 4) / 1e9:.2f} GB) "
                  "also exceed the 126 MB L2",
            "parallelism": f"replicas x{world} (independent batches per GPU)"}


def _to_dev(device):
    import torch

    def t(a, dtype=torch.float32):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(
            device=device, dtype=dtype)
    return t


def time_scan(p, steps, warmup, flush, device, time_chunk=0):
    """Per-step device time of ssm_scan_fwd on resident inputs, L2 flushed before each
    step.  Returns (seconds per step, kernel launches per step, wall seconds, window)."""
    import torch
    import selective_state_space_132_b300 as ssm

    io = torch.bfloat16 if p.io == "bf16" else torch.float32
    t = _to_dev(device)
    x, dl, z, Bm, Cm = t(p.x, io), t(p.delta, io), t(p.z, io), t(p.B, io), t(p.C, io)
    A, Dv, bias = t(p.A), t(p.D), t(p.bias)
    y = torch.empty_like(x)
    hf = torch.empty((p.batch, p.dim, p.dstate), dtype=torch.float32, device=device)
    nbytes = ssm.scan_workspace_size(p.batch, p.seqlen, p.dim, p.dstate, io, time_chunk)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    launches = ssm.scan_launches_per_call(p.batch, p.seqlen, p.dim, p.dstate, io, time_chunk)
    stream = torch.cuda.current_stream()

    def step():
        ssm.scan_fwd(x, dl, A, Bm, Cm, D=Dv, z=z, delta_bias=bias, y=y, h_final=hf,
                     workspace=ws, time_chunk=time_chunk, stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    t0 = time.time()
    for i in range(steps):
        flush()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.time() - t0
    per = [a.elapsed_time(b) * 1e-3 for a, b in ev]
    return per, launches, wall, (t0, t0 + wall)


def e2e_scan(p, steps, device, slices=8):
    """Same metric through the public API with pinned host buffers: every step copies
    the inputs host->device, runs the scan and reads y and the final state back.

    The work is cut into `slices` pieces that flow through three streams: while piece
    i is scanned, piece i + 1 is copied in and piece i - 1 is copied out (PCIe carries
    both directions at once).  Pieces are batch rows when the batch has enough of them,
    else stretches of time (batch 1: contiguous), the state handed from one stretch to
    the next through h0 / h_final of the public call.  Events order the reuse of each
    piece's device buffers across steps.  Timed by the host clock, synchronised on
    both sides."""
    import torch
    import selective_state_space_132_b300 as ssm

    io = torch.bfloat16 if p.io == "bf16" else torch.float32

    def pin(a, dtype=io):
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dtype).pin_memory()
    hx, hdl, hz, hB, hC = pin(p.x), pin(p.delta), pin(p.z), pin(p.B), pin(p.C)
    A = torch.from_numpy(p.A).to(device)
    Dv = torch.from_numpy(p.D).to(device)
    bias = torch.from_numpy(p.bias).to(device)
    hy = torch.empty(hx.shape, dtype=io).pin_memory()
    hh = torch.empty((p.batch, p.dim, p.dstate), dtype=torch.float32).pin_memory()
    h2d = sum(a.numel() * a.element_size() for a in (hx, hdl, hz, hB, hC))
    d2h = hy.numel() * hy.element_size() + hh.numel() * hh.element_size()
    dx, ddl, dz, dB, dC = (torch.empty(a.shape, dtype=a.dtype, device=device)
                           for a in (hx, hdl, hz, hB, hC))
    dy = torch.empty(hx.shape, dtype=io, device=device)
    by_time = p.batch < slices and p.batch == 1
    n = max(1, min(slices, p.seqlen if by_time else p.batch))
    extent = p.seqlen if by_time else p.batch
    bounds = [(extent * i // n, extent * (i + 1) // n) for i in range(n)]
    # final state of each piece (time pieces chain through them); the last is the result
    dh = [torch.empty(hh.shape, dtype=torch.float32, device=device) for _ in bounds]

    def sl(a, b0, b1):
        return a[:, b0:b1] if by_time else a[b0:b1]
    s_in, s_run, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev_in = [torch.cuda.Event() for _ in bounds]
    ev_run = [torch.cuda.Event() for _ in bounds]
    ev_out = [torch.cuda.Event() for _ in bounds]
    cur = torch.cuda.current_stream(device)
    for i in range(n):           # nothing to wait for before the first step
        ev_run[i].record(cur)
        ev_out[i].record(cur)

    def step():
        for i, (b0, b1) in enumerate(bounds):
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_run[i])         # the previous scan of this piece is done
                for d_, h_ in ((dx, hx), (ddl, hdl), (dz, hz), (dB, hB), (dC, hC)):
                    sl(d_, b0, b1).copy_(sl(h_, b0, b1), non_blocking=True)
                ev_in[i].record(s_in)
            with torch.cuda.stream(s_run):
                s_run.wait_event(ev_in[i])
                s_run.wait_event(ev_out[i])        # the previous outputs left this piece
                if by_time:
                    ssm.scan_fwd(sl(dx, b0, b1), sl(ddl, b0, b1), A, sl(dB, b0, b1),
                                 sl(dC, b0, b1), D=Dv, z=sl(dz, b0, b1), delta_bias=bias,
                                 h0=dh[i - 1] if i > 0 else None, y=sl(dy, b0, b1),
                                 h_final=dh[i], stream=s_run)
                else:
                    ssm.scan_fwd(dx[b0:b1], ddl[b0:b1], A, dB[b0:b1], dC[b0:b1], D=Dv,
                                 z=dz[b0:b1], delta_bias=bias, y=dy[b0:b1],
                                 h_final=dh[0][b0:b1], stream=s_run)
                ev_run[i].record(s_run)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_run[i])
                sl(hy, b0, b1).copy_(sl(dy, b0, b1), non_blocking=True)
                if by_time and i == n - 1:
                    hh.copy_(dh[i], non_blocking=True)
                elif not by_time:
                    hh[b0:b1].copy_(dh[0][b0:b1], non_blocking=True)
                ev_out[i].record(s_out)

    for _ in range(2):
        step()
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize(device)
    kind = "time stretches (state chained through h0 / h_final)" if by_time else "batch slices"
    return (time.perf_counter() - t0) / steps, h2d, d2h, f"{n} {kind}"


class L2Flush:
    """Evicts the timed kernel's data from the 126 MB L2 before each timed call: a
    256 MB write, then a 256 MB read of a second buffer.  The read leaves clean lines in
    L2, so the timed kernel does not pay for writing the flush's dirty lines back."""

    def __init__(self, device):
        import torch
        n = L2_FLUSH_BYTES // 4
        self.w = torch.empty(n, dtype=torch.float32, device=device)
        self.r = torch.zeros(n, dtype=torch.float32, device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)

    def __call__(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)


def _gpu_lead():
    """A short device-side spin (about 0.5 ms) queued before the start event of a timed
    call that follows a synchronize: the host marshals the call and enqueues it while the
    device spins, so the measured window holds the call's work and no host gap."""
    import torch
    torch.cuda._sleep(1_000_000)


def _median_event_time(step, flush, iters):
    import torch
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    times = []
    for _ in range(iters):
        flush()
        _gpu_lead()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        step()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) * 1e-3)
    return float(np.median(times))


def time_ssd(p, iters, flush, device):
    import torch
    import selective_state_space_132_b300 as ssm
    io = torch.bfloat16
    t = _to_dev(device)
    x, dl, Bm, Cm = t(p.x, io), t(p.delta, io), t(p.B, io), t(p.C, io)
    A, Dv, bias = t(p.A), t(p.D), t(p.bias)
    y = torch.empty_like(x)
    hf = torch.empty((p.batch, p.heads, p.headdim, p.dstate), dtype=torch.float32,
                     device=device)
    ws = torch.empty(ssm.ssd_workspace_size(x, dl, A, Bm, Cm, p.chunk), dtype=torch.uint8,
                     device=device)

    def step():
        ssm.ssd_chunk_fwd(x, dl, A, Bm, Cm, D=Dv, delta_bias=bias, chunk_size=p.chunk, y=y,
                          h_final=hf, workspace=ws)
    return _median_event_time(step, flush, iters)


def time_decode(p, steps, flush, device):
    """Per-step time of ssm_step_decode with the state in place over `steps` distinct
    token steps, all generated on the device before timing (the recipe's distributions,
    torch's seeded generator; about 7.9 MB per step).  Returns (median with L2 flushed
    before each of the first 50 steps, mean over all steps back to back)."""
    import torch
    import selective_state_space_132_b300 as ssm
    io = torch.bfloat16
    t = _to_dev(device)
    state = t(p.state0)
    A, Dv, bias = t(p.A), t(p.D), t(p.bias)
    g = torch.Generator(device=device)
    g.manual_seed(p.seed)
    shp = (steps, p.batch, p.dim)
    xs = torch.randn(shp, generator=g, device=device).to(io)
    dls = (0.5 * torch.randn(shp, generator=g, device=device)).to(io)
    zs = torch.randn(shp, generator=g, device=device).to(io)
    Bs = torch.randn((steps, p.batch, p.dstate), generator=g, device=device).to(io)
    Cs = torch.randn((steps, p.batch, p.dstate), generator=g, device=device).to(io)
    y = torch.empty((p.batch, p.dim), dtype=io, device=device)

    def step(i):
        ssm.step_decode(state, xs[i], dls[i], A, Bs[i], Cs[i], D=Dv, z=zs[i],
                        delta_bias=bias, y=y)
    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    flushed = []
    for i in range(min(steps, 50)):
        flush()
        _gpu_lead()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        step(i)
        b.record()
        torch.cuda.synchronize()
        flushed.append(a.elapsed_time(b) * 1e-3)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for i in range(steps):
        step(i)
    b.record()
    torch.cuda.synchronize()
    return float(np.median(flushed)), a.elapsed_time(b) * 1e-3 / steps


def ssd_decode_bytes_per_step(nb, H, P, G, N, e):
    return 2 * nb * H * P * N * 4 + 2 * nb * H * P * e + nb * H * e + 2 * nb * G * N * e + 3 * H * 4


def time_ssd_decode(nb, H, P, G, N, flush, device, iters=30):
    """Median per-step time of ssm_ssd_step_decode (multi-head decode step, state in
    place) with L2 flushed before each step; seeded synthetic state and tokens."""
    import torch
    import selective_state_space_132_b300 as ssm
    p = W.ssd_problem(nb, 1, H, P, G, N, io="bf16", seed=1005, h0=True)
    t = _to_dev(device)
    io = torch.bfloat16
    state = t(p.h0)
    x, dl = t(p.x[:, 0], io), t(p.delta[:, 0], io)
    Bm, Cm = t(p.B[:, 0], io), t(p.C[:, 0], io)
    A, Dv, bias = t(p.A), t(p.D), t(p.bias)
    y = torch.empty_like(x)

    def step():
        ssm.ssd_step_decode(state, x, dl, A, Bm, Cm, D=Dv, delta_bias=bias, y=y)
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    times = []
    for _ in range(iters):
        flush()
        _gpu_lead()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        step()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) * 1e-3)
    return float(np.median(times))


def conv1d_bytes(nb, L, D, K, e):
    return 2 * nb * L * D * e + D * K * 4 + D * 4


def time_conv1d(nb, L, D, K, flush, device, iters=30):
    """Median time of ssm_conv1d (causal depthwise Conv1D + SiLU), L2 flushed."""
    import torch
    import selective_state_space_132_b300 as ssm
    rng = np.random.default_rng(1006)
    t = _to_dev(device)
    x = t(rng.standard_normal((nb, L, D), dtype=np.float32), torch.bfloat16)
    w = t(rng.standard_normal((D, K), dtype=np.float32) / np.sqrt(K))
    bias = t(rng.standard_normal(D, dtype=np.float32) * 0.1)
    out = torch.empty_like(x)
    return _median_event_time(lambda: ssm.conv1d(x, w, bias, out=out), flush, iters)


def scan_bwd_bytes(nb, L, D, N, e, gate=True):
    """Each input read once (x, delta, z, dy; B, C; A, D, bias), each gradient written
    once (dx, ddelta, dz in the I/O type; dB, dC, dA, dD, dbias in fp32)."""
    tok = nb * L * D * e
    return (4 if gate else 3) * tok + 2 * nb * L * N * e + (3 if gate else 2) * tok \
        + 2 * nb * L * N * 4 + 2 * D * N * 4 + 4 * D * 4


def time_scan_bwd(p, flush, device, iters=10, checkpoints=False):
    """Median time of one ssm_scan_bwd call on the scan problem p, including the zeroing
    of the summed gradients, L2 flushed before each call.  The states are recomputed:
    from checkpoints of the kernel's own (default), or from the checkpoints a forward
    call with checkpoints wrote (ssm_scan_bwd_ckpt); then also returns the median times
    of that forward call and of the plain forward call."""
    import torch
    import selective_state_space_132_b300 as ssm
    t = _to_dev(device)
    io = torch.bfloat16 if p.io == "bf16" else torch.float32
    x, dl, z = t(p.x, io), t(p.delta, io), t(p.z, io)
    Bm, Cm = t(p.B, io), t(p.C, io)
    A, Dv, bias = t(p.A), t(p.D), t(p.bias)
    dy = torch.randn_like(x)
    if not checkpoints:
        ws = torch.empty(ssm.scan_bwd_workspace_size(p.batch, p.seqlen, p.dim, p.dstate, io),
                         dtype=torch.uint8, device=device)
        return _median_event_time(
            lambda: ssm.scan_bwd(dy, x, dl, A, Bm, Cm, D=Dv, z=z, delta_bias=bias,
                                 workspace=ws), flush, iters)
    ck = torch.empty(ssm.scan_ckpt_shape(p.batch, p.seqlen, p.dim, p.dstate),
                     dtype=torch.float32, device=device)
    y = torch.empty_like(x)
    hf = torch.empty((p.batch, p.dim, p.dstate), dtype=torch.float32, device=device)

    def fwd(with_ck):
        ssm.scan_fwd(x, dl, A, Bm, Cm, D=Dv, z=z, delta_bias=bias, y=y, h_final=hf,
                     checkpoints=ck if with_ck else None)
    t_fwd_ck = _median_event_time(lambda: fwd(True), flush, iters)
    t_fwd = _median_event_time(lambda: fwd(False), flush, iters)
    fwd(True)
    ws = torch.empty(256, dtype=torch.uint8, device=device)
    t_bwd = _median_event_time(
        lambda: ssm.scan_bwd(dy, x, dl, A, Bm, Cm, D=Dv, z=z, delta_bias=bias, workspace=ws,
                             checkpoints=ck), flush, iters)
    return t_bwd, t_fwd_ck, t_fwd, ck.numel() * 4


def cpu_baseline_scan(p, target_s=10.0, max_s=30.0):
    """The fp64 oracle as it stands on a bounded channel sample of the workload: on all
    host cores (the reported value) and on one core; returns updates/s and what the
    samples were."""
    import oracle
    threads = oracle.default_threads()

    def run(nch, th):
        args = p.oracle_args()
        sel = slice(0, nch)
        for k in ("x", "delta", "z"):
            args[k] = np.ascontiguousarray(getattr(p, k)[:, :, sel])
        args["A"], args["Dv"], args["bias"] = p.A[sel], p.D[sel], p.bias[sel]
        t0 = time.perf_counter()
        oracle.scan(**args, threads=th)
        return time.perf_counter() - t0

    def sample(th, goal):
        nch = min(p.dim, 16)
        dt = run(nch, th)
        while dt < goal / 4 and nch < p.dim:
            nch = min(p.dim, nch * 4)
            dt = run(nch, th)
            if dt > max_s:
                break
        return nch, dt
    nch, dt = sample(threads, target_s)
    n1, dt1 = sample(1, target_s / 2)
    updates = p.batch * p.seqlen * nch * p.dstate
    upd1 = p.batch * p.seqlen * n1 * p.dstate
    return {"value": updates / dt, "unit": "state-updates/s", "cores": threads,
            "kind": "oracle",
            "sample": f"batch {p.batch} x L {p.seqlen} x {nch} of {p.dim} channels x N "
                      f"{p.dstate} ({updates:.3e} updates, {dt:.1f} s, fp64 C + OpenMP)",
            "value_1_thread": upd1 / dt1,
            "sample_1_thread": f"{n1} channels ({upd1:.3e} updates, {dt1:.1f} s, one core)"}


def _oracle_timed(fn, units, unit, sample):
    """The fp64 oracle as it stands on a bounded sample, all host cores."""
    import oracle
    t0 = time.perf_counter()
    fn(oracle.default_threads())
    dt = time.perf_counter() - t0
    return {"value": units / dt, "unit": unit, "cores": oracle.default_threads(),
            "kind": "oracle", "sample": f"{sample} ({dt:.2f} s, fp64 C + OpenMP)"}


def _oracle_decode(p, steps=10):
    import oracle
    state = p.state0.astype(np.float64)
    toks = [p.tokens(s) for s in range(steps)]

    def run(th):
        for tok in toks:
            oracle.decode_step(state, tok["x"], tok["delta"], p.A, tok["B"], tok["C"], Dv=p.D,
                               z=tok["z"], bias=p.bias, threads=th)
    return _oracle_timed(run, steps * p.updates_per_step, "state-updates/s",
                         f"{steps} steps of the whole batch")


def run_ours(args, world, rank, local):
    import torch
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    hbm, tf_burst, tf_sus, peak_kind = measured_peaks()
    p = W.config_problem(WORKLOADS[args.workload])
    flush = L2Flush(device)
    units = p.updates
    e = 2 if p.io == "bf16" else 4
    algo = scan_bytes(p.batch, p.seqlen, p.dim, p.dstate, e)

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    per, launches, wall, window = time_scan(p, args.steps, args.warmup, flush, device)
    barrier(world)
    torch.cuda.synchronize()
    if sampler:
        time.sleep(0.1)
        sampler.stop()
    dev_s = float(np.sum(per))
    sec_per_step = max_over_ranks(dev_s, world) / args.steps
    value = aggregate(units, sec_per_step, world)
    achieved = algo / float(np.mean(per)) / 1e9
    rate = units / float(np.mean(per))        # state updates/s of one launch (this rank)
    alu_peak = scan_dispatch_peak(device)
    src_hash = kernel_source_hash(SCAN_SOURCES)
    traffic = PROFILED_TRAFFIC.get(src_hash, {}).get(args.workload)
    out = {
        "metric": "selective-scan state updates/s (B*L*D*N)",
        "value": value, "unit": "state-updates/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sec_per_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; reference recipe)",
        "config": bench_config(args.workload, p, world),
        # the scan is bound by instruction dispatch (ceilings: dispatch 669 us against
        # 331 us of HBM time at this workload), so the roofline is the ALU one; the HBM
        # fraction sits beside it
        "roofline": {"bound": "alu", "achieved": rate, "peak": alu_peak,
                     "unit": "state-updates/s", "frac": rate / alu_peak, "traffic": traffic,
                     "peak_basis": f"{torch.cuda.get_device_properties(device).multi_processor_count}"
                                   " SMs x 4 sub-partitions x 32 lanes x 2032 MHz dispatch "
                                   f"slots / {DISPATCH_SLOTS_PER_UPDATE} slots per state update "
                                   "(one ex2 at two, four fp32 operations at one)",
                     "hbm": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                             "frac": achieved / hbm, "traffic": traffic, "peak_kind": peak_kind,
                             "algorithmic_bytes_per_launch": algo,
                             "frac_of_nominal_8000": achieved / 8000.0},
                     # what the kernel's own binding units show under ncu (null once the
                     # sources differ from the capture's)
                     "profiled_occupancy": PROFILED_OCCUPANCY.get(src_hash, {}).get(args.workload),
                     "source_hash": src_hash},
        "gpu_launches": launches * args.steps,
        "wall_ms_per_step_incl_flush": wall / args.steps * 1e3,
        "ceilings": scan_ceilings(p, algo, hbm, device),
        "device": torch.cuda.get_device_name(device),
    }
    # end to end on every rank at once (each with its own pinned host buffers): the
    # job's updates over the slowest rank's time
    barrier(world)
    e2e_s, h2d, d2h, nslices = e2e_scan(p, min(args.steps, 20), device)
    e2e_max = max_over_ranks(e2e_s, world)
    if rank == 0:
        out["clocks"] = sampler.summary(*window) if sampler else None
        out["e2e"] = {"value": aggregate(units, e2e_max, world), "unit": "state-updates/s",
                      "h2d_bytes_per_step": h2d * world, "d2h_bytes_per_step": d2h * world,
                      "ms_per_step": e2e_max * 1e3,
                      "pipeline": f"{nslices}; copy in, scan and copy out on three "
                                  "streams"}
        if world == 1 and not args.no_cpu:
            out["cpu_baseline"] = cpu_baseline_scan(p)
        if not args.no_extras and world == 1:
            ks = ClockSampler(local)
            ks.start()
            try:
                out["kernels"] = extras(device, flush, hbm, tf_sus, skip=(args.workload,),
                                        sampler=ks)
            finally:
                ks.stop()
    return out


def extras(device, flush, hbm, tf_sus, only=None, iters=None, skip=(), sampler=None):
    """The other workloads, one measurement each (parity cases, not the bench line).
    `only` runs one of them alone and `iters` sets its timed iterations (both used to
    profile one kernel with ncu)."""
    import torch

    def n(default):
        return default if iters is None else iters

    def scan_cfg(index, nch):
        def run():
            p = W.config_problem(index)
            per, launches, _, _ = time_scan(p, n(5 if index == 2 else 20), 3, flush, device)
            s = float(np.median(per))
            b = scan_bytes(p.batch, p.seqlen, p.dim, p.dstate, 2)
            import oracle
            args = p.oracle_args()
            for k in ("x", "delta", "z"):
                args[k] = np.ascontiguousarray(getattr(p, k)[:, :, :nch])
            args["A"], args["Dv"], args["bias"] = p.A[:nch], p.D[:nch], p.bias[:nch]
            orc = _oracle_timed(lambda th: oracle.scan(**args, threads=th),
                                p.batch * p.seqlen * nch * p.dstate, "state-updates/s",
                                f"{nch} of {p.dim} channels, whole sequence")
            return {"ms": s * 1e3, "updates_per_s": p.updates / s, "gbs": b / s / 1e9,
                    "hbm_frac": b / s / 1e9 / hbm, "launches": launches, "oracle": orc}
        return run

    def ssd():
        p = W.config_problem(3)
        s = time_ssd(p, n(5), flush, device)
        b = ssd_bytes(p.batch, p.seqlen, p.heads, p.headdim, p.ngroups, p.dstate, 2)
        # the tensor-core kernel works in 128-step chunks whatever chunk_size asks for
        fl = ssd_flops(p.batch, p.seqlen, p.heads, p.headdim, p.ngroups, p.dstate, 128)
        import oracle
        nh = 4
        args = p.oracle_args()
        args["x"] = np.ascontiguousarray(p.x[:1, :, :nh])
        args["delta"] = np.ascontiguousarray(p.delta[:1, :, :nh])
        args["Bm"], args["Cm"] = p.B[:1], p.C[:1]
        args["A"], args["Dv"], args["bias"] = p.A[:nh], p.D[:nh], p.bias[:nh]
        orc = _oracle_timed(lambda th: oracle.ssd(**args, threads=th),
                            p.seqlen * nh * p.headdim * p.dstate, "state-updates/s",
                            f"batch row 0, {nh} of {p.heads} heads, whole sequence")
        return {"ms": s * 1e3, "updates_per_s": p.updates / s, "gbs": b / s / 1e9,
                "hbm_frac": b / s / 1e9 / hbm, "tensor_tflops": fl / s / 1e12,
                "tensor_frac_sustained": fl / s / 1e12 / tf_sus, "kernel_chunk": 128,
                "oracle": orc}

    def decode():
        p = W.config_problem(4)
        steps = p.steps if iters is None else iters
        s_flush, s_hot = time_decode(p, steps, flush, device)
        b = decode_bytes_per_step(p.batch, p.dim, p.dstate, 2)
        return {"ms_per_step_l2_flushed": s_flush * 1e3, "ms_per_step_back_to_back": s_hot * 1e3,
                "updates_per_s": p.updates_per_step / s_flush,
                "gbs_l2_flushed": b / s_flush / 1e9, "hbm_frac_l2_flushed": b / s_flush / 1e9 / hbm,
                "gbs_back_to_back": b / s_hot / 1e9,
                "note": "1000 distinct token steps; back-to-back steps keep much of the 84 MB "
                        "state in the 126 MB L2",
                "oracle": _oracle_decode(p)}

    def ssd_decode():
        s = time_ssd_decode(64, 80, 64, 1, 128, flush, device, iters=n(30))
        b = ssd_decode_bytes_per_step(64, 80, 64, 1, 128, 2)
        import oracle
        q = W.ssd_problem(64, 1, 80, 64, 1, 128, io="bf16", seed=1005, h0=True)
        state = q.h0.astype(np.float64)
        orc = _oracle_timed(
            lambda th: [oracle.ssd_decode_step(state, q.x[:, 0], q.delta[:, 0], q.A, q.B[:, 0],
                                               q.C[:, 0], Dv=q.D, bias=q.bias, threads=th)
                        for _ in range(3)],
            3 * 64 * 80 * 64 * 128, "state-updates/s", "3 steps of the whole batch")
        return {"ms_per_step_l2_flushed": s * 1e3, "updates_per_s": 64 * 80 * 64 * 128 / s,
                "gbs_l2_flushed": b / s / 1e9, "hbm_frac_l2_flushed": b / s / 1e9 / hbm,
                "oracle": orc}

    def conv1d():
        s = time_conv1d(8, 2048, 1536, 4, flush, device, iters=n(30))
        b = conv1d_bytes(8, 2048, 1536, 4, 2)
        import oracle
        rng = np.random.default_rng(1006)
        x = rng.standard_normal((8, 2048, 1536))
        w = rng.standard_normal((1536, 4)) / 2
        orc = _oracle_timed(lambda th: oracle.conv1d(x, w, threads=th), 8 * 2048 * 1536,
                            "outputs/s", "the whole block shape")
        return {"ms": s * 1e3, "gbs": b / s / 1e9, "hbm_frac": b / s / 1e9 / hbm,
                "outputs_per_s": 8 * 2048 * 1536 / s, "oracle": orc}

    def scan_bwd():
        p = W.config_problem(1)
        s = time_scan_bwd(p, flush, device, iters=n(10))
        b = scan_bwd_bytes(p.batch, p.seqlen, p.dim, p.dstate, 2)
        import oracle
        gy = np.random.default_rng(7).standard_normal((1, p.seqlen, p.dim))
        orc = _oracle_timed(
            lambda th: oracle.scan_bwd(gy, p.x[:1], p.delta[:1], p.A, p.B[:1], p.C[:1],
                                       Dv=p.D, z=p.z[:1], bias=p.bias, threads=th),
            p.seqlen * p.dim * p.dstate, "state-updates/s", "batch row 0 of 8")
        sc, f_ck, f, ck_bytes = time_scan_bwd(p, flush, device, iters=n(10), checkpoints=True)
        return {"ms": s * 1e3, "updates_per_s": p.updates / s, "gbs": b / s / 1e9,
                "hbm_frac": b / s / 1e9 / hbm,
                "note": "states recomputed: a checkpoint pass and a reverse pass",
                "from_forward_checkpoints": {
                    "ms": sc * 1e3, "updates_per_s": p.updates / sc,
                    "forward_with_checkpoints_ms": f_ck * 1e3, "forward_ms": f * 1e3,
                    "checkpoint_bytes": ck_bytes,
                    "note": "the forward call keeps the state every 16 steps and the "
                            "backward starts from them (reverse pass only)"},
                "oracle": orc}

    runners = {
        "scan_bf16_B8_D1536_L2048_N16": scan_cfg(1, 256),
        "scan_bf16_B1_D2048_L131072_N16": scan_cfg(2, 64),
        "ssd_bf16_B4_L8192_H80_P64_N128_G1_Q256": ssd,
        "decode_bf16_B256_D5120_N16_x1000": decode,
        "ssd_decode_bf16_B64_H80_P64_N128": ssd_decode,
        "conv1d_silu_bf16_B8_L2048_D1536_K4": conv1d,
        "scan_bwd_bf16_B8_D1536_L2048_N16": scan_bwd,
    }
    if only is not None and only not in runners:
        raise SystemExit(f"unknown extra {only!r}; one of {sorted(runners)}")
    res = {}
    for name, fn in runners.items():
        if (only is not None and name != only) or name in skip:
            continue
        t0 = time.time()
        res[name] = fn()
        if sampler is not None:
            # the SM clocks and throttle reasons while this workload ran
            res[name]["clocks"] = sampler.summary(t0, time.time())
        torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------ reference arm
def run_reference(args, world):
    """The fp64 oracle, as it stands, on the host cores; one step = one oracle run over
    a bounded channel sample of the same workload."""
    import oracle
    p = W.config_problem(WORKLOADS[args.workload])
    threads = oracle.default_threads()
    budget_s = 120.0 / max(1, args.steps + args.warmup)

    def make(nch):
        a = p.oracle_args()
        sel = slice(0, nch)
        for k in ("x", "delta", "z"):
            a[k] = np.ascontiguousarray(getattr(p, k)[:, :, sel], np.float64)
        a["A"], a["Dv"], a["bias"] = p.A[sel], p.D[sel], p.bias[sel]
        for k in ("Bm", "Cm"):
            a[k] = np.ascontiguousarray(a[k], np.float64)
        return a
    nch = 8
    a = make(nch)
    t0 = time.perf_counter()
    oracle.scan(**a, threads=threads)
    rate = p.batch * p.seqlen * nch * p.dstate / (time.perf_counter() - t0)
    nch = int(max(1, min(p.dim, rate * budget_s / (p.batch * p.seqlen * p.dstate))))
    a = make(nch)
    for _ in range(args.warmup):
        oracle.scan(**a, threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.scan(**a, threads=threads)
    dt = (time.perf_counter() - t0) / args.steps
    units = p.batch * p.seqlen * nch * p.dstate
    value = units / dt
    sample = (f"batch {p.batch} x L {p.seqlen} x {nch} of {p.dim} channels x N {p.dstate} "
              f"per step ({units:.3e} updates)")
    return {
        "impl": "reference", "metric": "selective-scan state updates/s (B*L*D*N)",
        "value": value, "unit": "state-updates/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; reference recipe)",
        "config": bench_config(args.workload, p, world),
        "cpu_baseline": {"value": value, "unit": "state-updates/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "state-updates/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(k for k in WORKLOADS if k.startswith("scan")),
                    default="scan_bf16_B1_D2048_L131072_N16")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--only-extra", default=None,
                    help="run one of the other workloads alone and print its measurement")
    ap.add_argument("--extra-iters", type=int, default=None,
                    help="timed iterations of --only-extra (after 3 warm-up calls)")
    args = ap.parse_args(argv)
    if args.only_extra is not None:
        import torch
        device = torch.device("cuda", 0)
        hbm, _, tf_sus, _ = measured_peaks()
        flush = L2Flush(device)
        res = extras(device, flush, hbm, tf_sus, only=args.only_extra, iters=args.extra_iters)
        print(json.dumps({"extra": args.only_extra, **res[args.only_extra]}))
        return 0
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        if int(os.environ.get("RANK", "0")) != 0:
            return 0
        print(json.dumps(run_reference(args, world)))
        return 0
    world, rank, local = dist_setup()
    out = run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
