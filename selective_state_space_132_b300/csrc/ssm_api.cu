// C ABI of libssm.so: host-side validation, workspace sizing and dispatch to the
// kernels.  Every check runs before any launch; on failure nothing is enqueued.
#include "../../include/ssm.h"
#include <nvtx3/nvToolsExt.h>

#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace {
// An NVTX range around each compute entry point, so that profilers can attribute
// kernels to the library call that launched them (a no-op without a profiler).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};


using ssm::kStatusBytes;

constexpr int kVersion = 1 * 10000 + 0 * 100 + 0;

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t io_size(int32_t dt) { return dt == SSM_BF16 ? 2 : 4; }

// [p, p + bytes) overlaps [q, q + qbytes)
bool overlaps(const void *p, size_t bytes, const void *q, size_t qbytes) {
    if (!p || !q || bytes == 0 || qbytes == 0) return false;
    auto a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return a < b + qbytes && b < a + bytes;
}

ssm_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA; }

// ------------------------------------------------------------------ scan
ssm_status check_scan(const ssm_scan_args *a, bool pointers = true) {
    if (!a) return SSM_ERR_INVALID_ARG;
    if (a->batch < 0 || a->seqlen < 0 || a->dim < 0 || a->dstate < 1) return SSM_ERR_INVALID_ARG;
    if (a->io_dtype != SSM_F32 && a->io_dtype != SSM_BF16) return SSM_ERR_INVALID_ARG;
    if (a->delta_softplus != 0 && a->delta_softplus != 1) return SSM_ERR_INVALID_ARG;
    if (a->time_chunk < 0 || a->time_chunk % 32 != 0) return SSM_ERR_INVALID_ARG;
    if (a->discretization != SSM_DISC_EULER && a->discretization != SSM_DISC_ZOH)
        return SSM_ERR_INVALID_ARG;
    if (a->dstate > 64) return SSM_ERR_UNSUPPORTED;
    if (a->batch > 65535) return SSM_ERR_UNSUPPORTED;
    if (a->seqlen > (int64_t)1 << 40 || a->dim > (int64_t)1 << 31) return SSM_ERR_UNSUPPORTED;
    if (!pointers) return SSM_OK;
    const bool tokens = a->batch * a->seqlen * a->dim > 0;
    const bool rows = a->batch * a->seqlen > 0;
    if (tokens && (!a->x || !a->delta || !a->y)) return SSM_ERR_INVALID_ARG;
    if (rows && a->dim > 0 && (!a->B || !a->C)) return SSM_ERR_INVALID_ARG;
    if (a->dim > 0 && !a->A) return SSM_ERR_INVALID_ARG;
    const size_t e = io_size(a->io_dtype);
    const void *io_ptrs[] = {a->x, a->delta, a->B, a->C, a->z, a->y};
    for (const void *p : io_ptrs)
        if (!aligned(p, e)) return SSM_ERR_ALIGNMENT;
    const void *f_ptrs[] = {a->A, a->D, a->delta_bias, a->h0, a->h_final};
    for (const void *p : f_ptrs)
        if (!aligned(p, 4)) return SSM_ERR_ALIGNMENT;
    const size_t tok_bytes = (size_t)(a->batch * a->seqlen * a->dim) * e;
    const size_t bc_bytes = (size_t)(a->batch * a->seqlen * a->dstate) * e;
    const size_t st_bytes = (size_t)(a->batch * a->dim * a->dstate) * 4;
    if (overlaps(a->y, tok_bytes, a->x, tok_bytes) || overlaps(a->y, tok_bytes, a->delta, tok_bytes) ||
        overlaps(a->y, tok_bytes, a->z, tok_bytes) || overlaps(a->y, tok_bytes, a->B, bc_bytes) ||
        overlaps(a->y, tok_bytes, a->C, bc_bytes) || overlaps(a->h_final, st_bytes, a->h0, st_bytes) ||
        overlaps(a->y, tok_bytes, a->h_final, st_bytes))
        return SSM_ERR_INVALID_ARG;
    return SSM_OK;
}

// The plan depends on sizes and flags only: the TMA-staged kernel's plan when the
// sizes allow it (pointers that turn out unaligned at call time run the general
// kernel on the same plan).  The workspace always holds the device status word.
size_t scan_ws(const ssm_scan_args *a, int64_t *chunk_len, int *nchunks) {
    const int bf = a->io_dtype == SSM_BF16;
    const int tma_bps = ssm::scan_tma_sizes_ok(bf, a->seqlen, a->dim, a->dstate)
                            ? ssm::scan_tma_blocks_per_sm(bf, a->dstate)
                            : 0;
    ssm::scan_plan(a->batch, a->seqlen, a->dim, a->dstate, a->time_chunk, tma_bps, chunk_len,
                   nchunks);
    return ssm::scan_workspace_bytes(a->batch, a->dim, a->dstate, *nchunks);
}

// ------------------------------------------------------------------ ssd
ssm_status check_ssd(const ssm_ssd_args *a, bool pointers = true) {
    if (!a) return SSM_ERR_INVALID_ARG;
    if (a->batch < 0 || a->seqlen < 0 || a->nheads < 1 || a->headdim < 1 || a->ngroups < 1 ||
        a->dstate < 1 || a->chunk_size < 0)
        return SSM_ERR_INVALID_ARG;
    if (a->nheads % a->ngroups != 0) return SSM_ERR_INVALID_ARG;
    if (a->io_dtype != SSM_F32 && a->io_dtype != SSM_BF16) return SSM_ERR_INVALID_ARG;
    if (a->delta_softplus != 0 && a->delta_softplus != 1) return SSM_ERR_INVALID_ARG;
    if (a->dstate > 256) return SSM_ERR_UNSUPPORTED;
    if (a->batch * a->nheads * a->headdim > ((int64_t)1 << 31)) return SSM_ERR_UNSUPPORTED;
    if (!pointers) return SSM_OK;
    const bool rows = a->batch * a->seqlen > 0;
    if (rows && (!a->x || !a->delta || !a->y || !a->B || !a->C)) return SSM_ERR_INVALID_ARG;
    if (!a->A) return SSM_ERR_INVALID_ARG;
    const size_t e = io_size(a->io_dtype);
    const void *io_ptrs[] = {a->x, a->delta, a->B, a->C, a->z, a->y};
    for (const void *p : io_ptrs)
        if (!aligned(p, e)) return SSM_ERR_ALIGNMENT;
    const void *f_ptrs[] = {a->A, a->D, a->delta_bias, a->h0, a->h_final};
    for (const void *p : f_ptrs)
        if (!aligned(p, 4)) return SSM_ERR_ALIGNMENT;
    if (a->workspace && !aligned(a->workspace, 256)) return SSM_ERR_ALIGNMENT;
    const size_t tok = (size_t)(a->batch * a->seqlen * a->nheads * a->headdim) * e;
    const size_t bc = (size_t)(a->batch * a->seqlen * a->ngroups * a->dstate) * e;
    const size_t dl = (size_t)(a->batch * a->seqlen * a->nheads) * e;
    const size_t st = (size_t)(a->batch * a->nheads * a->headdim * a->dstate) * 4;
    if (overlaps(a->y, tok, a->x, tok) || overlaps(a->y, tok, a->z, tok) ||
        overlaps(a->y, tok, a->B, bc) || overlaps(a->y, tok, a->C, bc) ||
        overlaps(a->y, tok, a->delta, dl) || overlaps(a->h_final, st, a->h0, st) ||
        overlaps(a->y, tok, a->h_final, st))
        return SSM_ERR_INVALID_ARG;
    return SSM_OK;
}

ssm::SSDParams ssd_params(const ssm_ssd_args *a) {
    ssm::SSDParams p{};
    p.batch = a->batch;
    p.seqlen = a->seqlen;
    p.nheads = a->nheads;
    p.headdim = a->headdim;
    p.ngroups = a->ngroups;
    p.dstate = a->dstate;
    p.chunk = a->chunk_size > 0 ? a->chunk_size : 256;
    p.io_bf16 = a->io_dtype == SSM_BF16;
    p.softplus = a->delta_softplus;
    p.x = a->x;
    p.delta = a->delta;
    p.Bm = a->B;
    p.Cm = a->C;
    p.z = a->z;
    p.A = a->A;
    p.Dv = a->D;
    p.bias = a->delta_bias;
    p.h0 = a->h0;
    p.y = a->y;
    p.h_final = a->h_final;
    p.status = a->workspace;
    p.work = a->workspace ? static_cast<char *>(a->workspace) + kStatusBytes : nullptr;
    p.work_bytes = a->workspace_bytes > kStatusBytes ? a->workspace_bytes - kStatusBytes : 0;
    return p;
}

// ------------------------------------------------------------------ decode
ssm_status check_decode(const ssm_decode_args *a) {
    if (!a) return SSM_ERR_INVALID_ARG;
    if (a->batch < 0 || a->dim < 0 || a->dstate < 1) return SSM_ERR_INVALID_ARG;
    if (a->io_dtype != SSM_F32 && a->io_dtype != SSM_BF16) return SSM_ERR_INVALID_ARG;
    if (a->delta_softplus != 0 && a->delta_softplus != 1) return SSM_ERR_INVALID_ARG;
    if (a->dstate > 64) return SSM_ERR_UNSUPPORTED;
    if (a->discretization != SSM_DISC_EULER && a->discretization != SSM_DISC_ZOH)
        return SSM_ERR_INVALID_ARG;
    if (a->batch * a->dim * 16 > ((int64_t)1 << 40)) return SSM_ERR_UNSUPPORTED;
    if (a->batch * a->dim > 0 &&
        (!a->state || !a->x || !a->delta || !a->B || !a->C || !a->A || !a->y))
        return SSM_ERR_INVALID_ARG;
    const size_t e = io_size(a->io_dtype);
    const void *io_ptrs[] = {a->x, a->delta, a->B, a->C, a->z, a->y};
    for (const void *p : io_ptrs)
        if (!aligned(p, e)) return SSM_ERR_ALIGNMENT;
    const void *f_ptrs[] = {a->state, a->A, a->D, a->delta_bias};
    for (const void *p : f_ptrs)
        if (!aligned(p, 4)) return SSM_ERR_ALIGNMENT;
    const size_t tok = (size_t)(a->batch * a->dim) * e;
    const size_t st = (size_t)(a->batch * a->dim * a->dstate) * 4;
    if (overlaps(a->y, tok, a->x, tok) || overlaps(a->y, tok, a->delta, tok) ||
        overlaps(a->y, tok, a->z, tok) || overlaps(a->y, tok, a->state, st))
        return SSM_ERR_INVALID_ARG;
    if (a->workspace) {
        if (a->workspace_bytes < ssm::kStatusBytes) return SSM_ERR_WORKSPACE;
        if (!aligned(a->workspace, 256)) return SSM_ERR_ALIGNMENT;
    }
    return SSM_OK;
}

// ------------------------------------------------------------------ multi-head decode
ssm_status check_ssd_decode(const ssm_ssd_decode_args *a) {
    if (!a) return SSM_ERR_INVALID_ARG;
    if (a->batch < 0 || a->nheads < 1 || a->headdim < 1 || a->ngroups < 1 || a->dstate < 1)
        return SSM_ERR_INVALID_ARG;
    if (a->nheads % a->ngroups != 0) return SSM_ERR_INVALID_ARG;
    if (a->io_dtype != SSM_F32 && a->io_dtype != SSM_BF16) return SSM_ERR_INVALID_ARG;
    if (a->delta_softplus != 0 && a->delta_softplus != 1) return SSM_ERR_INVALID_ARG;
    if (a->dstate > 256) return SSM_ERR_UNSUPPORTED;
    if (a->batch * a->nheads * a->headdim * 32 > ((int64_t)1 << 40)) return SSM_ERR_UNSUPPORTED;
    if (a->batch > 0 &&
        (!a->state || !a->x || !a->delta || !a->B || !a->C || !a->A || !a->y))
        return SSM_ERR_INVALID_ARG;
    const size_t e = io_size(a->io_dtype);
    const void *io_ptrs[] = {a->x, a->delta, a->B, a->C, a->z, a->y};
    for (const void *p : io_ptrs)
        if (!aligned(p, e)) return SSM_ERR_ALIGNMENT;
    const void *f_ptrs[] = {a->state, a->A, a->D, a->delta_bias};
    for (const void *p : f_ptrs)
        if (!aligned(p, 4)) return SSM_ERR_ALIGNMENT;
    const size_t tok = (size_t)(a->batch * a->nheads * a->headdim) * e;
    const size_t st = (size_t)(a->batch * a->nheads * a->headdim * a->dstate) * 4;
    if (overlaps(a->y, tok, a->x, tok) || overlaps(a->y, tok, a->z, tok) ||
        overlaps(a->y, tok, a->state, st))
        return SSM_ERR_INVALID_ARG;
    return SSM_OK;
}

// ------------------------------------------------------------------ scan backward
ssm_status check_scan_bwd(const ssm_scan_bwd_args *a, bool pointers = true) {
    if (!a) return SSM_ERR_INVALID_ARG;
    if (a->batch < 0 || a->seqlen < 0 || a->dim < 0 || a->dstate < 1) return SSM_ERR_INVALID_ARG;
    if (a->io_dtype != SSM_F32 && a->io_dtype != SSM_BF16) return SSM_ERR_INVALID_ARG;
    if (a->delta_softplus != 0 && a->delta_softplus != 1) return SSM_ERR_INVALID_ARG;
    if (a->discretization != SSM_DISC_EULER && a->discretization != SSM_DISC_ZOH)
        return SSM_ERR_INVALID_ARG;
    if (a->dstate > 64) return SSM_ERR_UNSUPPORTED;
    if (a->batch > 65535) return SSM_ERR_UNSUPPORTED;
    if (a->seqlen > (int64_t)1 << 40 || a->dim > (int64_t)1 << 31) return SSM_ERR_UNSUPPORTED;
    if (!pointers) return SSM_OK;
    const bool tokens = a->batch * a->seqlen * a->dim > 0;
    if (tokens && (!a->x || !a->delta || !a->B || !a->C || !a->dy || !a->dx || !a->ddelta ||
                   !a->dB || !a->dC))
        return SSM_ERR_INVALID_ARG;
    if (tokens && (a->z != nullptr) != (a->dz != nullptr)) return SSM_ERR_INVALID_ARG;
    if (a->dim > 0 && (!a->A || !a->dA)) return SSM_ERR_INVALID_ARG;
    const size_t e = io_size(a->io_dtype);
    const void *io_ptrs[] = {a->x, a->delta, a->B, a->C, a->z, a->dy, a->dx, a->ddelta, a->dz};
    for (const void *p : io_ptrs)
        if (!aligned(p, e)) return SSM_ERR_ALIGNMENT;
    const void *f_ptrs[] = {a->A, a->D, a->delta_bias, a->h0, a->dh_final, a->dA, a->dB,
                            a->dC, a->dD, a->ddelta_bias, a->dh0};
    for (const void *p : f_ptrs)
        if (!aligned(p, 4)) return SSM_ERR_ALIGNMENT;
    const size_t tok = (size_t)(a->batch * a->seqlen * a->dim) * e;
    const size_t bc_io = (size_t)(a->batch * a->seqlen * a->dstate) * e;
    const size_t bc32 = (size_t)(a->batch * a->seqlen * a->dstate) * 4;
    const size_t st = (size_t)(a->batch * a->dim * a->dstate) * 4;
    const size_t dn = (size_t)(a->dim * a->dstate) * 4, d4 = (size_t)a->dim * 4;
    struct Buf { const void *p; size_t n; };
    const Buf ins[] = {{a->x, tok}, {a->delta, tok}, {a->B, bc_io}, {a->C, bc_io}, {a->z, tok},
                       {a->A, dn}, {a->D, d4}, {a->delta_bias, d4}, {a->h0, st},
                       {a->dy, tok}, {a->dh_final, st}};
    const Buf outs[] = {{a->dx, tok}, {a->ddelta, tok}, {a->dz, tok}, {a->dA, dn}, {a->dB, bc32},
                        {a->dC, bc32}, {a->dD, d4}, {a->ddelta_bias, d4}, {a->dh0, st}};
    for (size_t i = 0; i < sizeof(outs) / sizeof(outs[0]); ++i) {
        for (const Buf &in : ins)
            if (overlaps(outs[i].p, outs[i].n, in.p, in.n)) return SSM_ERR_INVALID_ARG;
        for (size_t j = 0; j < i; ++j)
            if (overlaps(outs[i].p, outs[i].n, outs[j].p, outs[j].n)) return SSM_ERR_INVALID_ARG;
    }
    return SSM_OK;
}

size_t scan_bwd_ws(const ssm_scan_bwd_args *a) {
    const size_t ck = ssm::scan_bwd_ckpt_floats(a->batch, a->seqlen, a->dim, a->dstate) * 4;
    return ssm::kStatusBytes + (ck + 255) / 256 * 256;
}

// ------------------------------------------------------------------ conv1d
ssm_status check_conv1d(const ssm_conv1d_args *a) {
    if (!a) return SSM_ERR_INVALID_ARG;
    if (a->batch < 0 || a->seqlen < 0 || a->dim < 0 || a->width < 1) return SSM_ERR_INVALID_ARG;
    if (a->io_dtype != SSM_F32 && a->io_dtype != SSM_BF16) return SSM_ERR_INVALID_ARG;
    if (a->silu != 0 && a->silu != 1) return SSM_ERR_INVALID_ARG;
    if (a->width > ssm::conv1d_max_width()) return SSM_ERR_UNSUPPORTED;
    const bool work = a->batch * a->seqlen * a->dim > 0;
    if (work && (!a->x || !a->out || !a->weight)) return SSM_ERR_INVALID_ARG;
    const size_t e = io_size(a->io_dtype);
    const void *io_ptrs[] = {a->x, a->x_prev, a->out};
    for (const void *p : io_ptrs)
        if (!aligned(p, e)) return SSM_ERR_ALIGNMENT;
    if (!aligned(a->weight, 4) || !aligned(a->bias, 4)) return SSM_ERR_ALIGNMENT;
    const size_t tok = (size_t)(a->batch * a->seqlen * a->dim) * e;
    const size_t prev = (size_t)(a->batch * (a->width - 1) * a->dim) * e;
    if (overlaps(a->out, tok, a->x, tok) || overlaps(a->out, tok, a->x_prev, prev))
        return SSM_ERR_INVALID_ARG;
    if (a->workspace) {
        if (a->workspace_bytes < ssm::kStatusBytes) return SSM_ERR_WORKSPACE;
        if (!aligned(a->workspace, 256)) return SSM_ERR_ALIGNMENT;
    }
    return SSM_OK;
}

}  // namespace

namespace ssm {
// Full argument check of a scan call (sizes, flags, pointers), for other entry points.
ssm_status check_scan_args(const ssm_scan_args *a) { return check_scan(a, true); }
}  // namespace ssm

extern "C" {

const char *ssm_status_string(ssm_status s) {
    switch (s) {
        case SSM_OK: return "ok";
        case SSM_ERR_INVALID_ARG: return "invalid argument";
        case SSM_ERR_UNSUPPORTED: return "unsupported size or configuration";
        case SSM_ERR_ALIGNMENT: return "misaligned pointer";
        case SSM_ERR_WORKSPACE: return "workspace missing or too small";
        case SSM_ERR_CUDA: return "CUDA runtime error";
        case SSM_ERR_TIMEOUT: return "a bounded device wait timed out";
        case SSM_ERR_BOUNDS: return "a kernel index check failed (debug-bounds build)";
    }
    return "unknown status";
}

int ssm_version(void) { return kVersion; }

ssm_status ssm_scan_workspace_size(const ssm_scan_args *a, size_t *bytes) {
    if (!bytes) return SSM_ERR_INVALID_ARG;
    ssm_status s = check_scan(a, false);
    if (s != SSM_OK) return s;
    int64_t cl;
    int k;
    *bytes = scan_ws(a, &cl, &k);
    return SSM_OK;
}

ssm_status ssm_scan_plan(const ssm_scan_args *a, int64_t *chunk_len, int32_t *nchunks,
                         int32_t *launches) {
    if (!chunk_len || !nchunks || !launches) return SSM_ERR_INVALID_ARG;
    ssm_status s = check_scan(a, false);
    if (s != SSM_OK) return s;
    int64_t cl;
    int k;
    scan_ws(a, &cl, &k);
    *chunk_len = cl;
    *nchunks = k;
    // the TMA kernel runs a split sequence in one launch (look-back carry), the general
    // kernel in two (summary pass, output pass)
    const bool tma = ssm::scan_tma_sizes_ok(a->io_dtype == SSM_BF16, a->seqlen, a->dim, a->dstate);
    *launches = (a->batch == 0 || a->dim == 0) ? 0 : (k > 1 && !tma ? 2 : 1);
    return SSM_OK;
}

}  // extern "C"

namespace {
int ckpt_shift(int64_t dstate) {
    int sh = 0;
    while ((1 << sh) < ssm::scan_ckpt_steps(dstate)) ++sh;
    return sh;
}
// Bytes of the state checkpoints of these sizes: (B, ceil(L / T), D, N) fp32.
size_t ckpt_bytes_for(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate) {
    return ssm::scan_bwd_ckpt_floats(batch, seqlen, dim, dstate) * sizeof(float);
}
// The scan call; `budget` and `publish` differ from the defaults only in the look-back
// self-test; `ckpt` (nullable) receives the backward pass's state checkpoints.
ssm_status scan_fwd_impl(const ssm_scan_args *a, ssm_stream_t stream, long long budget,
                         int publish, float *ckpt = nullptr) {
    ssm_status s = check_scan(a);
    if (s != SSM_OK) return s;
    int64_t cl;
    int k;
    if (a->batch == 0 || a->dim == 0) return SSM_OK;  // nothing to write
    const size_t need = scan_ws(a, &cl, &k);
    if (!a->workspace || a->workspace_bytes < need) return SSM_ERR_WORKSPACE;
    if (!aligned(a->workspace, 256)) return SSM_ERR_ALIGNMENT;
    ssm::ScanParams p{};
    p.batch = a->batch;
    p.seqlen = a->seqlen;
    p.dim = a->dim;
    p.dstate = a->dstate;
    p.io_bf16 = a->io_dtype == SSM_BF16;
    p.softplus = a->delta_softplus;
    p.x = a->x;
    p.delta = a->delta;
    p.Bm = a->B;
    p.Cm = a->C;
    p.z = a->z;
    p.A = a->A;
    p.Dv = a->D;
    p.bias = a->delta_bias;
    p.h0 = a->h0;
    p.y = a->y;
    p.h_final = a->h_final;
    p.chunk_len = cl;
    p.nchunks = k;
    p.status = a->workspace;
    p.zoh = a->discretization == SSM_DISC_ZOH;
    p.wait_budget = budget;
    p.publish = publish;
    p.ckpt = ckpt;
    p.ckpt_shift = ckpt_shift(a->dstate);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the status word starts at zero
    if (cudaMemsetAsync(a->workspace, 0, kStatusBytes, st) != cudaSuccess) return SSM_ERR_CUDA;
    if (k > 1) {
        char *ws = static_cast<char *>(a->workspace) + kStatusBytes;
        const size_t rows = (size_t)a->batch * k * a->dim;
        p.hloc = reinterpret_cast<float *>(ws);
        p.dsum = reinterpret_cast<float *>(ws + (rows * a->dstate * sizeof(float) + 255) / 256 * 256);
        size_t off, lb;
        ssm::scan_lookback_region(a->batch, a->dim, a->dstate, k, &off, &lb);
        // so do the look-back ticket and flags
        if (cudaMemsetAsync(static_cast<char *>(a->workspace) + off, 0, lb, st) != cudaSuccess)
            return SSM_ERR_CUDA;
        p.ticket = reinterpret_cast<uint32_t *>(static_cast<char *>(a->workspace) + off);
        p.flags = p.ticket + 1;
    }
    return from_cuda(ssm::launch_scan(p, st));
}
}  // namespace

extern "C" {

ssm_status ssm_scan_fwd(const ssm_scan_args *a, ssm_stream_t stream) {
    NvtxRange nvtx("ssm_scan_fwd");
    return scan_fwd_impl(a, stream, ssm::kScanWaitCycles, 1);
}

ssm_status ssm_scan_ckpt_size(const ssm_scan_args *a, int64_t *steps, size_t *bytes) {
    if (!steps || !bytes) return SSM_ERR_INVALID_ARG;
    ssm_status s = check_scan(a, false);
    if (s != SSM_OK) return s;
    *steps = ssm::scan_ckpt_steps(a->dstate);
    *bytes = ckpt_bytes_for(a->batch, a->seqlen, a->dim, a->dstate);
    return SSM_OK;
}

ssm_status ssm_scan_fwd_ckpt(const ssm_scan_args *a, float *ckpt, size_t ckpt_bytes,
                             ssm_stream_t stream) {
    NvtxRange nvtx("ssm_scan_fwd_ckpt");
    ssm_status s = check_scan(a);
    if (s != SSM_OK) return s;
    const size_t need = ckpt_bytes_for(a->batch, a->seqlen, a->dim, a->dstate);
    if (need > 0 && !ckpt) return SSM_ERR_INVALID_ARG;
    if (ckpt_bytes < need) return SSM_ERR_INVALID_ARG;
    if (ckpt && !aligned(ckpt, 16)) return SSM_ERR_ALIGNMENT;
    // the checkpoints are an output: they may overlap no input and no other output
    const size_t e = io_size(a->io_dtype);
    const size_t tok = (size_t)(a->batch * a->seqlen * a->dim) * e;
    const size_t bc = (size_t)(a->batch * a->seqlen * a->dstate) * e;
    const size_t st = (size_t)(a->batch * a->dim * a->dstate) * 4;
    const void *toks[] = {a->x, a->delta, a->z, a->y};
    for (const void *q : toks)
        if (overlaps(ckpt, need, q, tok)) return SSM_ERR_INVALID_ARG;
    if (overlaps(ckpt, need, a->B, bc) || overlaps(ckpt, need, a->C, bc) ||
        overlaps(ckpt, need, a->h0, st) || overlaps(ckpt, need, a->h_final, st) ||
        overlaps(ckpt, need, a->A, (size_t)(a->dim * a->dstate) * 4) ||
        overlaps(ckpt, need, a->workspace, a->workspace_bytes))
        return SSM_ERR_INVALID_ARG;
    return scan_fwd_impl(a, stream, ssm::kScanWaitCycles, 1, need > 0 ? ckpt : nullptr);
}

ssm_status ssm_check_scan_lookback(const ssm_scan_args *a, int64_t budget_cycles,
                                   ssm_stream_t stream) {
    if (budget_cycles < 1 || budget_cycles > ssm::kScanWaitCycles) return SSM_ERR_INVALID_ARG;
    ssm_status s = check_scan(a);
    if (s != SSM_OK) return s;
    int64_t cl;
    int k;
    scan_ws(a, &cl, &k);
    // only a split sequence on the TMA kernel waits on its predecessors
    if (k < 2 || !ssm::scan_tma_sizes_ok(a->io_dtype == SSM_BF16, a->seqlen, a->dim, a->dstate))
        return SSM_ERR_UNSUPPORTED;
    return scan_fwd_impl(a, stream, budget_cycles, 0);
}

ssm_status ssm_ssd_workspace_size(const ssm_ssd_args *a, size_t *bytes) {
    if (!bytes) return SSM_ERR_INVALID_ARG;
    ssm_status s = check_ssd(a, false);
    if (s != SSM_OK) return s;
    *bytes = ssm::ssd_workspace_bytes(ssd_params(a));
    return SSM_OK;
}

ssm_status ssm_ssd_plan(const ssm_ssd_args *a, int32_t *tensor_core) {
    if (!tensor_core) return SSM_ERR_INVALID_ARG;
    ssm_status s = check_ssd(a);
    if (s != SSM_OK) return s;
    *tensor_core = ssm::ssd_tc_eligible(ssd_params(a)) ? 1 : 0;
    return SSM_OK;
}

ssm_status ssm_ssd_chunk_fwd(const ssm_ssd_args *a, ssm_stream_t stream) {
    NvtxRange nvtx("ssm_ssd_chunk_fwd");
    ssm_status s = check_ssd(a);
    if (s != SSM_OK) return s;
    ssm::SSDParams p = ssd_params(a);
    const size_t need = ssm::ssd_workspace_bytes(p);
    if (!a->workspace || a->workspace_bytes < need) return SSM_ERR_WORKSPACE;
    if (a->batch == 0) return SSM_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(a->workspace, 0, ssm::ssd_clear_bytes(p), st);
    if (e != cudaSuccess) return SSM_ERR_CUDA;
    return from_cuda(ssm::launch_ssd(p, st));
}

ssm_status ssm_step_decode(const ssm_decode_args *a, ssm_stream_t stream) {
    NvtxRange nvtx("ssm_step_decode");
    ssm_status s = check_decode(a);
    if (s != SSM_OK) return s;
    if (a->batch * a->dim == 0) return SSM_OK;
    ssm::DecodeParams p{};
    p.batch = a->batch;
    p.dim = a->dim;
    p.dstate = a->dstate;
    p.io_bf16 = a->io_dtype == SSM_BF16;
    p.softplus = a->delta_softplus;
    p.zoh = a->discretization == SSM_DISC_ZOH;
    p.state = a->state;
    p.x = a->x;
    p.delta = a->delta;
    p.Bm = a->B;
    p.Cm = a->C;
    p.z = a->z;
    p.A = a->A;
    p.Dv = a->D;
    p.bias = a->delta_bias;
    p.y = a->y;
    p.status = a->workspace;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (a->workspace && cudaMemsetAsync(a->workspace, 0, ssm::kStatusBytes, st) != cudaSuccess)
        return SSM_ERR_CUDA;
    return from_cuda(ssm::launch_decode(p, st));
}

ssm_status ssm_ssd_step_decode(const ssm_ssd_decode_args *a, ssm_stream_t stream) {
    NvtxRange nvtx("ssm_ssd_step_decode");
    ssm_status s = check_ssd_decode(a);
    if (s != SSM_OK) return s;
    if (a->batch == 0) return SSM_OK;
    ssm::SSDDecodeParams p{};
    p.batch = a->batch;
    p.nheads = a->nheads;
    p.headdim = a->headdim;
    p.ngroups = a->ngroups;
    p.dstate = a->dstate;
    p.io_bf16 = a->io_dtype == SSM_BF16;
    p.softplus = a->delta_softplus;
    p.state = a->state;
    p.x = a->x;
    p.delta = a->delta;
    p.Bm = a->B;
    p.Cm = a->C;
    p.z = a->z;
    p.A = a->A;
    p.Dv = a->D;
    p.bias = a->delta_bias;
    p.y = a->y;
    return from_cuda(ssm::launch_ssd_decode(p, reinterpret_cast<cudaStream_t>(stream)));
}

ssm_status ssm_scan_bwd_workspace_size(const ssm_scan_bwd_args *a, size_t *bytes) {
    if (!bytes) return SSM_ERR_INVALID_ARG;
    ssm_status s = check_scan_bwd(a, false);
    if (s != SSM_OK) return s;
    *bytes = scan_bwd_ws(a);
    return SSM_OK;
}

}  // extern "C"

namespace {
// The backward call; `ckpt` (nullable) holds the state checkpoints a forward pass wrote,
// otherwise the kernel computes them in the workspace.
ssm_status scan_bwd_impl(const ssm_scan_bwd_args *a, ssm_stream_t stream, const float *ckpt,
                         size_t ckpt_bytes) {
    ssm_status s = check_scan_bwd(a);
    if (s != SSM_OK) return s;
    if (ckpt) {
        if (ckpt_bytes < ckpt_bytes_for(a->batch, a->seqlen, a->dim, a->dstate))
            return SSM_ERR_INVALID_ARG;
        if (!aligned(ckpt, 16)) return SSM_ERR_ALIGNMENT;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int64_t rows = a->batch * a->seqlen;
    // the sums start at zero; with no channels or no rows only they are written
    if (a->dim > 0 && a->dA) {
        if (cudaMemsetAsync(a->dA, 0, (size_t)(a->dim * a->dstate) * 4, st) != cudaSuccess)
            return SSM_ERR_CUDA;
    }
    if (a->dD && cudaMemsetAsync(a->dD, 0, (size_t)a->dim * 4, st) != cudaSuccess)
        return SSM_ERR_CUDA;
    if (a->ddelta_bias && cudaMemsetAsync(a->ddelta_bias, 0, (size_t)a->dim * 4, st) != cudaSuccess)
        return SSM_ERR_CUDA;
    if (rows > 0) {
        const size_t bc = (size_t)(rows * a->dstate) * 4;
        if (cudaMemsetAsync(a->dB, 0, bc, st) != cudaSuccess ||
            cudaMemsetAsync(a->dC, 0, bc, st) != cudaSuccess)
            return SSM_ERR_CUDA;
    }
    if (a->batch * a->dim == 0) return SSM_OK;
    if (a->seqlen == 0) {
        // no steps: dh0 = dh_final
        if (a->dh0) {
            const size_t st_bytes = (size_t)(a->batch * a->dim * a->dstate) * 4;
            cudaError_t e = a->dh_final
                                ? cudaMemcpyAsync(a->dh0, a->dh_final, st_bytes,
                                                  cudaMemcpyDeviceToDevice, st)
                                : cudaMemsetAsync(a->dh0, 0, st_bytes, st);
            if (e != cudaSuccess) return SSM_ERR_CUDA;
        }
        return SSM_OK;
    }
    // with given checkpoints the workspace holds only the status word
    const size_t need = ckpt ? ssm::kStatusBytes : scan_bwd_ws(a);
    if (!a->workspace || a->workspace_bytes < need) return SSM_ERR_WORKSPACE;
    if (!aligned(a->workspace, 256)) return SSM_ERR_ALIGNMENT;
    ssm::ScanBwdParams p{};
    p.batch = a->batch;
    p.seqlen = a->seqlen;
    p.dim = a->dim;
    p.dstate = a->dstate;
    p.io_bf16 = a->io_dtype == SSM_BF16;
    p.softplus = a->delta_softplus;
    p.zoh = a->discretization == SSM_DISC_ZOH;
    p.x = a->x;
    p.delta = a->delta;
    p.B = a->B;
    p.C = a->C;
    p.z = a->z;
    p.dy = a->dy;
    p.A = a->A;
    p.D = a->D;
    p.bias = a->delta_bias;
    p.h0 = a->h0;
    p.dh_final = a->dh_final;
    p.dx = a->dx;
    p.ddelta = a->ddelta;
    p.dz = a->dz;
    p.dA = a->dA;
    p.dB = a->dB;
    p.dC = a->dC;
    p.dD = a->dD;
    p.ddelta_bias = a->ddelta_bias;
    p.dh0 = a->dh0;
    p.ckpt = ckpt ? const_cast<float *>(ckpt)
                  : reinterpret_cast<float *>(static_cast<char *>(a->workspace) + ssm::kStatusBytes);
    p.ckpt_given = ckpt ? 1 : 0;
    p.status = a->workspace;
    if (cudaMemsetAsync(a->workspace, 0, ssm::kStatusBytes, st) != cudaSuccess) return SSM_ERR_CUDA;
    return from_cuda(ssm::launch_scan_bwd(p, st));
}
}  // namespace

extern "C" {

ssm_status ssm_scan_bwd(const ssm_scan_bwd_args *a, ssm_stream_t stream) {
    NvtxRange nvtx("ssm_scan_bwd");
    return scan_bwd_impl(a, stream, nullptr, 0);
}

ssm_status ssm_scan_bwd_ckpt(const ssm_scan_bwd_args *a, const float *ckpt, size_t ckpt_bytes,
                             ssm_stream_t stream) {
    NvtxRange nvtx("ssm_scan_bwd_ckpt");
    if (!ckpt) return SSM_ERR_INVALID_ARG;
    return scan_bwd_impl(a, stream, ckpt, ckpt_bytes);
}

ssm_status ssm_conv1d(const ssm_conv1d_args *a, ssm_stream_t stream) {
    NvtxRange nvtx("ssm_conv1d");
    ssm_status s = check_conv1d(a);
    if (s != SSM_OK) return s;
    if (a->batch * a->seqlen * a->dim == 0) return SSM_OK;
    ssm::Conv1dParams p{};
    p.batch = a->batch;
    p.seqlen = a->seqlen;
    p.dim = a->dim;
    p.width = a->width;
    p.io_bf16 = a->io_dtype == SSM_BF16;
    p.silu = a->silu;
    p.x = a->x;
    p.x_prev = a->x_prev;
    p.weight = a->weight;
    p.bias = a->bias;
    p.out = a->out;
    p.status = a->workspace;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (a->workspace && cudaMemsetAsync(a->workspace, 0, ssm::kStatusBytes, st) != cudaSuccess)
        return SSM_ERR_CUDA;
    return from_cuda(ssm::launch_conv1d(p, st));
}

ssm_status ssm_read_device_status(const void *workspace, ssm_stream_t stream,
                                  ssm_status *device_status) {
    if (!workspace || !device_status) return SSM_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return SSM_ERR_CUDA;
    int32_t code = 0;
    if (cudaMemcpy(&code, workspace, sizeof(code), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SSM_ERR_CUDA;
    *device_status = static_cast<ssm_status>(code);
    return SSM_OK;
}

}  // extern "C"
