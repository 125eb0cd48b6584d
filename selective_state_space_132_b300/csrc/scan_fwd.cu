// Selective (S6) scan, forward.
//
// What it computes (tildalice.io Mamba review, sections "Selection Mechanism",
// "Δ의 직관적 이해" and "Mamba 블록 아키텍처"; D skip from the yongggg review,
// section "State Space Model"), per batch b and channel d:
//   dl_t = softplus(delta_t + bias_d)
//   h_t  = exp(dl_t A_d) (.) h_{t-1} + (dl_t x_t) B_t        (N states, diagonal A)
//   y_t  = (C_t . h_t + D_d x_t) * silu(z_t)
// The discretised Abar and Bbar x and every h_t live only in registers: HBM sees
// x, delta, z, B, C once and y once ("hardware-aware algorithm" / kernel fusion
// of the review pages; the B300 design below is our own).
//
// B300 mapping
//   * A thread block owns 32 channels of one batch row and one time chunk.  Each
//     channel's N states are split over LPC adjacent lanes, NS states per lane
//     (N <= 4: 1 lane ... N <= 64: 8 lanes), so one warp holds 32 / LPC channels.
//     The recurrence runs sequentially in time inside each lane: it is the
//     work-efficient order (one exp, two FMA and one MUL per state update), and
//     the parallelism comes from the B * D * LPC independent lanes.
//   * Time is walked in tiles of 32 steps.  For each tile a prologue turns the
//     raw delta/x into fp32 dl and dl*x rows in shared memory (softplus done once
//     per (t, d), not once per lane); the scan reads them with 16-byte loads; the
//     per-lane partial readouts go to shared memory and an epilogue sums them,
//     adds D x, applies the gate and writes y coalesced.  The next tile's raw
//     inputs are fetched into registers while the current tile is scanned.
//   * Long sequences are cut into K time chunks processed by different blocks.
//     A first kernel (kSummary) scans chunks 0..K-2 from a zero state and keeps
//     only each chunk's end state and sum of steps; the output kernel starts
//     chunk c from h0 folded through the summaries of chunks < c:
//         h <- exp(A * sum_dl(c')) h + h_end(c')
//     which is the associative combine of the scan ("병렬 스캔") applied to whole
//     chunks.  Exact up to rounding.
#include "common.cuh"
#include "internal.h"

#include <algorithm>

namespace ssm {
namespace {

constexpr int kTT = 32;  // time steps per shared-memory tile
constexpr int kDT = 32;  // channels per thread block
constexpr int kRowF = kTT + 4;  // floats per per-channel row (16-byte aligned, conflict-free)

template <int LPC> struct YpStride {
    static constexpr int base = LPC * kRowF;
    static constexpr int value = ((base / 4) % 2 == 0) ? base + 4 : base;
};

template <int NS, int LPC, bool kSummary> struct ScanSmem {
    static constexpr int NP = NS * LPC;
    static constexpr int dl = 0;
    static constexpr int dx = dl + kDT * kRowF;
    static constexpr int Bs = dx + kDT * kRowF;
    static constexpr int Cs = Bs + kTT * NP;
    static constexpr int xs = Cs + (kSummary ? 0 : kTT * NP);
    static constexpr int zs = xs + (kSummary ? 0 : kDT * kRowF);
    static constexpr int yp = zs + (kSummary ? 0 : kDT * kRowF);
    static constexpr int total = yp + (kSummary ? 0 : kDT * YpStride<LPC>::value);
    static constexpr size_t bytes = sizeof(float) * total;
};

template <typename TIO, int NS, int LPC, bool kSummary, bool kFast, bool kCkpt>
__global__ void __launch_bounds__(kDT * LPC, 512 / (kDT * LPC)) scan_kernel(ScanParams p) {
    constexpr int NT = kDT * LPC;
    constexpr int NP = NS * LPC;
    constexpr int kQuadSlots = NT / kDT;  // threads per channel in prologue/epilogue
    constexpr int kQuadIters = (kTT / 4) / kQuadSlots;
    static_assert((kTT / 4) % kQuadSlots == 0, "tile/lanes mismatch");
    constexpr int kRawBC = (kTT * NP + NT - 1) / NT;
    constexpr int kYS = YpStride<LPC>::value;
    using SM = ScanSmem<NS, LPC, kSummary>;

    extern __shared__ __align__(16) float smem[];
    float *s_dl = smem + SM::dl;
    float *s_dx = smem + SM::dx;
    float *s_B = smem + SM::Bs;
    float *s_C = smem + SM::Cs;
    float *s_x = smem + SM::xs;
    float *s_z = smem + SM::zs;
    float *s_yp = smem + SM::yp;

    const TIO *__restrict__ gx = static_cast<const TIO *>(p.x);
    const TIO *__restrict__ gdl = static_cast<const TIO *>(p.delta);
    const TIO *__restrict__ gz = static_cast<const TIO *>(p.z);
    const TIO *__restrict__ gB = static_cast<const TIO *>(p.Bm);
    const TIO *__restrict__ gC = static_cast<const TIO *>(p.Cm);
    TIO *__restrict__ gy = static_cast<TIO *>(p.y);

    const int tid = threadIdx.x;
    const int64_t D = p.dim, L = p.seqlen;
    const int N = static_cast<int>(p.dstate);
    const int K = p.nchunks;
    DeviceStatus *status = static_cast<DeviceStatus *>(p.status);
    (void)status;
    const int b = blockIdx.y;
    const int c = blockIdx.z;
    const int d0 = blockIdx.x * kDT;

    // scan role: channel ch, lane j owns states j*NS .. j*NS+NS-1
    const int ch = tid / LPC, j = tid % LPC;
    const int64_t d = d0 + ch;
    const bool dval = d < D;
    // prologue / epilogue role: channel pd, quads pq + kQuadSlots*it
    const int pd = tid % kDT, pq = tid / kDT;
    const int64_t pdd = d0 + pd;
    const bool pdval = pdd < D;
    const float pbias = (pdval && p.bias) ? p.bias[pdd] : 0.f;
    const float pD = (pdval && p.Dv) ? p.Dv[pdd] : 0.f;
    const bool has_z = gz != nullptr;

    const int64_t t_begin = static_cast<int64_t>(c) * p.chunk_len;
    const int64_t t_end = min(L, t_begin + p.chunk_len);

    float a2[NS], h[NS], ia[NS];
#pragma unroll
    for (int k = 0; k < NS; ++k) {
        const int n = j * NS + k;
        const bool v = dval && n < N;
        const float an = v ? p.A[d * N + n] : 0.f;
        a2[k] = scale_A<kFast>(an);
        ia[k] = an != 0.f ? 1.f / an : 0.f;
        h[k] = (!kSummary && v && p.h0) ? p.h0[(b * D + d) * N + n] : 0.f;
    }
    if (!kSummary) {
        // fold the summaries of the chunks before this one into the initial state
        for (int cc = 0; cc < c; ++cc) {
            const int64_t row = (static_cast<int64_t>(b) * K + cc) * D + d;
            const float S = dval ? p.dsum[row] : 0.f;
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                const int n = j * NS + k;
                const float he = (dval && n < N) ? p.hloc[row * N + n] : 0.f;
                h[k] = fmaf(decay<kFast>(S, a2[k]), h[k], he);
            }
        }
    }
    float dsum_acc = 0.f;
    // checkpoints along the whole sequence (the backward pass's time tiles)
    const int64_t ck_tiles = kCkpt ? (L + (int64_t(1) << p.ckpt_shift) - 1) >> p.ckpt_shift : 0;
    (void)ck_tiles;

    // raw-input prefetch registers for one tile
    TIO rx[kQuadIters * 4], rdl[kQuadIters * 4], rz[kQuadIters * 4];
    TIO rB[kRawBC], rC[kRawBC];
    auto fetch = [&](int64_t t0) {
#pragma unroll
        for (int it = 0; it < kQuadIters; ++it) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int tl = 4 * (pq + kQuadSlots * it) + i;
                const int64_t t = t0 + tl;
                const int r = it * 4 + i;
                if (pdval && t < t_end) {
                    const int64_t off = (static_cast<int64_t>(b) * L + t) * D + pdd;
                    rx[r] = gx[off];
                    rdl[r] = gdl[off];
                    if (!kSummary && has_z) rz[r] = gz[off];
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kRawBC; ++r) {
            const int e = tid + r * NT;
            const int tl = e / NP, n = e % NP;
            const int64_t t = t0 + tl;
            if (e < kTT * NP && n < N && t < t_end) {
                const int64_t off = (static_cast<int64_t>(b) * L + t) * N + n;
                rB[r] = gB[off];
                if (!kSummary) rC[r] = gC[off];
            }
        }
    };

    if (t_begin < t_end) fetch(t_begin);

    for (int64_t t0 = t_begin; t0 < t_end; t0 += kTT) {
        // ---------------- prologue: dl, dl*x (and x, z) rows; B, C tile
#pragma unroll
        for (int it = 0; it < kQuadIters; ++it) {
            const int tq = 4 * (pq + kQuadSlots * it);
            float vdl[4], vdx[4], vx[4], vz[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = it * 4 + i;
                const bool v = pdval && (t0 + tq + i) < t_end;
                const float xv = v ? Io<TIO>::to_f(rx[r]) : 0.f;
                const float dlv = v ? step_size<kFast>(Io<TIO>::to_f(rdl[r]), pbias, p.softplus)
                                    : 0.f;
                vdl[i] = dlv;
                vdx[i] = p.zoh ? xv : dlv * xv;  // zoh: the coefficient multiplies x later
                vx[i] = xv;
                vz[i] = (v && has_z && !kSummary) ? Io<TIO>::to_f(rz[r]) : 0.f;
            }
            *reinterpret_cast<float4 *>(s_dl + pd * kRowF + tq) =
                make_float4(vdl[0], vdl[1], vdl[2], vdl[3]);
            *reinterpret_cast<float4 *>(s_dx + pd * kRowF + tq) =
                make_float4(vdx[0], vdx[1], vdx[2], vdx[3]);
            if (!kSummary) {
                *reinterpret_cast<float4 *>(s_x + pd * kRowF + tq) =
                    make_float4(vx[0], vx[1], vx[2], vx[3]);
                *reinterpret_cast<float4 *>(s_z + pd * kRowF + tq) =
                    make_float4(vz[0], vz[1], vz[2], vz[3]);
            }
        }
#pragma unroll
        for (int r = 0; r < kRawBC; ++r) {
            const int e = tid + r * NT;
            if (e < kTT * NP) {
                const int tl = e / NP, n = e % NP;
                const bool v = n < N && (t0 + tl) < t_end;
                s_B[e] = v ? Io<TIO>::to_f(rB[r]) : 0.f;
                if (!kSummary) s_C[e] = v ? Io<TIO>::to_f(rC[r]) : 0.f;
            }
        }
        __syncthreads();

        // prefetch the next tile while this one is scanned
        if (t0 + kTT < t_end) fetch(t0 + kTT);

        // ---------------- scan: NS states per lane, sequential in time
        const float *rowdl = s_dl + ch * kRowF;
        const float *rowdx = s_dx + ch * kRowF;
#pragma unroll
        for (int tq = 0; tq < kTT; tq += 4) {
            const float4 dl4 = *reinterpret_cast<const float4 *>(rowdl + tq);
            const float4 dx4 = *reinterpret_cast<const float4 *>(rowdx + tq);
            const float dlq[4] = {dl4.x, dl4.y, dl4.z, dl4.w};
            const float dxq[4] = {dx4.x, dx4.y, dx4.z, dx4.w};
            float yq[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if constexpr (kCkpt && !kSummary) {
                    // the state before step t0 + tq, at every checkpoint step (at least
                    // four steps apart, so only i = 0 can have one)
                    const int64_t t = t0 + tq + i;
                    if (i == 0 && (tq & ((1 << p.ckpt_shift) - 1)) == 0 && dval && t < t_end &&
                        in_bounds((t >> p.ckpt_shift) < ck_tiles && b < p.batch, status, 111)) {
                        float *ck = p.ckpt + ((b * ck_tiles + (t >> p.ckpt_shift)) * D + d) * N;
#pragma unroll
                        for (int k = 0; k < NS; ++k)
                            if (j * NS + k < N) ck[j * NS + k] = h[k];
                    }
                }
                float bv[NS], cv[NS];
#pragma unroll
                for (int k4 = 0; k4 < NS; k4 += 4) {
                    const float4 b4 =
                        *reinterpret_cast<const float4 *>(s_B + (tq + i) * NP + j * NS + k4);
                    bv[k4] = b4.x; bv[k4 + 1] = b4.y; bv[k4 + 2] = b4.z; bv[k4 + 3] = b4.w;
                    if (!kSummary) {
                        const float4 c4 =
                            *reinterpret_cast<const float4 *>(s_C + (tq + i) * NP + j * NS + k4);
                        cv[k4] = c4.x; cv[k4 + 1] = c4.y; cv[k4 + 2] = c4.z; cv[k4 + 3] = c4.w;
                    }
                }
                float acc = 0.f;
#pragma unroll
                for (int k = 0; k < NS; ++k) {
                    const float a = decay<kFast>(dlq[i], a2[k]);
                    float w = dxq[i] * bv[k];
                    if (p.zoh) {
                        const float vn = dlq[i] * a2[k] * (kFast ? kLn2 : 1.f);
                        w *= zoh_coef<kFast>(dlq[i], vn, a, ia[k]);
                    }
                    h[k] = fmaf(a, h[k], w);
                    if (!kSummary) acc = fmaf(cv[k], h[k], acc);
                }
                yq[i] = acc;
                if (kSummary) dsum_acc += dlq[i];
            }
            if (!kSummary)
                *reinterpret_cast<float4 *>(s_yp + ch * kYS + j * kRowF + tq) =
                    make_float4(yq[0], yq[1], yq[2], yq[3]);
        }
        __syncthreads();

        // ---------------- epilogue: reduce lanes, D skip, gate, store y
        if (!kSummary) {
#pragma unroll
            for (int it = 0; it < kQuadIters; ++it) {
                const int tq = 4 * (pq + kQuadSlots * it);
                float4 acc = *reinterpret_cast<const float4 *>(s_yp + pd * kYS + tq);
#pragma unroll
                for (int jj = 1; jj < LPC; ++jj) {
                    const float4 v = *reinterpret_cast<const float4 *>(s_yp + pd * kYS +
                                                                       jj * kRowF + tq);
                    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
                }
                const float4 x4 = *reinterpret_cast<const float4 *>(s_x + pd * kRowF + tq);
                const float4 z4 = *reinterpret_cast<const float4 *>(s_z + pd * kRowF + tq);
                const float av[4] = {acc.x, acc.y, acc.z, acc.w};
                const float xv[4] = {x4.x, x4.y, x4.z, x4.w};
                const float zv[4] = {z4.x, z4.y, z4.z, z4.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int64_t t = t0 + tq + i;
                    if (pdval && t < t_end && in_bounds(t < L && b < p.batch, status, 112)) {
                        float out = fmaf(pD, xv[i], av[i]);
                        if (has_z) out *= silu<kFast>(zv[i]);
                        gy[(static_cast<int64_t>(b) * L + t) * D + pdd] = Io<TIO>::from_f(out);
                    }
                }
            }
            __syncthreads();
        }
    }

    if (kSummary) {
        const int64_t row = (static_cast<int64_t>(b) * K + c) * D + d;
        if (dval && in_bounds(row < p.batch * K * D && c < K - 1, status, 113)) {
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                const int n = j * NS + k;
                if (n < N) p.hloc[row * N + n] = h[k];
            }
            if (j == 0) p.dsum[row] = dsum_acc;
        }
    } else if (c == K - 1 && p.h_final && dval && in_bounds(b < p.batch, status, 114)) {
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            const int n = j * NS + k;
            if (n < N) p.h_final[(static_cast<int64_t>(b) * D + d) * N + n] = h[k];
        }
    }
}

template <typename TIO, int NS, int LPC, bool kSummary, bool kCkpt = false>
cudaError_t launch_one(const ScanParams &p, int nchunks_grid, cudaStream_t stream) {
    constexpr bool kFast = std::is_same<TIO, __nv_bfloat16>::value;
    auto kern = scan_kernel<TIO, NS, LPC, kSummary, kFast, kCkpt>;
    const size_t smem = ScanSmem<NS, LPC, kSummary>::bytes;
    if (smem > 48 * 1024) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    dim3 grid(static_cast<unsigned>((p.dim + kDT - 1) / kDT), static_cast<unsigned>(p.batch),
              static_cast<unsigned>(nchunks_grid));
    kern<<<grid, kDT * LPC, smem, stream>>>(p);
    return cudaGetLastError();
}

template <typename TIO, int NS, int LPC>
cudaError_t launch_pair(const ScanParams &p, cudaStream_t stream) {
    if (p.nchunks > 1) {
        cudaError_t e = launch_one<TIO, NS, LPC, true>(p, p.nchunks - 1, stream);
        if (e != cudaSuccess) return e;
    }
    // the output pass writes the backward pass's state checkpoints when asked to
    return p.ckpt ? launch_one<TIO, NS, LPC, false, true>(p, p.nchunks, stream)
                  : launch_one<TIO, NS, LPC, false, false>(p, p.nchunks, stream);
}

template <typename TIO> cudaError_t launch_typed(const ScanParams &p, cudaStream_t stream) {
    const int64_t N = p.dstate;
    if (N <= 4) return launch_pair<TIO, 4, 1>(p, stream);
    if (N <= 8) return launch_pair<TIO, 4, 2>(p, stream);
    if (N <= 16) return launch_pair<TIO, 4, 4>(p, stream);
    if (N <= 32) return launch_pair<TIO, 4, 8>(p, stream);
    return launch_pair<TIO, 8, 8>(p, stream);
}

int lanes_for(int64_t N) { return N <= 4 ? 1 : N <= 8 ? 2 : N <= 16 ? 4 : 8; }

}  // namespace

int device_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0) {
        cudaGetLastError();
        return 148;  // B300
    }
    return sms;
}

void scan_plan(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int64_t time_chunk,
               int tma_blocks_per_sm, int64_t *chunk_len, int *nchunks) {
    int64_t cl;
    if (time_chunk > 0) {
        cl = (time_chunk + kTT - 1) / kTT * kTT;
    } else {
        // Each extra chunk costs a summary pass over that chunk (most of a scan of it),
        // so the sequence is split only when its chains alone cannot fill the GPU.
        //  * TMA kernel: a grid of at least half a wave of resident blocks is left
        //    whole (the 130M-layer shape, 384 blocks for 592 slots: 200 us whole,
        //    250-262 us split 2-8 ways).  A smaller grid is split into about six waves
        //    of blocks, so that the last wave's tail is short (long-context shape, 64
        //    blocks per chunk: 9 chunks (one wave) 2.85 ms, 32 chunks 2.66 ms, 64
        //    chunks 2.65 ms).
        //  * general kernel: about eight warps per SM.
        // Chunks stay at least 1024 steps long.
        int64_t k;
        if (tma_blocks_per_sm > 0) {
            const int64_t per_chunk = batch * ((dim + 31) / 32);
            const int64_t slots = static_cast<int64_t>(device_sm_count()) * tma_blocks_per_sm;
            k = (per_chunk <= 0 || 2 * per_chunk >= slots) ? 1
                                                           : (6 * slots + per_chunk - 1) / per_chunk;
        } else {
            const int64_t warps = batch * ((dim + kDT - 1) / kDT) * lanes_for(dstate);
            const int64_t target = static_cast<int64_t>(device_sm_count()) * 8;
            k = warps > 0 ? (target + warps - 1) / warps : 1;
        }
        const int64_t kmax = std::max<int64_t>(1, seqlen / 1024);
        k = std::max<int64_t>(1, std::min(k, kmax));
        cl = (seqlen + k - 1) / k;
        cl = std::max<int64_t>(kTT, (cl + kTT - 1) / kTT * kTT);
    }
    int64_t k = seqlen > 0 ? (seqlen + cl - 1) / cl : 1;
    *chunk_len = cl;
    *nchunks = static_cast<int>(std::max<int64_t>(1, k));
}

// Workspace: the device status word, then (when the sequence is split) the chunk end
// states (B, K, D, N) and step sums (B, K, D), then the look-back ticket and flags
// (1 + B K ceil(D / 32) words), each part on a 256-byte boundary.
void scan_lookback_region(int64_t batch, int64_t dim, int64_t dstate, int nchunks,
                          size_t *offset, size_t *bytes) {
    *offset = 0;
    *bytes = 0;
    if (nchunks <= 1) return;
    const size_t rows = static_cast<size_t>(batch) * nchunks * dim;
    *offset = kStatusBytes + (rows * dstate * sizeof(float) + 255) / 256 * 256 +
              (rows * sizeof(float) + 255) / 256 * 256;
    const size_t words = 1 + static_cast<size_t>(batch) * nchunks * ((dim + 31) / 32);
    *bytes = (words * 4 + 255) / 256 * 256;
}

size_t scan_workspace_bytes(int64_t batch, int64_t dim, int64_t dstate, int nchunks) {
    size_t bytes = kStatusBytes;  // device status word
    if (nchunks > 1) {
        size_t off, lb;
        scan_lookback_region(batch, dim, dstate, nchunks, &off, &lb);
        bytes = off + lb;
    }
    return bytes;
}

cudaError_t launch_scan(const ScanParams &p, cudaStream_t stream) {
    const void *ptrs[] = {p.x, p.delta, p.Bm, p.Cm, p.z, p.y};
    if (scan_tma_sizes_ok(p.io_bf16, p.seqlen, p.dim, p.dstate) && scan_tma_pointers_ok(ptrs, 6))
        return launch_scan_tma(p, stream);
    return p.io_bf16 ? launch_typed<__nv_bfloat16>(p, stream) : launch_typed<float>(p, stream);
}

}  // namespace ssm
