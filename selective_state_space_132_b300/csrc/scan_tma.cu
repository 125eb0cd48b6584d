// Selective (S6) scan, forward: the TMA-staged fast path.
//
// What it computes (tildalice.io Mamba review, sections "Selection Mechanism",
// "Δ의 직관적 이해" and "Mamba 블록 아키텍처"; the D skip from the yongggg review,
// section "State Space Model"), per batch b and channel d:
//   dl_t = softplus(delta_t + bias_d)
//   h_t  = exp(dl_t A_d) (.) h_{t-1} + (dl_t x_t) B_t        (N states, diagonal A)
//   y_t  = (C_t . h_t + D_d x_t) * silu(z_t)
// Abar, Bbar x and every h_t stay in registers; HBM sees each input once and y
// once (the pages' kernel-fusion idea, "하드웨어 인식 알고리즘"; the design here is
// our own for B300).
//
// B300 mapping
//   * A block owns the 32 channels of one token-tile row (64 bytes of bf16, 128 of
//     fp32) of one batch row: WPC warps of CPW = 32 / LPC channels each.  Each
//     channel's N states are split over LPC adjacent lanes, NS states per lane.  The
//     recurrence runs in time order inside each lane (one exp, one packed fp32x2
//     product and one packed FMA per pair of states).  At the 130M-layer shape (N 16,
//     LPC 4) that is 384 blocks of 4 warps, 3 blocks per SM.
//   * Inputs arrive through a two-stage TMA pipeline: 3-D tensor maps over
//     (channel, time, batch) give boxes of 32 channels x 32 steps for x, delta and z
//     (64/128-byte swizzle) and N states x 32 steps for B and C; boxes past the end
//     of a sequence are zero-filled by the TMA unit.  One thread issues the copies,
//     every thread waits on the stage's mbarrier (bounded by a clock budget).
//   * Per 32-step tile: (1) a prologue in which lane t turns row t of its warp's
//     channels into fp32 (dl, dl*x) pairs (softplus computed once per (t, d));
//     (2) the scan, reading (dl, dl*x) with 16-byte loads and B, C straight from the
//     TMA tile (bf16 pairs widened in registers, or fp32) as broadcast loads;
//     per-lane partial readouts go to shared memory; (3) an epilogue in which lane t
//     sums the partials of row t, adds D x, applies the gate, rounds to the I/O type
//     and writes a y tile that one TMA store sends to HBM.
//   * The bound on B300 is the shared-memory to register traffic (B, C and the
//     (dl, dl*x) pairs delivered to every lane), not HBM.
//   * Long sequences are cut into K time chunks (blockIdx.z).  A summary pass
//     (kSummary) scans chunks 0..K-2 from a zero state and keeps each chunk's end
//     state and step sum; the output pass folds the summaries of earlier chunks
//     into its initial state, h <- exp(A * sum dl) h + h_end: the associative
//     combine of the parallel scan ("병렬 스캔") applied to whole chunks.
#include <cudaTypedefs.h>

#include "../../include/ssm.h"

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tma_host.cuh"

namespace ssm {
namespace {

using ptx::f2;

constexpr int kT = 32;       // time steps per tile (one per lane in prologue/epilogue)
#ifndef SSM_SCAN_STAGES
#define SSM_SCAN_STAGES 2
#endif
constexpr int kStages = SSM_SCAN_STAGES;  // TMA pipeline depth
#ifndef SSM_SCAN_UNROLL
#define SSM_SCAN_UNROLL 4
#endif
constexpr int kU = SSM_SCAN_UNROLL;  // time steps per ILP block of the scan loop
// state checkpoints (every 4 to 32 steps) fall on the first step of an ILP block
static_assert(kU <= 4 && kT % kU == 0, "checkpoint steps must be multiples of kU");
#ifndef SSM_SCAN_LOOKBACK
#define SSM_SCAN_LOOKBACK 1
#endif
// a sequence split over time chunks runs in one launch (look-back carry) or two
constexpr bool kScanLookback = SSM_SCAN_LOOKBACK != 0;
#ifndef SSM_SCAN_SPLIT_RED
#define SSM_SCAN_SPLIT_RED 1
#endif
// the output pass of a split sequence adds the partial readouts of a channel's lanes
// with shuffles (smaller shared memory, more resident blocks)
constexpr bool kSplitRed = SSM_SCAN_SPLIT_RED != 0;

__host__ __device__ constexpr int align1k(int v) { return (v + 1023) / 1024 * 1024; }

// Shared-memory layout of one block: WPC warps, each owning CPW = 32 / LPC channels;
// the block's CPB = WPC * CPW channels form one token-tile row of ROWB bytes.
template <typename TIO, int NS, int LPC, int WPC, bool kSummary, bool kRed = false> struct Layout {
    static constexpr int CPW = 32 / LPC;
    static constexpr int CPB = CPW * WPC;
    static constexpr int N = NS * LPC;
    static constexpr int E = sizeof(TIO);
    static constexpr int ROWB = CPB * E;       // 32, 64 or 128 bytes (swizzle span)
    static constexpr int kTok = kT * ROWB;     // bytes of one x / delta / z tile
    static constexpr int kBC = kT * N * E;     // bytes of one B or C tile
    // bf16 B/C are read as bf16 pairs straight from the TMA tile and widened in
    // registers (half the shared-memory bytes of fp32 copies); fp32 B/C as they are
    static constexpr bool kRawBC = E == 2;
    // one pipeline stage: x, delta, z, B, C (no z, C in the summary pass)
    static constexpr int s_x = 0;
    static constexpr int s_dl = s_x + align1k(kTok);
    static constexpr int s_z = s_dl + align1k(kTok);
    static constexpr int s_B = s_z + (kSummary ? 0 : align1k(kTok));
    static constexpr int s_C = s_B + align1k(kBC);
    static constexpr int stage = s_C + (kSummary ? 0 : align1k(kBC));
    // bytes one stage receives (z only when a gate is given)
    __host__ __device__ static constexpr int tx_bytes(bool gate) {
        return (kSummary ? 2 : (gate ? 3 : 2)) * kTok + (kSummary ? 1 : 2) * kBC;
    }
    // fp32 (dl, dl x) pairs, one row of 2 kT floats per channel (16-byte aligned rows)
    static constexpr int kDlxRow = 2 * kT + 4;
    static constexpr int o_dlx = kStages * stage;
    // per warp: LPC slots of partial readouts [slot][t][channel], t-stride CPW + 4
    // (conflict-free row reads) and slot stride = 8 mod 32 (conflict-free writes);
    // with kRed the LPC lanes of a channel add their partials with shuffles first and
    // one slot holds the sums (a quarter of the shared memory, more blocks per SM)
    static constexpr int kSlots = kRed ? 1 : LPC;
    static constexpr int kPartT = CPW + 4;
    static constexpr int kPart = (kT * kPartT + 31) / 32 * 32 + 8;
    static constexpr int o_part = o_dlx + align1k(CPB * kDlxRow * 4);
    static constexpr int o_y = o_part + (kSummary ? 0 : align1k(WPC * kSlots * kPart * 4));
    static constexpr int o_bar = o_y + (kSummary ? 0 : 2 * align1k(kTok));
    // summary pass with bf16 I/O: B widened to fp32 once per tile by the block
    static constexpr int o_bf32 = align1k(o_bar + kStages * 8);
    static constexpr int bytes = (kSummary && E == 2 ? o_bf32 + kT * N * 4 : o_bar + kStages * 8) +
                                 1024;  // + slack to align the base
};

struct TmaMaps {
    CUtensorMap x, dl, z, B, C, y;
};

// Byte offset of 16-byte chunk `q` of row `t` in a token tile: the TMA swizzle
// of a ROWB-byte row (32/64/128-byte mode) XORs the chunk index with address bits 7+.
template <int ROWB> __device__ __forceinline__ int tok_chunk(int t, int q) {
    return t * ROWB + ((q ^ ((t * ROWB >> 7) & (ROWB / 16 - 1))) << 4);
}

// 16-byte chunk of 8 bf16 or 4 fp32 values as floats.
template <typename TIO> struct Chunk;
template <> struct Chunk<float> {
    static constexpr int EC = 4;
    static __device__ __forceinline__ void load(const unsigned char *p, float (&v)[4]) {
        const float4 q = *reinterpret_cast<const float4 *>(p);
        v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    }
    static __device__ __forceinline__ void store(unsigned char *p, const float (&v)[4]) {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};
template <> struct Chunk<__nv_bfloat16> {
    static constexpr int EC = 8;
    static __device__ __forceinline__ void load(const unsigned char *p, float (&v)[8]) {
        const uint4 q = *reinterpret_cast<const uint4 *>(p);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const f2 e = ptx::bf2_to_f2(w[i]);
            v[2 * i] = e.x;
            v[2 * i + 1] = e.y;
        }
    }
    static __device__ __forceinline__ void store(unsigned char *p, const float (&v)[8]) {
        uint4 q;
        q.x = ptx::f2_to_bf2(v[0], v[1]);
        q.y = ptx::f2_to_bf2(v[2], v[3]);
        q.z = ptx::f2_to_bf2(v[4], v[5]);
        q.w = ptx::f2_to_bf2(v[6], v[7]);
        *reinterpret_cast<uint4 *>(p) = q;
    }
};

// Decay factors of a pair of states: exp(dl * A) (accurate) or 2^(dl * A log2 e).
template <bool kFast> __device__ __forceinline__ f2 decay2(float dl, f2 a) {
    const f2 v = ptx::mul2(f2{dl, dl}, a);
    if (kFast) return f2{ex2_approx(v.x), ex2_approx(v.y)};
    return f2{expf(v.x), expf(v.y)};
}

// One pass over chunk c of batch row b for the block's channel slab (channels d0 ..
// d0 + CPB - 1): the summary pass (kSummary: from a zero state, keeping the chunk's end
// state and step sum) or the output pass (from h0 folded through the summaries of the
// chunks before c).  kLB selects the single-launch form: the output pass first acquires
// the summaries of the earlier chunks (each published by its block with a release
// store) and the summary pass publishes its own.  Returns false after a bounded wait
// gave up (the status word then says so).
template <typename TIO, int NS, int LPC, int WPC, bool kSummary, bool kZoh, bool kLB,
          bool kRed, bool kCkpt>
__device__ __forceinline__ bool chunk_pass(const TmaMaps &maps, const ScanParams &p, int b,
                                           int c, int d0, int slab) {
    using LY = Layout<TIO, NS, LPC, WPC, kSummary, kRed>;
    using CK = Chunk<TIO>;
    constexpr int CPW = LY::CPW, CPB = LY::CPB, N = LY::N, ROWB = LY::ROWB;
    constexpr int EC = CK::EC;                  // elements per 16-byte chunk
    constexpr int QW = CPW / EC;                // chunks of a warp's channels in one row
    constexpr bool kFast = std::is_same<TIO, __nv_bfloat16>::value;
    static_assert(NS % 2 == 0 && CPW % EC == 0, "layout");
    static_assert(ROWB == 32 || ROWB == 64 || ROWB == 128, "token rows must match a TMA swizzle");

    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + LY::o_bar);
    float *dlx = reinterpret_cast<float *>(smem + LY::o_dlx);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int64_t D = p.dim, L = p.seqlen;
    const int K = p.nchunks;
    const bool has_z = p.z != nullptr;
    DeviceStatus *status = static_cast<DeviceStatus *>(p.status);
    float *part = reinterpret_cast<float *>(smem + LY::o_part) + warp * LY::kSlots * LY::kPart;
    const int nslabs = static_cast<int>((D + CPB - 1) / CPB);

    const int64_t t_begin = static_cast<int64_t>(c) * p.chunk_len;
    const int64_t t_end = min(L, t_begin + p.chunk_len);
    const int ntiles = static_cast<int>((t_end - t_begin + kT - 1) / kT);

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) ptx::mbar_init(&bars[s], 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    // the barriers are invalidated when the pass ends, so that the block's next pass
    // can reuse their shared memory
    auto release_barriers = [&]() {
        __syncthreads();
        if (tid == 0)
            for (int s = 0; s < kStages; ++s) ptx::mbar_inval(&bars[s]);
        __syncthreads();
    };
    if (kLB && !kSummary && c > 0) {
        // acquire the summaries of chunks 0 .. c - 1 of this slab (their blocks took
        // earlier tickets, so they have started and publish before they wait on anything)
        int late = 0;
        if (tid == 0) {
            const long long t0 = clock64();
            for (int cc = 0; cc < c && !late; ++cc) {
                const uint32_t *f = p.flags + (static_cast<int64_t>(b) * K + cc) * nslabs + slab;
                while (ptx::ld_acquire_u32(f) == 0u) {
                    if (clock64() - t0 > p.wait_budget) {
                        late = 1;
                        break;
                    }
                    __nanosleep(128);
                }
            }
        }
        if (__syncthreads_or(late)) {
            if (tid == 0) report_status(status, SSM_ERR_TIMEOUT, 13);
            release_barriers();
            return false;  // nothing was issued yet
        }
    }

    auto issue = [&](int tile) {  // thread 0 only
        const int s = tile % kStages;
        unsigned char *st = smem + s * LY::stage;
        const int t0 = static_cast<int>(t_begin + static_cast<int64_t>(tile) * kT);
        // the channel coordinate must start a 16-byte row segment (else the copy faults):
        // a debug-bounds build that finds one that does not records it and loads slab 0
        const int dc = in_bounds(d0 >= 0 && d0 < D && (d0 * LY::E) % 16 == 0 && t0 >= 0 &&
                                     t0 < L && b < p.batch, status, 101)
                           ? d0 : 0;
        ptx::mbar_arrive_expect_tx(&bars[s], LY::tx_bytes(has_z));
        ptx::tma_load_3d(st + LY::s_x, &maps.x, &bars[s], dc, t0, b);
        ptx::tma_load_3d(st + LY::s_dl, &maps.dl, &bars[s], dc, t0, b);
        ptx::tma_load_3d(st + LY::s_B, &maps.B, &bars[s], 0, t0, b);
        if (!kSummary) {
            if (has_z) ptx::tma_load_3d(st + LY::s_z, &maps.z, &bars[s], dc, t0, b);
            ptx::tma_load_3d(st + LY::s_C, &maps.C, &bars[s], 0, t0, b);
        }
    };
    if (tid == 0) {
        ptx::prefetch_tmap(&maps.x);
        for (int i = 0; i < kStages && i < ntiles; ++i) issue(i);
    }

    // ---------------- per-thread constants
    // scan role: channel sc of this warp, lane slot j owns states j*NS .. j*NS+NS-1
    const int sc = lane / LPC, j = lane % LPC;
    const int64_t sd = d0 + warp * CPW + sc;
    const bool sdval = sd < D;
    f2 a2[NS / 2], h[NS / 2], ia[NS / 2];
#pragma unroll
    for (int k = 0; k < NS / 2; ++k) {
        float av[2], hv[2], iv[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int n = j * NS + 2 * k + e;
            const float an = sdval ? p.A[sd * N + n] : 0.f;
            av[e] = scale_A<kFast>(an);
            iv[e] = an != 0.f ? 1.f / an : 0.f;
            hv[e] = (!kSummary && sdval && p.h0) ? p.h0[(b * D + sd) * N + n] : 0.f;
        }
        a2[k] = f2{av[0], av[1]};
        h[k] = f2{hv[0], hv[1]};
        ia[k] = f2{iv[0], iv[1]};
    }
    (void)ia;
    if (!kSummary) {
        // fold the summaries of the chunks before this one into the initial state
        for (int cc = 0; cc < c; ++cc) {
            const int64_t row = (static_cast<int64_t>(b) * K + cc) * D + sd;
            const float S = sdval ? __ldcg(p.dsum + row) : 0.f;
#pragma unroll
            for (int k = 0; k < NS / 2; ++k) {
                const int n = j * NS + 2 * k;
                const f2 he = sdval ? f2{__ldcg(p.hloc + row * N + n), __ldcg(p.hloc + row * N + n + 1)}
                                    : f2{0.f, 0.f};
                h[k] = ptx::fma2(decay2<kFast>(S, a2[k]), h[k], he);
            }
        }
    }
    // prologue / epilogue role: row t = lane, this warp's CPW channels
    float pbias[CPW], pD[CPW];
#pragma unroll
    for (int cc = 0; cc < CPW; ++cc) {
        const int64_t d = d0 + warp * CPW + cc;
        pbias[cc] = (d < D && p.bias) ? p.bias[d] : 0.f;
        pD[cc] = (!kSummary && d < D && p.Dv) ? p.Dv[d] : 0.f;
    }
    float dsum = 0.f;
    int failed_tile = -1;
    // checkpoints along the whole sequence (the backward pass's time tiles)
    const int64_t ck_tiles = kCkpt ? (L + (int64_t(1) << p.ckpt_shift) - 1) >> p.ckpt_shift : 0;
    (void)ck_tiles;

    for (int tile = 0; tile < ntiles; ++tile) {
        const int s = tile % kStages;
        const unsigned char *st = smem + s * LY::stage;
        const int64_t t0 = t_begin + static_cast<int64_t>(tile) * kT;
        const bool got = ptx::mbar_wait(&bars[s], (tile / kStages) & 1);

        // ---------------- prologue (only after this thread's own wait succeeded)
        constexpr bool kWidenB = kSummary && LY::kRawBC;
        const float *Bf = kWidenB ? reinterpret_cast<const float *>(smem + LY::o_bf32)
                                  : reinterpret_cast<const float *>(st + LY::s_B);   // fp32 I/O
        const float *Cf = reinterpret_cast<const float *>(st + LY::s_C);
        if (got) {
            if constexpr (kWidenB) {
                // the block widens the tile's B (kT x N bf16) once for all its lanes
                const uint32_t *src = reinterpret_cast<const uint32_t *>(st + LY::s_B);
                float2 *dst = reinterpret_cast<float2 *>(smem + LY::o_bf32);
                for (int e = tid; e < kT * N / 2; e += 32 * WPC) {
                    const ptx::f2 v = ptx::bf2_to_f2(src[e]);
                    dst[e] = make_float2(v.x, v.y);
                }
            }
            const bool tval = t0 + lane < t_end;
#pragma unroll
            for (int q = 0; q < QW; ++q) {
                const int qc = warp * QW + q;  // chunk index within the row
                float vd[EC], vx[EC];
                CK::load(st + LY::s_dl + tok_chunk<ROWB>(lane, qc), vd);
                CK::load(st + LY::s_x + tok_chunk<ROWB>(lane, qc), vx);
#pragma unroll
                for (int e = 0; e < EC; ++e) {
                    const int cc = q * EC + e;
                    const float dl = tval ? step_size<kFast>(vd[e], pbias[cc], p.softplus) : 0.f;
                    *reinterpret_cast<float2 *>(dlx + (warp * CPW + cc) * LY::kDlxRow + 2 * lane) =
                        make_float2(dl, kZoh ? vx[e] : dl * vx[e]);
                }
            }
        }
        if (!__syncthreads_and(got ? 1 : 0)) {
            failed_tile = tile;
            break;
        }

        // ---------------- scan: NS states per lane, in time order, kU steps per block
        {
            const float *row = dlx + (warp * CPW + sc) * LY::kDlxRow;
            // the whole tile unrolled at up to 4 states per lane (N = 16: 198 / 2533 us
            // against 206 / 2690 us unrolled by 2 at the 130M / long-context shapes);
            // more states per lane would spill
            constexpr int kTbUnroll = NS <= 4 ? kT / kU : 2;
#pragma unroll kTbUnroll
            for (int tb = 0; tb < kT; tb += kU) {
                float dl[kU], dx[kU];
#pragma unroll
                for (int u = 0; u < kU; u += 2) {
                    const float4 q = *reinterpret_cast<const float4 *>(row + 2 * (tb + u));
                    dl[u] = q.x; dx[u] = q.y; dl[u + 1] = q.z; dx[u + 1] = q.w;
                }
                f2 bp[kU][NS / 2], cp[kU][NS / 2];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    if constexpr (LY::kRawBC && !kWidenB) {
                        // NS bf16 values = NS / 2 words per row, 8- or 16-byte loads
                        const uint32_t *Bw = reinterpret_cast<const uint32_t *>(st + LY::s_B) +
                                             ((tb + u) * N + j * NS) / 2;
                        const uint32_t *Cw = reinterpret_cast<const uint32_t *>(st + LY::s_C) +
                                             ((tb + u) * N + j * NS) / 2;
                        constexpr int kW = (NS / 2) % 4 == 0 ? 4 : 2;
#pragma unroll
                        for (int k = 0; k < NS / 2; k += kW) {
                            uint32_t wb[kW], wc[kW];
                            if constexpr (kW == 4) {
                                const uint4 b4 = *reinterpret_cast<const uint4 *>(Bw + k);
                                wb[0] = b4.x; wb[1] = b4.y; wb[2] = b4.z; wb[3] = b4.w;
                                if (!kSummary) {
                                    const uint4 c4 = *reinterpret_cast<const uint4 *>(Cw + k);
                                    wc[0] = c4.x; wc[1] = c4.y; wc[2] = c4.z; wc[3] = c4.w;
                                }
                            } else {
                                const uint2 b2 = *reinterpret_cast<const uint2 *>(Bw + k);
                                wb[0] = b2.x; wb[1] = b2.y;
                                if (!kSummary) {
                                    const uint2 c2 = *reinterpret_cast<const uint2 *>(Cw + k);
                                    wc[0] = c2.x; wc[1] = c2.y;
                                }
                            }
#pragma unroll
                            for (int i = 0; i < kW; ++i) {
                                bp[u][k + i] = ptx::bf2_to_f2(wb[i]);
                                if (!kSummary) cp[u][k + i] = ptx::bf2_to_f2(wc[i]);
                            }
                        }
                        continue;
                    }
                    const float *Bt = Bf + (tb + u) * N + j * NS;
                    const float *Ct = Cf + (tb + u) * N + j * NS;
#pragma unroll
                    for (int k = 0; k < NS / 2; k += 2) {
                        if (k + 1 < NS / 2) {
                            const float4 bq = *reinterpret_cast<const float4 *>(Bt + 2 * k);
                            bp[u][k] = f2{bq.x, bq.y};
                            bp[u][k + 1] = f2{bq.z, bq.w};
                            if (!kSummary) {
                                const float4 cq = *reinterpret_cast<const float4 *>(Ct + 2 * k);
                                cp[u][k] = f2{cq.x, cq.y};
                                cp[u][k + 1] = f2{cq.z, cq.w};
                            }
                        } else {
                            const float2 bq = *reinterpret_cast<const float2 *>(Bt + 2 * k);
                            bp[u][k] = f2{bq.x, bq.y};
                            if (!kSummary) {
                                const float2 cq = *reinterpret_cast<const float2 *>(Ct + 2 * k);
                                cp[u][k] = f2{cq.x, cq.y};
                            }
                        }
                    }
                }
                f2 av[kU][NS / 2], uv[kU][NS / 2];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
#pragma unroll
                    for (int k = 0; k < NS / 2; ++k) {
                        av[u][k] = decay2<kFast>(dl[u], a2[k]);
                        if (kZoh) {
                            // dx holds x here: B̄ x = ((exp(dl A) - 1) / A) B x
                            constexpr float kToNat = kFast ? kLn2 : 1.f;
                            const f2 v = ptx::mul2(f2{dl[u] * kToNat, dl[u] * kToNat}, a2[k]);
                            const f2 cf{zoh_coef<kFast>(dl[u], v.x, av[u][k].x, ia[k].x),
                                        zoh_coef<kFast>(dl[u], v.y, av[u][k].y, ia[k].y)};
                            uv[u][k] = ptx::mul2(cf, ptx::mul2(f2{dx[u], dx[u]}, bp[u][k]));
                        } else {
                            uv[u][k] = ptx::mul2(f2{dx[u], dx[u]}, bp[u][k]);
                        }
                    }
                }
                if constexpr (kCkpt && !kSummary) {
                    // the state before step t0 + tb, at every checkpoint step (checkpoints
                    // are at least kU steps apart, so only a block's first step has one)
                    const int64_t t = t0 + tb;
                    if ((tb & ((1 << p.ckpt_shift) - 1)) == 0 && sdval && t < t_end &&
                        in_bounds((t >> p.ckpt_shift) < ck_tiles && b < p.batch, status, 102)) {
                        float2 *ck = reinterpret_cast<float2 *>(
                            p.ckpt + ((b * ck_tiles + (t >> p.ckpt_shift)) * D + sd) * N + j * NS);
#pragma unroll
                        for (int k = 0; k < NS / 2; ++k) ck[k] = make_float2(h[k].x, h[k].y);
                    }
                }
                float acc[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    f2 s2{0.f, 0.f};
#pragma unroll
                    for (int k = 0; k < NS / 2; ++k) {
                        h[k] = ptx::fma2(av[u][k], h[k], uv[u][k]);
                        if (!kSummary) s2 = ptx::fma2(cp[u][k], h[k], s2);
                    }
                    acc[u] = s2.x + s2.y;
                    if (kSummary) dsum += dl[u];
                }
                if (!kSummary && !kRed) {
#pragma unroll
                    for (int u = 0; u < kU; ++u)
                        part[j * LY::kPart + (tb + u) * LY::kPartT + sc] = acc[u];
                }
                if (!kSummary && kRed) {
                    // sum over the channel's LPC adjacent lanes as a reduce-scatter: at
                    // lane bit m every lane keeps the steps whose bit m matches its own
                    // and adds the partner's copy, so lane slot j ends with the sums of
                    // the steps u with u % LPC == j (same pairing as a butterfly)
                    constexpr int kOut = kU / LPC;
                    static_assert(kU % LPC == 0, "an ILP block holds whole lane groups");
#pragma unroll
                    for (int m = 1, cnt = kU; m < LPC; m <<= 1, cnt >>= 1) {
                        const bool hi = (j & m) != 0;
#pragma unroll
                        for (int i = 0; i < cnt / 2; ++i) {
                            const float keep = hi ? acc[2 * i + 1] : acc[2 * i];
                            const float send = hi ? acc[2 * i] : acc[2 * i + 1];
                            acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < kOut; ++i)
                        part[(tb + i * LPC + j) * LY::kPartT + sc] = acc[i];
                }
            }
        }
        __syncwarp();

        // ---------------- epilogue: row t = lane, this warp's channels
        if (!kSummary) {
            unsigned char *ytile = smem + LY::o_y + (tile & 1) * align1k(LY::kTok);
            float acc[CPW];
#pragma unroll
            for (int cc = 0; cc < CPW; cc += 4) {
                float4 a4 = *reinterpret_cast<const float4 *>(part + lane * LY::kPartT + cc);
#pragma unroll
                for (int jj = 1; jj < LY::kSlots; ++jj) {
                    const float4 v = *reinterpret_cast<const float4 *>(
                        part + jj * LY::kPart + lane * LY::kPartT + cc);
                    const f2 lo = ptx::add2(f2{a4.x, a4.y}, f2{v.x, v.y});
                    const f2 hi = ptx::add2(f2{a4.z, a4.w}, f2{v.z, v.w});
                    a4 = make_float4(lo.x, lo.y, hi.x, hi.y);
                }
                acc[cc] = a4.x; acc[cc + 1] = a4.y; acc[cc + 2] = a4.z; acc[cc + 3] = a4.w;
            }
#pragma unroll
            for (int q = 0; q < QW; ++q) {
                const int qc = warp * QW + q;
                float vx[EC], vz[EC], out[EC];
                CK::load(st + LY::s_x + tok_chunk<ROWB>(lane, qc), vx);
                if (has_z) CK::load(st + LY::s_z + tok_chunk<ROWB>(lane, qc), vz);
#pragma unroll
                for (int e = 0; e < EC; ++e) {
                    const int cc = q * EC + e;
                    float o = fmaf(pD[cc], vx[e], acc[cc]);
                    if (has_z) o *= silu<kFast>(vz[e]);
                    out[e] = o;
                }
                CK::store(ytile + tok_chunk<ROWB>(lane, qc), out);
            }
            ptx::fence_proxy_async_smem();
        }
        __syncthreads();
        if (tid == 0) {
            if (!kSummary && in_bounds(d0 >= 0 && d0 < D && (d0 * LY::E) % 16 == 0 && t0 >= 0 &&
                                           t0 < L, status, 103)) {
                ptx::tma_store_3d(&maps.y, smem + LY::o_y + (tile & 1) * align1k(LY::kTok), d0,
                                  static_cast<int>(t0), b);
                ptx::bulk_commit();
                ptx::bulk_wait_read<1>();  // the y tile the next tile writes is free again
            }
            // refill this stage with the tile kStages ahead
            if (tile + kStages < ntiles) issue(tile + kStages);
        }
    }

    if (failed_tile >= 0) {
        if (tid == 0) report_status(status, SSM_ERR_TIMEOUT, kSummary ? 11 : 12);
        // let the copies still in flight land before the block's shared memory is
        // released (each wait again bounded)
        for (int i = failed_tile; i < failed_tile + kStages && i < ntiles; ++i)
            if (!ptx::mbar_wait(&bars[i % kStages], (i / kStages) & 1)) break;
        if (!kSummary && tid == 0) ptx::bulk_wait<0>();
        return false;
    }
    if (!kSummary && tid == 0) ptx::bulk_wait<0>();

    if (kSummary) {
        const int64_t row = (static_cast<int64_t>(b) * K + c) * D + sd;
        if (sdval && in_bounds(row < p.batch * K * D && c < K - 1, status, 104)) {
#pragma unroll
            for (int k = 0; k < NS / 2; ++k) {
                const int n = j * NS + 2 * k;
                *reinterpret_cast<float2 *>(p.hloc + row * N + n) = make_float2(h[k].x, h[k].y);
            }
            // every lane of the channel accumulated the same sum; one writes it
            if (j == 0) p.dsum[row] = dsum;
        }
        if (kLB) {
            // publish: the block's summary writes happen before the flag's release
            __threadfence();
            __syncthreads();
            if (tid == 0 && p.publish &&
                in_bounds(b < p.batch && c < K && slab < nslabs, status, 105))
                ptx::st_release_u32(p.flags + (static_cast<int64_t>(b) * K + c) * nslabs + slab, 1u);
        }
    } else if (c == K - 1 && p.h_final && sdval && in_bounds(b < p.batch, status, 106)) {
#pragma unroll
        for (int k = 0; k < NS / 2; ++k) {
            const int n = j * NS + 2 * k;
            *reinterpret_cast<float2 *>(p.h_final + (b * D + sd) * N + n) =
                make_float2(h[k].x, h[k].y);
        }
    }
    release_barriers();
    return true;
}

// Two-launch form: the summary pass over chunks 0 .. K-2, then the output pass.
template <typename TIO, int NS, int LPC, int WPC, bool kSummary, bool kZoh, bool kRed,
          bool kCkpt>
__device__ __forceinline__ void scan_tma_entry(const TmaMaps &maps, const ScanParams &p) {
    using LY = Layout<TIO, NS, LPC, WPC, kSummary, kRed>;
    DeviceStatus *status = static_cast<DeviceStatus *>(p.status);
    // the first block of the first launch of a call clears the status word
    if (p.clear_status && status && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0 &&
        blockIdx.z == 0)
        status->code = 0;
    (void)chunk_pass<TIO, NS, LPC, WPC, kSummary, kZoh, false, kRed, kCkpt>(
        maps, p, blockIdx.y, blockIdx.z, blockIdx.x * LY::CPB, blockIdx.x);
}

template <typename TIO, int NS, int LPC, int WPC, bool kSummary, bool kZoh, bool kRed,
          bool kCkpt>
__global__ void __launch_bounds__(32 * WPC) scan_tma_kernel(const __grid_constant__ TmaMaps maps,
                                                            ScanParams p) {
    scan_tma_entry<TIO, NS, LPC, WPC, kSummary, kZoh, kRed, kCkpt>(maps, p);
}

// The same pass under a register budget instead of launch bounds, for the bf16 Euler
// output pass at four states per lane over four lanes: there the fully unrolled tile gets 72-80
// registers and no spill, against 56 registers and a 16-byte spill under the launch
// bounds (130M-layer shape: 191 against 198 us on B300).  Other instantiations spill
// under the budget and keep the launch bounds.
template <typename TIO, int NS, int LPC, int WPC, bool kSummary, bool kZoh, bool kRed,
          bool kCkpt>
__global__ void __maxnreg__(96) scan_tma_kernel_r96(const __grid_constant__ TmaMaps maps,
                                                    ScanParams p) {
    scan_tma_entry<TIO, NS, LPC, WPC, kSummary, kZoh, kRed, kCkpt>(maps, p);
}

// Single-launch form with a decoupled look-back.  Blocks take their work from an atomic
// ticket in chunk-major order (every slab of chunk 0, then of chunk 1, ...): a block
// scans its chunk from a zero state and publishes the summary (all chunks but the last),
// then acquires the summaries of the earlier chunks of its slab, folds them into its
// initial state and runs the output pass.  A block waits only on blocks with smaller
// tickets, which have started and publish before they wait themselves, so the waits end;
// they are bounded all the same.  Every chunk but the last is still read twice (summary
// and output), as in the two-launch form; what goes is the launch boundary between the
// passes and the idle tail of the first launch.
template <typename TIO, int NS, int LPC, int WPC, bool kZoh, bool kRed, bool kCkpt>
__global__ void __launch_bounds__(32 * WPC) scan_tma_lb_kernel(const __grid_constant__ TmaMaps maps,
                                                               ScanParams p) {
    using LY = Layout<TIO, NS, LPC, WPC, false, kRed>;
    __shared__ int s_ticket;
    if (threadIdx.x == 0) s_ticket = static_cast<int>(atomicAdd(p.ticket, 1u));
    __syncthreads();
    const int ticket = s_ticket;
    const int nslabs = static_cast<int>((p.dim + LY::CPB - 1) / LY::CPB);
    const int per_chunk = static_cast<int>(p.batch) * nslabs;
    const int c = ticket / per_chunk, r = ticket % per_chunk;
    const int b = r / nslabs, slab = r % nslabs;
    if (c < p.nchunks - 1 &&
        !chunk_pass<TIO, NS, LPC, WPC, true, kZoh, true, kRed, false>(maps, p, b, c,
                                                                      slab * LY::CPB, slab))
        return;
    (void)chunk_pass<TIO, NS, LPC, WPC, false, kZoh, true, kRed, kCkpt>(maps, p, b, c,
                                                                          slab * LY::CPB, slab);
}

// ---------------------------------------------------------------- host side
template <typename TIO, int NS, int LPC, int WPC, bool kSummary, bool kZoh, bool kRed,
          bool kCkpt>
cudaError_t launch_tma_one(const ScanParams &p, const TmaMaps &maps, int nchunks_grid,
                           cudaStream_t stream) {
    using LY = Layout<TIO, NS, LPC, WPC, kSummary, kRed>;
    void (*kern)(const TmaMaps, ScanParams);
    if constexpr (std::is_same<TIO, __nv_bfloat16>::value && NS == 4 && LPC == 4 && !kSummary &&
                  !kZoh)
        kern = scan_tma_kernel_r96<TIO, NS, LPC, WPC, kSummary, kZoh, kRed, kCkpt>;
    else
        kern = scan_tma_kernel<TIO, NS, LPC, WPC, kSummary, kZoh, kRed, kCkpt>;
    if (LY::bytes > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             LY::bytes);
        if (e != cudaSuccess) return e;
    }
    dim3 grid(static_cast<unsigned>((p.dim + LY::CPB - 1) / LY::CPB),
              static_cast<unsigned>(p.batch), static_cast<unsigned>(nchunks_grid));
    kern<<<grid, 32 * WPC, LY::bytes, stream>>>(maps, p);
    return cudaGetLastError();
}

// Blocks of 32 channels: WPC = LPC warps of 32 / LPC channels each.
template <typename TIO, int NS, int LPC, bool kZoh, bool kCkpt>
cudaError_t launch_tma_pair(ScanParams p, cudaStream_t stream) {
    constexpr int WPC = LPC;
    using LY = Layout<TIO, NS, LPC, WPC, false>;
    const bool bf = std::is_same<TIO, __nv_bfloat16>::value;
    TmaMaps m{};
    const int64_t B = p.batch, L = p.seqlen, D = p.dim, N = p.dstate;
    bool ok = make_tma_map_3d(&m.x, p.x, bf, B, L, D, LY::CPB, kT, LY::ROWB) &&
              make_tma_map_3d(&m.dl, p.delta, bf, B, L, D, LY::CPB, kT, LY::ROWB) &&
              make_tma_map_3d(&m.B, p.Bm, bf, B, L, N, static_cast<int>(N), kT, 0) &&
              make_tma_map_3d(&m.C, p.Cm, bf, B, L, N, static_cast<int>(N), kT, 0) &&
              make_tma_map_3d(&m.y, p.y, bf, B, L, D, LY::CPB, kT, LY::ROWB);
    if (ok && p.z) ok = make_tma_map_3d(&m.z, p.z, bf, B, L, D, LY::CPB, kT, LY::ROWB);
    if (!ok) return cudaErrorInvalidValue;
    p.clear_status = 1;
    if (p.nchunks > 1 && p.flags && kScanLookback) {
        // one launch, the chunk summaries handed over through the look-back flags (the
        // caller zeroed the status word, the ticket and the flags)
        using LR = Layout<TIO, NS, LPC, WPC, false, kSplitRed>;
        auto kern = scan_tma_lb_kernel<TIO, NS, LPC, WPC, kZoh, kSplitRed, kCkpt>;
        if (LR::bytes > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 LR::bytes);
            if (e != cudaSuccess) return e;
        }
        const int64_t blocks = static_cast<int64_t>(p.nchunks) * p.batch * ((D + LR::CPB - 1) / LR::CPB);
        kern<<<static_cast<unsigned>(blocks), 32 * WPC, LR::bytes, stream>>>(m, p);
        return cudaGetLastError();
    }
    if (p.nchunks > 1) {
        cudaError_t e = launch_tma_one<TIO, NS, LPC, WPC, true, kZoh, false, false>(
            p, m, p.nchunks - 1, stream);
        if (e != cudaSuccess) return e;
        p.clear_status = 0;
        return launch_tma_one<TIO, NS, LPC, WPC, false, kZoh, kSplitRed, kCkpt>(p, m, p.nchunks,
                                                                                stream);
    }
    return launch_tma_one<TIO, NS, LPC, WPC, false, kZoh, false, kCkpt>(p, m, p.nchunks, stream);
}

// with or without state checkpoints for the backward pass
template <typename TIO, int NS, int LPC, bool kZoh>
cudaError_t launch_tma_ck(const ScanParams &p, cudaStream_t stream) {
    return p.ckpt ? launch_tma_pair<TIO, NS, LPC, kZoh, true>(p, stream)
                  : launch_tma_pair<TIO, NS, LPC, kZoh, false>(p, stream);
}

}  // namespace

// Lane slots per channel (LPC, NS = N / LPC states per lane) for each supported N;
// 32-channel blocks hold LPC warps of 32 / LPC channels.
static int scan_tma_lpc(int io_bf16, int64_t dstate) {
    switch (dstate) {
        case 4: return io_bf16 ? 0 : 2;  // 8-byte bf16 B/C rows are below the TMA minimum
        case 8: return 2;
        case 16: return 4;
        case 32: return 4;
        case 64: return 4;
        default: return 0;
    }
}

namespace {
// Resident blocks per SM of the output kernel, from its shared memory (228 KiB per SM,
// 1 KiB reserved per block) and its warps (64 per SM).
template <typename TIO, int NS, int LPC> int blocks_per_sm() {
    using LY = Layout<TIO, NS, LPC, LPC, false>;
    const int by_smem = (228 * 1024) / (LY::bytes + 1024);
    const int by_warps = 64 / LPC;
    const int b = by_smem < by_warps ? by_smem : by_warps;
    return b > 0 ? b : 1;
}
}  // namespace

int scan_tma_blocks_per_sm(int io_bf16, int64_t dstate) {
    if (io_bf16) {
        switch (dstate) {
            case 8: return blocks_per_sm<__nv_bfloat16, 4, 2>();
            case 16: return blocks_per_sm<__nv_bfloat16, 4, 4>();
            case 32: return blocks_per_sm<__nv_bfloat16, 8, 4>();
            case 64: return blocks_per_sm<__nv_bfloat16, 16, 4>();
            default: return 0;
        }
    }
    switch (dstate) {
        case 4: return blocks_per_sm<float, 2, 2>();
        case 8: return blocks_per_sm<float, 4, 2>();
        case 16: return blocks_per_sm<float, 4, 4>();
        case 32: return blocks_per_sm<float, 8, 4>();
        case 64: return blocks_per_sm<float, 16, 4>();
        default: return 0;
    }
}

bool scan_tma_sizes_ok(int io_bf16, int64_t seqlen, int64_t dim, int64_t dstate) {
    const int64_t e = io_bf16 ? 2 : 4;
    if (scan_tma_lpc(io_bf16, dstate) == 0) return false;
    if (dstate * e % 16 != 0 || dim * e % 16 != 0) return false;
    return seqlen > 0 && seqlen < (int64_t(1) << 31) && dim < (int64_t(1) << 31);
}

bool scan_tma_pointers_ok(const void *const *ptrs, int nptrs) {
    for (int i = 0; i < nptrs; ++i)
        if (ptrs[i] && reinterpret_cast<uintptr_t>(ptrs[i]) % 16 != 0) return false;
    return tma_encoder() != nullptr;
}

template <bool kZoh> cudaError_t launch_scan_tma_disc(const ScanParams &p, cudaStream_t stream) {
    const int64_t N = p.dstate;
    if (p.io_bf16) {
        using T = __nv_bfloat16;
        if (N == 8) return launch_tma_ck<T, 4, 2, kZoh>(p, stream);
        if (N == 16) return launch_tma_ck<T, 4, 4, kZoh>(p, stream);
        if (N == 32) return launch_tma_ck<T, 8, 4, kZoh>(p, stream);
        if (N == 64) return launch_tma_ck<T, 16, 4, kZoh>(p, stream);
    } else {
        using T = float;
        if (N == 4) return launch_tma_ck<T, 2, 2, kZoh>(p, stream);
        if (N == 8) return launch_tma_ck<T, 4, 2, kZoh>(p, stream);
        if (N == 16) return launch_tma_ck<T, 4, 4, kZoh>(p, stream);
        if (N == 32) return launch_tma_ck<T, 8, 4, kZoh>(p, stream);
        if (N == 64) return launch_tma_ck<T, 16, 4, kZoh>(p, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_scan_tma(const ScanParams &p, cudaStream_t stream) {
    return p.zoh ? launch_scan_tma_disc<true>(p, stream) : launch_scan_tma_disc<false>(p, stream);
}

}  // namespace ssm
