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
//   * One warp per thread block.  The warp owns CPW = 32 / LPC channels of one
//     batch row; each channel's N states are split over LPC adjacent lanes, NS
//     states per lane.  The recurrence runs in time order inside each lane (one
//     exp, two packed fp32x2 products and two packed FMAs per pair of states).
//     Small single-warp blocks keep the 148 SMs evenly loaded (about ten blocks
//     per SM at the 130M-layer shape) and need no block-wide barrier.
//   * Inputs arrive through a two-stage TMA pipeline: 3-D tensor maps over
//     (channel, time, batch) give boxes of CPW channels x 32 steps for x, delta
//     and z and N states x 32 steps for B and C; boxes past the end of a sequence
//     are zero-filled by the TMA unit.  One lane issues the copies, every lane
//     waits on the stage's mbarrier (bounded by a clock budget).
//   * Per 32-step tile: (1) a prologue in which lane t turns row t of the tile
//     into fp32 (dl, dl*x) pairs (softplus computed once per (t, d)) and converts
//     B and C to fp32; (2) the scan, reading (dl, dl*x) with 16-byte loads and B,
//     C as broadcast 16-byte loads; per-lane partial readouts go to shared
//     memory; (3) an epilogue in which lane t sums the partials of row t, adds
//     D x, applies the gate, rounds to the I/O type and writes a y tile that one
//     TMA store sends to HBM.
//   * Long sequences are cut into K time chunks (blockIdx.z).  A summary pass
//     (kSummary) scans chunks 0..K-2 from a zero state and keeps each chunk's end
//     state and step sum; the output pass folds the summaries of earlier chunks
//     into its initial state, h <- exp(A * sum dl) h + h_end: the associative
//     combine of the parallel scan ("병렬 스캔") applied to whole chunks.
#include <cudaTypedefs.h>

#include "../../include/ssm.h"

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace ssm {
namespace {

using ptx::f2;

constexpr int kT = 32;       // time steps per tile (one per lane in prologue/epilogue)
constexpr int kStages = 2;   // TMA pipeline depth

__host__ __device__ constexpr int align128(int v) { return (v + 127) / 128 * 128; }

template <typename TIO, int NS, int LPC, bool kSummary> struct Layout {
    static constexpr int CPW = 32 / LPC;  // channels per block
    static constexpr int N = NS * LPC;
    static constexpr int E = sizeof(TIO);
    static constexpr int kTok = kT * CPW * E;  // bytes of one x / delta / z tile
    static constexpr int kBC = kT * N * E;     // bytes of one B or C tile
    // one pipeline stage: x, delta, z, B, C (no z, C in the summary pass)
    static constexpr int s_x = 0;
    static constexpr int s_dl = s_x + align128(kTok);
    static constexpr int s_z = s_dl + align128(kTok);
    static constexpr int s_B = s_z + (kSummary ? 0 : align128(kTok));
    static constexpr int s_C = s_B + align128(kBC);
    static constexpr int stage = s_C + (kSummary ? 0 : align128(kBC));
    // bytes one stage receives (z only when a gate is given)
    __host__ __device__ static constexpr int tx_bytes(bool gate) {
        return (kSummary ? 2 : (gate ? 3 : 2)) * kTok + (kSummary ? 1 : 2) * kBC;
    }
    // work buffers after the stages
    static constexpr int kDlxRow = 2 * kT + 4;  // floats per channel row of (dl, dl x)
    static constexpr int o_dlx = kStages * stage;
    static constexpr int o_Bf = o_dlx + align128(CPW * kDlxRow * 4);
    static constexpr int o_Cf = o_Bf + align128(kT * N * 4);
    // floats per lane slot of the partial readouts; the CPW-float pad puts the
    // LPC slots of one time step on distinct banks
    static constexpr int kPart = kT * CPW + CPW;
    static constexpr int o_part = o_Cf + (kSummary ? 0 : align128(kT * N * 4));
    static constexpr int o_y = o_part + (kSummary ? 0 : align128(LPC * kPart * 4));
    static constexpr int o_bar = o_y + (kSummary ? 0 : 2 * align128(kTok));
    static constexpr int bytes = o_bar + kStages * 8;
};

struct TmaMaps {
    CUtensorMap x, dl, z, B, C, y;
};

// Element loads of one tile row (CPW consecutive channels) as floats.
template <typename TIO, int CPW> struct Row;
template <int CPW> struct Row<float, CPW> {
    static __device__ __forceinline__ void load(const unsigned char *p, float (&v)[CPW]) {
#pragma unroll
        for (int c = 0; c < CPW; c += 4) {
            const float4 q = *reinterpret_cast<const float4 *>(p + 4 * c);
            v[c] = q.x; v[c + 1] = q.y; v[c + 2] = q.z; v[c + 3] = q.w;
        }
    }
    static __device__ __forceinline__ void store(unsigned char *p, const float (&v)[CPW]) {
#pragma unroll
        for (int c = 0; c < CPW; c += 4)
            *reinterpret_cast<float4 *>(p + 4 * c) = make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
    }
};
template <int CPW> struct Row<__nv_bfloat16, CPW> {
    static __device__ __forceinline__ void load(const unsigned char *p, float (&v)[CPW]) {
#pragma unroll
        for (int c = 0; c < CPW; c += 8) {
            const uint4 q = *reinterpret_cast<const uint4 *>(p + 2 * c);
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const f2 e = ptx::bf2_to_f2(w[i]);
                v[c + 2 * i] = e.x;
                v[c + 2 * i + 1] = e.y;
            }
        }
    }
    static __device__ __forceinline__ void store(unsigned char *p, const float (&v)[CPW]) {
#pragma unroll
        for (int c = 0; c < CPW; c += 8) {
            uint4 q;
            q.x = ptx::f2_to_bf2(v[c], v[c + 1]);
            q.y = ptx::f2_to_bf2(v[c + 2], v[c + 3]);
            q.z = ptx::f2_to_bf2(v[c + 4], v[c + 5]);
            q.w = ptx::f2_to_bf2(v[c + 6], v[c + 7]);
            *reinterpret_cast<uint4 *>(p + 2 * c) = q;
        }
    }
};

// Decay factors of a pair of states: exp(dl * A) (accurate) or 2^(dl * A log2 e).
template <bool kFast> __device__ __forceinline__ f2 decay2(float dl, f2 a) {
    const f2 v = ptx::mul2(f2{dl, dl}, a);
    if (kFast) return f2{ex2_approx(v.x), ex2_approx(v.y)};
    return f2{expf(v.x), expf(v.y)};
}

template <typename TIO, int NS, int LPC, bool kSummary>
__global__ void __launch_bounds__(32) scan_tma_kernel(const __grid_constant__ TmaMaps maps,
                                                      ScanParams p) {
    using LY = Layout<TIO, NS, LPC, kSummary>;
    constexpr int CPW = LY::CPW;
    constexpr int N = LY::N;
    constexpr bool kFast = std::is_same<TIO, __nv_bfloat16>::value;
    static_assert(NS % 2 == 0, "states per lane must be even (packed pairs)");
    static_assert(CPW * sizeof(TIO) % 16 == 0 && N * sizeof(TIO) % 16 == 0, "TMA row sizes");

    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + LY::o_bar);
    float *dlx = reinterpret_cast<float *>(smem + LY::o_dlx);
    float *Bf = reinterpret_cast<float *>(smem + LY::o_Bf);
    float *Cf = reinterpret_cast<float *>(smem + LY::o_Cf);
    float *part = reinterpret_cast<float *>(smem + LY::o_part);

    const int lane = threadIdx.x;
    const int64_t D = p.dim, L = p.seqlen;
    const int K = p.nchunks;
    const int b = blockIdx.y;
    const int c = blockIdx.z;
    const int d0 = blockIdx.x * CPW;
    const bool has_z = p.z != nullptr;
    DeviceStatus *status = static_cast<DeviceStatus *>(p.status);

    // the first block of the first launch of a call clears the status word
    if (p.clear_status && status && lane == 0 && blockIdx.x == 0 && blockIdx.y == 0 &&
        blockIdx.z == 0)
        status->code = 0;

    const int64_t t_begin = static_cast<int64_t>(c) * p.chunk_len;
    const int64_t t_end = min(L, t_begin + p.chunk_len);
    const int ntiles = static_cast<int>((t_end - t_begin + kT - 1) / kT);

    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) ptx::mbar_init(&bars[s], 1);
        ptx::fence_mbar_init();
    }
    __syncwarp();

    auto issue = [&](int tile) {  // lane 0 only
        const int s = tile % kStages;
        unsigned char *st = smem + s * LY::stage;
        const int t0 = static_cast<int>(t_begin + static_cast<int64_t>(tile) * kT);
        ptx::mbar_arrive_expect_tx(&bars[s], LY::tx_bytes(has_z));
        ptx::tma_load_3d(st + LY::s_x, &maps.x, &bars[s], d0, t0, b);
        ptx::tma_load_3d(st + LY::s_dl, &maps.dl, &bars[s], d0, t0, b);
        ptx::tma_load_3d(st + LY::s_B, &maps.B, &bars[s], 0, t0, b);
        if (!kSummary) {
            if (has_z) ptx::tma_load_3d(st + LY::s_z, &maps.z, &bars[s], d0, t0, b);
            ptx::tma_load_3d(st + LY::s_C, &maps.C, &bars[s], 0, t0, b);
        }
    };
    if (lane == 0) {
        ptx::prefetch_tmap(&maps.x);
        for (int i = 0; i < kStages && i < ntiles; ++i) issue(i);
    }

    // ---------------- per-lane constants
    // scan role: channel sc, lane slot j owns states j*NS .. j*NS+NS-1
    const int sc = lane / LPC, j = lane % LPC;
    const int64_t sd = d0 + sc;
    const bool sdval = sd < D;
    f2 a2[NS / 2], h[NS / 2];
#pragma unroll
    for (int k = 0; k < NS / 2; ++k) {
        float av[2], hv[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int n = j * NS + 2 * k + e;
            av[e] = sdval ? scale_A<kFast>(p.A[sd * N + n]) : 0.f;
            hv[e] = (!kSummary && sdval && p.h0) ? p.h0[(b * D + sd) * N + n] : 0.f;
        }
        a2[k] = f2{av[0], av[1]};
        h[k] = f2{hv[0], hv[1]};
    }
    if (!kSummary) {
        // fold the summaries of the chunks before this one into the initial state
        for (int cc = 0; cc < c; ++cc) {
            const int64_t row = (static_cast<int64_t>(b) * K + cc) * D + sd;
            const float S = sdval ? p.dsum[row] : 0.f;
#pragma unroll
            for (int k = 0; k < NS / 2; ++k) {
                const int n = j * NS + 2 * k;
                const f2 he = sdval ? f2{p.hloc[row * N + n], p.hloc[row * N + n + 1]} : f2{0.f, 0.f};
                h[k] = ptx::fma2(decay2<kFast>(S, a2[k]), h[k], he);
            }
        }
    }
    // prologue / epilogue role: row t = lane of the tile, all CPW channels
    float pbias[CPW], pD[CPW];
#pragma unroll
    for (int cc = 0; cc < CPW; ++cc) {
        const int64_t d = d0 + cc;
        pbias[cc] = (d < D && p.bias) ? p.bias[d] : 0.f;
        pD[cc] = (!kSummary && d < D && p.Dv) ? p.Dv[d] : 0.f;
    }
    float dsum = 0.f;
    int failed_tile = -1;

    for (int tile = 0; tile < ntiles; ++tile) {
        const int s = tile % kStages;
        const unsigned char *st = smem + s * LY::stage;
        const int64_t t0 = t_begin + static_cast<int64_t>(tile) * kT;
        if (!ptx::mbar_wait(&bars[s], (tile / kStages) & 1)) {
            failed_tile = tile;
            break;
        }
        // ---------------- prologue: row t = lane
        {
            const bool tval = t0 + lane < t_end;
            float vx[CPW], vd[CPW];
            Row<TIO, CPW>::load(st + LY::s_dl + lane * CPW * sizeof(TIO), vd);
            Row<TIO, CPW>::load(st + LY::s_x + lane * CPW * sizeof(TIO), vx);
#pragma unroll
            for (int cc = 0; cc < CPW; ++cc) {
                const float dl = tval ? step_size<kFast>(vd[cc], pbias[cc], p.softplus) : 0.f;
                *reinterpret_cast<float2 *>(dlx + cc * LY::kDlxRow + 2 * lane) =
                    make_float2(dl, dl * vx[cc]);
            }
            // B (and C) row t to fp32
            float vb[N];
            Row<TIO, N>::load(st + LY::s_B + lane * N * sizeof(TIO), vb);
            Row<float, N>::store(reinterpret_cast<unsigned char *>(Bf + lane * N), vb);
            if (!kSummary) {
                Row<TIO, N>::load(st + LY::s_C + lane * N * sizeof(TIO), vb);
                Row<float, N>::store(reinterpret_cast<unsigned char *>(Cf + lane * N), vb);
            }
        }
        __syncwarp();

        // ---------------- scan: NS states per lane, in time order
        {
            const float *row = dlx + sc * LY::kDlxRow;
#pragma unroll 4
            for (int tt = 0; tt < kT; tt += 2) {
                const float4 q = *reinterpret_cast<const float4 *>(row + 2 * tt);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float dl = i ? q.z : q.x;
                    const float dx = i ? q.w : q.y;
                    const float *Bt = Bf + (tt + i) * N + j * NS;
                    const float *Ct = Cf + (tt + i) * N + j * NS;
                    f2 acc{0.f, 0.f};
                    f2 bp[NS / 2], cp[NS / 2];
                    if constexpr (NS % 4 == 0) {
#pragma unroll
                        for (int k = 0; k < NS / 2; k += 2) {
                            const float4 bq = *reinterpret_cast<const float4 *>(Bt + 2 * k);
                            bp[k] = f2{bq.x, bq.y};
                            bp[k + 1 < NS / 2 ? k + 1 : k] = f2{bq.z, bq.w};
                            if (!kSummary) {
                                const float4 cq = *reinterpret_cast<const float4 *>(Ct + 2 * k);
                                cp[k] = f2{cq.x, cq.y};
                                cp[k + 1 < NS / 2 ? k + 1 : k] = f2{cq.z, cq.w};
                            }
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < NS / 2; ++k) {
                            const float2 bq = *reinterpret_cast<const float2 *>(Bt + 2 * k);
                            bp[k] = f2{bq.x, bq.y};
                            if (!kSummary) {
                                const float2 cq = *reinterpret_cast<const float2 *>(Ct + 2 * k);
                                cp[k] = f2{cq.x, cq.y};
                            }
                        }
                    }
#pragma unroll
                    for (int k = 0; k < NS / 2; ++k) {
                        const f2 a = decay2<kFast>(dl, a2[k]);
                        const f2 u = ptx::mul2(f2{dx, dx}, bp[k]);
                        h[k] = ptx::fma2(a, h[k], u);
                        if (!kSummary) acc = ptx::fma2(cp[k], h[k], acc);
                    }
                    if (!kSummary) part[j * LY::kPart + (tt + i) * CPW + sc] = acc.x + acc.y;
                    if (kSummary) dsum += dl;
                }
            }
        }
        __syncwarp();

        // ---------------- epilogue: row t = lane
        if (!kSummary) {
            const int yb = tile & 1;
            unsigned char *ytile = smem + LY::o_y + yb * align128(LY::kTok);
            if (lane == 0) ptx::bulk_wait_read<1>();  // the store that last used this buffer
            __syncwarp();
            float acc[CPW], vx[CPW], vz[CPW];
#pragma unroll
            for (int cc = 0; cc < CPW; cc += 4) {
                float4 a4 = *reinterpret_cast<const float4 *>(part + lane * CPW + cc);
#pragma unroll
                for (int jj = 1; jj < LPC; ++jj) {
                    const float4 v = *reinterpret_cast<const float4 *>(part + jj * LY::kPart +
                                                                       lane * CPW + cc);
                    a4.x += v.x; a4.y += v.y; a4.z += v.z; a4.w += v.w;
                }
                acc[cc] = a4.x; acc[cc + 1] = a4.y; acc[cc + 2] = a4.z; acc[cc + 3] = a4.w;
            }
            Row<TIO, CPW>::load(st + LY::s_x + lane * CPW * sizeof(TIO), vx);
            if (has_z) Row<TIO, CPW>::load(st + LY::s_z + lane * CPW * sizeof(TIO), vz);
#pragma unroll
            for (int cc = 0; cc < CPW; ++cc) {
                float out = fmaf(pD[cc], vx[cc], acc[cc]);
                if (has_z) out *= silu<kFast>(vz[cc]);
                acc[cc] = out;
            }
            Row<TIO, CPW>::store(ytile + lane * CPW * sizeof(TIO), acc);
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                ptx::tma_store_3d(&maps.y, ytile, d0, static_cast<int>(t0), b);
                ptx::bulk_commit();
            }
        }
        __syncwarp();
        // refill this stage with the tile kStages ahead
        if (lane == 0 && tile + kStages < ntiles) issue(tile + kStages);
    }

    if (failed_tile >= 0) {
        if (lane == 0) report_status(status, SSM_ERR_TIMEOUT, kSummary ? 11 : 12);
        // let the copies still in flight land before the block's shared memory is
        // released (each wait again bounded)
        for (int i = failed_tile; i < failed_tile + kStages && i < ntiles; ++i)
            if (!ptx::mbar_wait(&bars[i % kStages], (i / kStages) & 1)) break;
    }
    if (!kSummary && lane == 0) ptx::bulk_wait<0>();

    if (kSummary) {
        const int64_t row = (static_cast<int64_t>(b) * K + c) * D + sd;
        if (sdval) {
#pragma unroll
            for (int k = 0; k < NS / 2; ++k) {
                const int n = j * NS + 2 * k;
                *reinterpret_cast<float2 *>(p.hloc + row * N + n) = make_float2(h[k].x, h[k].y);
            }
            // every lane of the channel accumulated the same sum; one writes it
            if (j == 0) p.dsum[row] = dsum;
        }
    } else if (c == K - 1 && p.h_final && sdval) {
#pragma unroll
        for (int k = 0; k < NS / 2; ++k) {
            const int n = j * NS + 2 * k;
            *reinterpret_cast<float2 *>(p.h_final + (b * D + sd) * N + n) =
                make_float2(h[k].x, h[k].y);
        }
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// 3-D map over a (B, L, W) row-major tensor, box (bw, bt, 1).
bool make_map(CUtensorMap *m, const void *base, bool bf16, int64_t B, int64_t L, int64_t W,
              int bw, int bt) {
    auto enc = encoder();
    if (!enc) return false;
    const size_t e = bf16 ? 2 : 4;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(W), static_cast<cuuint64_t>(L),
                          static_cast<cuuint64_t>(B)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(W * e), static_cast<cuuint64_t>(L * W * e)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(bw), static_cast<cuuint32_t>(bt), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                     3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <typename TIO, int NS, int LPC, bool kSummary>
cudaError_t launch_tma_one(const ScanParams &p, const TmaMaps &maps, int nchunks_grid,
                           cudaStream_t stream) {
    using LY = Layout<TIO, NS, LPC, kSummary>;
    auto kern = scan_tma_kernel<TIO, NS, LPC, kSummary>;
    if (LY::bytes > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             LY::bytes);
        if (e != cudaSuccess) return e;
    }
    dim3 grid(static_cast<unsigned>((p.dim + LY::CPW - 1) / LY::CPW),
              static_cast<unsigned>(p.batch), static_cast<unsigned>(nchunks_grid));
    kern<<<grid, 32, LY::bytes, stream>>>(maps, p);
    return cudaGetLastError();
}

template <typename TIO, int NS, int LPC>
cudaError_t launch_tma_pair(ScanParams p, cudaStream_t stream) {
    using LY = Layout<TIO, NS, LPC, false>;
    const bool bf = std::is_same<TIO, __nv_bfloat16>::value;
    TmaMaps m{};
    const int64_t B = p.batch, L = p.seqlen, D = p.dim, N = p.dstate;
    bool ok = make_map(&m.x, p.x, bf, B, L, D, LY::CPW, kT) &&
              make_map(&m.dl, p.delta, bf, B, L, D, LY::CPW, kT) &&
              make_map(&m.B, p.Bm, bf, B, L, N, static_cast<int>(N), kT) &&
              make_map(&m.C, p.Cm, bf, B, L, N, static_cast<int>(N), kT) &&
              make_map(&m.y, p.y, bf, B, L, D, LY::CPW, kT);
    if (ok && p.z) ok = make_map(&m.z, p.z, bf, B, L, D, LY::CPW, kT);
    if (!ok) return cudaErrorInvalidValue;
    p.clear_status = 1;
    if (p.nchunks > 1) {
        cudaError_t e = launch_tma_one<TIO, NS, LPC, true>(p, m, p.nchunks - 1, stream);
        if (e != cudaSuccess) return e;
        p.clear_status = 0;
    }
    return launch_tma_one<TIO, NS, LPC, false>(p, m, p.nchunks, stream);
}

}  // namespace

int scan_tma_lanes(int64_t dstate) {
    switch (dstate) {
        case 4: return 2;
        case 8: return 2;
        case 16: return kScanLanes16;
        case 32: return 4;
        case 64: return 4;
        default: return 0;
    }
}

bool scan_tma_sizes_ok(int io_bf16, int64_t seqlen, int64_t dim, int64_t dstate) {
    const int64_t e = io_bf16 ? 2 : 4;
    const int lpc = scan_tma_lanes(dstate);
    if (lpc == 0) return false;
    if (io_bf16 && dstate == 4) return false;  // 8-byte B/C rows are below the TMA minimum
    if (dstate * e % 16 != 0 || dim * e % 16 != 0) return false;
    if ((32 / lpc) * e % 16 != 0) return false;
    return seqlen > 0 && seqlen < (int64_t(1) << 31) && dim < (int64_t(1) << 31);
}

bool scan_tma_pointers_ok(const void *const *ptrs, int nptrs) {
    for (int i = 0; i < nptrs; ++i)
        if (ptrs[i] && reinterpret_cast<uintptr_t>(ptrs[i]) % 16 != 0) return false;
    return encoder() != nullptr;
}

cudaError_t launch_scan_tma(const ScanParams &p, cudaStream_t stream) {
    const int64_t N = p.dstate;
    if (p.io_bf16) {
        using T = __nv_bfloat16;
        if (N == 8) return launch_tma_pair<T, 4, 2>(p, stream);
        if (N == 16) return launch_tma_pair<T, 16 / kScanLanes16, kScanLanes16>(p, stream);
        if (N == 32) return launch_tma_pair<T, 8, 4>(p, stream);
        if (N == 64) return launch_tma_pair<T, 16, 4>(p, stream);
    } else {
        using T = float;
        if (N == 4) return launch_tma_pair<T, 2, 2>(p, stream);
        if (N == 8) return launch_tma_pair<T, 4, 2>(p, stream);
        if (N == 16) return launch_tma_pair<T, 16 / kScanLanes16, kScanLanes16>(p, stream);
        if (N == 32) return launch_tma_pair<T, 8, 4>(p, stream);
        if (N == 64) return launch_tma_pair<T, 16, 4>(p, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace ssm
