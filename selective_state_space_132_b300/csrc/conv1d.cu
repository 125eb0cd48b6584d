// Causal depthwise convolution along time with an optional SiLU: the Conv1D (k = 4) +
// SiLU step in front of the selective scan in the block of the tildalice review
// (section "Mamba 블록 아키텍처" and its reference class: a depthwise Conv1D with K - 1
// steps of left padding, cropped to L):
//   out[b, t, d] = silu( bias_d + sum_{k<K} w[d, k] x[b, t - (K-1) + k, d] )
// with x at t < 0 taken from x_prev (the K - 1 inputs just before this call) or zero.
//
// B300 mapping: one read of x and one write of out, so HBM bound.  A thread owns a
// 16-byte chunk of channels (8 bf16 or 4 fp32) of one batch row and walks a run of
// 32 time steps in four batches of 8 rows, loading each batch while the previous one
// is computed (two register buffers), and keeps the last K - 1 inputs in registers;
// a warp reads and writes 512 contiguous bytes per row.  The K taps of its
// channels stay in registers.
// Shapes whose rows cannot be split into aligned 16-byte chunks run one channel per
// thread.
#include <cudaTypedefs.h>

#include "../../include/ssm.h"
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tma_host.cuh"

namespace ssm {
namespace {

constexpr int kBlock = 128;
constexpr int kR = 8;      // rows per batch: one batch is loaded while the previous computes
constexpr int kNB = 4;     // batches per thread
constexpr int kT = kR * kNB;   // time steps per thread
constexpr int kMaxK = 8;


// Raw 16-byte (or one-element) rows and their widening to fp32.
template <typename TIO, int VEC> struct Vec;
template <> struct Vec<__nv_bfloat16, 8> {
    using Raw = uint4;
    static __device__ __forceinline__ Raw zero() { return make_uint4(0, 0, 0, 0); }
    static __device__ __forceinline__ Raw load(const __nv_bfloat16 *p) {
        return __ldg(reinterpret_cast<const uint4 *>(p));
    }
    static __device__ __forceinline__ void widen(const Raw &q, float (&v)[8]) {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, const float (&v)[8]) {
        uint4 q;
        uint32_t *w = &q.x;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&h2);
        }
        *reinterpret_cast<uint4 *>(p) = q;
    }
};
template <> struct Vec<float, 4> {
    using Raw = float4;
    static __device__ __forceinline__ Raw zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
    static __device__ __forceinline__ Raw load(const float *p) {
        return __ldg(reinterpret_cast<const float4 *>(p));
    }
    static __device__ __forceinline__ void widen(const Raw &q, float (&v)[4]) {
        v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    }
    static __device__ __forceinline__ void store(float *p, const float (&v)[4]) {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};
template <typename TIO> struct Vec<TIO, 1> {
    using Raw = TIO;
    static __device__ __forceinline__ Raw zero() { return Io<TIO>::from_f(0.f); }
    static __device__ __forceinline__ Raw load(const TIO *p) { return *p; }
    static __device__ __forceinline__ void widen(const Raw &q, float (&v)[1]) {
        v[0] = Io<TIO>::to_f(q);
    }
    static __device__ __forceinline__ void store(TIO *p, const float (&v)[1]) {
        *p = Io<TIO>::from_f(v[0]);
    }
};

// One thread: VEC channels of one batch row over kT steps.  Consecutive threads take
// consecutive channel chunks, so a warp's loads and stores cover contiguous bytes.
template <typename TIO, int VEC, int K, bool kFast>
__global__ void __launch_bounds__(kBlock) conv1d_kernel(Conv1dParams p) {
    using V = Vec<TIO, VEC>;
    const TIO *__restrict__ gx = static_cast<const TIO *>(p.x);
    const TIO *__restrict__ gprev = static_cast<const TIO *>(p.x_prev);
    TIO *__restrict__ gout = static_cast<TIO *>(p.out);
    const int64_t D = p.dim, L = p.seqlen;
    const int64_t nchunk = (D + VEC - 1) / VEC;
    const int64_t ntb = (L + kT - 1) / kT;
    const int64_t item = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    if (item >= p.batch * ntb * nchunk) return;
    const int64_t ci = item % nchunk;
    const int64_t tb = (item / nchunk) % ntb;
    const int64_t b = item / (nchunk * ntb);
    const int64_t t0 = tb * kT;
    const int64_t d0 = ci * VEC;

    float w[VEC][K], bias[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
        const bool in = d0 + v < D;
#pragma unroll
        for (int k = 0; k < K; ++k) w[v][k] = in ? p.weight[(d0 + v) * K + k] : 0.f;
        bias[v] = (in && p.bias) ? p.bias[d0 + v] : 0.f;
    }
    // the K - 1 inputs before t0 and the first batch of rows are loaded together; each
    // later batch is loaded before the previous one is computed (two register buffers)
    typename V::Raw halo[K > 1 ? K - 1 : 1], cur[kR], nxt[kR];
#pragma unroll
    for (int k = 0; k < K - 1; ++k) {
        const int64_t s = t0 - (K - 1) + k;
        if (s >= 0) halo[k] = V::load(gx + (b * L + s) * D + d0);
        else if (gprev) halo[k] = V::load(gprev + (b * (K - 1) + (K - 1 + s)) * D + d0);
        else halo[k] = V::zero();
    }
    const int nrows = static_cast<int>(min(static_cast<int64_t>(kT), L - t0));
#pragma unroll
    for (int r = 0; r < kR; ++r)
        if (r < nrows) cur[r] = V::load(gx + (b * L + t0 + r) * D + d0);
    // win[k] holds x at t - (K - 1) + k for the step about to be computed
    float win[K][VEC];
#pragma unroll
    for (int k = 0; k < K - 1; ++k) V::widen(halo[k], win[k]);
#pragma unroll
    for (int bi = 0; bi < kNB; ++bi) {
        if (bi + 1 < kNB) {
#pragma unroll
            for (int r = 0; r < kR; ++r) {
                const int rr = (bi + 1) * kR + r;
                if (rr < nrows) nxt[r] = V::load(gx + (b * L + t0 + rr) * D + d0);
            }
        }
#pragma unroll
        for (int r = 0; r < kR; ++r) {
            const int rr = bi * kR + r;
            if (rr < nrows) {
                V::widen(cur[r], win[K - 1]);
                float out[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    float acc = bias[e];
#pragma unroll
                    for (int k = 0; k < K; ++k) acc = fmaf(w[e][k], win[k][e], acc);
                    out[e] = p.silu ? silu<kFast>(acc) : acc;
                }
                V::store(gout + (b * L + t0 + rr) * D + d0, out);
#pragma unroll
                for (int k = 0; k < K - 1; ++k)
#pragma unroll
                    for (int e = 0; e < VEC; ++e) win[k][e] = win[k + 1][e];
            }
        }
#pragma unroll
        for (int r = 0; r < kR; ++r) cur[r] = nxt[r];
    }
}

// ---------------------------------------------------------------- TMA-tiled kernel
// Persistent blocks walk tiles of TT = 128 steps x one 128-byte row of channels (64 bf16
// or 32 fp32) of one batch row.  A block takes a contiguous range of tiles in
// channel-slab-major order, so its taps change only at a slab boundary and consecutive
// tiles are consecutive time strips.  A three-stage TMA pipeline brings each tile with
// its K - 1 halo rows: the box starts K - 1 steps before the tile, and rows before t = 0
// are zero-filled by the TMA unit (or taken from x_prev).  Each thread computes
// RPT = 4 consecutive rows of one 16-byte chunk from shared memory; the outputs go to a
// double-buffered shared tile that one TMA store writes back.  The rows never pass
// through the LSU queue of a thread, and the thread body is small.
#ifndef SSM_CONV_TT
#define SSM_CONV_TT 128
#endif
#ifndef SSM_CONV_STAGES
#define SSM_CONV_STAGES 3
#endif
constexpr int kBlockT = 256;
constexpr int kTT = SSM_CONV_TT;   // steps per tile
constexpr int kStagesT = SSM_CONV_STAGES;
constexpr int kRowB = 128;         // bytes of channels per tile row
constexpr int kStageB = ((kTT + kMaxK - 1) * kRowB + 1023) / 1024 * 1024;
constexpr int kYB = kTT * kRowB;
constexpr int kOffY = kStagesT * kStageB;
constexpr int kOffBar = kOffY + 2 * kYB;
constexpr int kTmaSmem = kOffBar + kStagesT * 8 + 1024;   // + slack to align the base
static_assert(kTT % 32 == 0 && kTT + kMaxK - 1 <= 256, "a TMA box spans at most 256 steps");
static_assert(kStagesT >= 2 && kTmaSmem <= 227 * 1024, "stages must fit in shared memory");

struct Conv1dMaps {
    CUtensorMap x, y;
};

template <typename TIO, int K, bool kFast>
__global__ void __launch_bounds__(kBlockT) conv1d_tma_kernel(const __grid_constant__ Conv1dMaps maps,
                                                             const Conv1dParams p) {
    using V = Vec<TIO, 16 / sizeof(TIO)>;
    constexpr int VEC = 16 / sizeof(TIO);
    constexpr int TD = kRowB / sizeof(TIO);     // channels per tile
    constexpr int CH = kRowB / 16;              // 16-byte chunks per row (8)
    constexpr int RPT = kTT * CH / kBlockT;     // rows per thread (4)
    constexpr uint32_t kTx = (kTT + K - 1) * kRowB;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    DeviceStatus *status = static_cast<DeviceStatus *>(p.status);

    const int tid = threadIdx.x;
    const int q = tid % CH, rg = tid / CH;
    const int64_t D = p.dim, L = p.seqlen;
    // tile indices fit in 32 bits (the host checks the tile count), so the per-tile
    // coordinates take 32-bit divisions
    const uint32_t nds = static_cast<uint32_t>((D + TD - 1) / TD);
    const uint32_t nts = static_cast<uint32_t>((L + kTT - 1) / kTT);
    const uint32_t nstrips = static_cast<uint32_t>(p.batch) * nts;
    const uint32_t ntiles = nds * nstrips;
    // this block's contiguous range [k0, k1) of tiles
    const uint32_t G = gridDim.x, per = ntiles / G, rem = ntiles % G;
    const uint32_t k0 = blockIdx.x * per + (blockIdx.x < rem ? blockIdx.x : rem);
    const uint32_t k1 = k0 + per + (blockIdx.x < rem ? 1 : 0);
    auto coords = [&](uint32_t k, int &d0, int &t0, int &b) {
        const uint32_t slab = k / nstrips, strip = k - slab * nstrips;
        const uint32_t bb = strip / nts;
        d0 = static_cast<int>(slab * TD);
        b = static_cast<int>(bb);
        t0 = static_cast<int>((strip - bb * nts) * kTT);
    };

    if (tid == 0) {
        for (int s = 0; s < kStagesT; ++s) ptx::mbar_init(&bars[s], 1);
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&maps.x);
        ptx::prefetch_tmap(&maps.y);
        for (int s = 0; s < kStagesT && k0 + s < k1; ++s) {
            int d0, t0, b;
            coords(k0 + s, d0, t0, b);
            ptx::mbar_arrive_expect_tx(&bars[s], kTx);
            // a debug-bounds build records a slab start off the 16-byte grid (and loads slab 0)
            const int dc = in_bounds(d0 < D && (d0 * static_cast<int>(sizeof(TIO))) % 16 == 0 &&
                                         b < p.batch && t0 < L, status, 141) ? d0 : 0;
            ptx::tma_load_3d(smem + s * kStageB, &maps.x, &bars[s], dc, t0 - (K - 1), b);
        }
    }
    __syncthreads();

    const TIO *gprev = static_cast<const TIO *>(p.x_prev);
    float wf[VEC * K], bias[VEC];
    int cur_d0 = -1;
    bool cin = false;
    int64_t failed = -1;
    for (uint32_t k = k0; k < k1; ++k) {
        const int it = static_cast<int>(k - k0);
        const int s = it % kStagesT;
        // the y buffer of this tile was last stored two tiles ago
        if (tid == 0) ptx::bulk_wait_read<1>();
        const bool got = ptx::mbar_wait(&bars[s], (it / kStagesT) & 1);
        if (!__syncthreads_and(got ? 1 : 0)) {
            failed = k;
            break;
        }
        int d0, t0, b;
        coords(k, d0, t0, b);
        const int dq = d0 + q * VEC;            // first channel of this thread's chunk
        if (d0 != cur_d0) {
            // the taps of the chunk's VEC channels are VEC * K consecutive floats
            // (16-byte aligned: dq is a multiple of VEC); D is a multiple of VEC, so a
            // chunk is either wholly inside the tensor or wholly past it
            cur_d0 = d0;
            cin = dq < D;
#pragma unroll
            for (int i = 0; i < VEC * K / 4; ++i) {
                const float4 v = cin ? __ldg(reinterpret_cast<const float4 *>(p.weight + dq * K) + i)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                wf[4 * i] = v.x; wf[4 * i + 1] = v.y; wf[4 * i + 2] = v.z; wf[4 * i + 3] = v.w;
            }
#pragma unroll
            for (int i = 0; i < VEC / 4; ++i) {
                const float4 v = (cin && p.bias)
                                     ? __ldg(reinterpret_cast<const float4 *>(p.bias + dq) + i)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                bias[4 * i] = v.x; bias[4 * i + 1] = v.y; bias[4 * i + 2] = v.z;
                bias[4 * i + 3] = v.w;
            }
        }
        const unsigned char *st = smem + s * kStageB;
        unsigned char *yb = smem + kOffY + (it & 1) * kYB;
        // stage row j holds step t0 - (K - 1) + j; output row r needs stage rows r .. r + K - 1
        auto row = [&](int j, float (&v)[VEC]) {
            const int t = t0 - (K - 1) + j;
            if (t < 0 && gprev && cin) {
                V::widen(V::load(gprev + (static_cast<int64_t>(b) * (K - 1) + (K - 1 + t)) * D + dq), v);
            } else {
                V::widen(*reinterpret_cast<const typename V::Raw *>(st + j * kRowB + q * 16), v);
            }
        };
        float win[K][VEC];
#pragma unroll
        for (int kk = 0; kk < K - 1; ++kk) row(rg * RPT + kk, win[kk]);
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int orow = rg * RPT + r;
            row(orow + K - 1, win[K - 1]);
            float out[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                float acc = bias[e];
#pragma unroll
                for (int kk = 0; kk < K; ++kk) acc = fmaf(wf[e * K + kk], win[kk][e], acc);
                out[e] = p.silu ? silu<kFast>(acc) : acc;
            }
            V::store(reinterpret_cast<TIO *>(yb + orow * kRowB + q * 16), out);
#pragma unroll
            for (int kk = 0; kk < K - 1; ++kk)
#pragma unroll
                for (int e = 0; e < VEC; ++e) win[kk][e] = win[kk + 1][e];
        }
        ptx::fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            if (in_bounds(d0 < D && (d0 * static_cast<int>(sizeof(TIO))) % 16 == 0 && b < p.batch &&
                              t0 >= 0 && t0 < L, status, 142))
                ptx::tma_store_3d(&maps.y, yb, d0, t0, b);
            ptx::bulk_commit();
            if (k + kStagesT < k1) {
                int nd0, nt0, nb;
                coords(k + kStagesT, nd0, nt0, nb);
                ptx::mbar_arrive_expect_tx(&bars[s], kTx);
                const int dc = in_bounds(nd0 < D && (nd0 * static_cast<int>(sizeof(TIO))) % 16 == 0 &&
                                             nb < p.batch && nt0 < L, status, 141) ? nd0 : 0;
                ptx::tma_load_3d(smem + s * kStageB, &maps.x, &bars[s], dc, nt0 - (K - 1), nb);
            }
        }
    }
    if (failed >= 0) {
        if (tid == 0) {
            report_status(status, SSM_ERR_TIMEOUT, 40);
            // give every load still in flight one more bounded wait before the shared
            // memory is released
            for (int64_t j = failed; j < failed + kStagesT && j < k1; ++j) {
                const int jt = static_cast<int>(j - k0);
                (void)ptx::mbar_wait(&bars[jt % kStagesT], (jt / kStagesT) & 1);
            }
        }
        __syncthreads();
    }
    if (tid == 0) ptx::bulk_wait<0>();
}

template <typename TIO, int K>
cudaError_t launch_tma_k(const Conv1dParams &p, cudaStream_t stream) {
    constexpr bool kFast = std::is_same<TIO, __nv_bfloat16>::value;
    constexpr int TD = kRowB / sizeof(TIO);
    Conv1dMaps m;
    const bool bf = sizeof(TIO) == 2;
    constexpr int kRowE = kRowB / static_cast<int>(sizeof(TIO));   // channels per tile row
    if (!make_tma_map_3d(&m.x, p.x, bf, p.batch, p.seqlen, p.dim, kRowE, kTT + K - 1, 0) ||
        !make_tma_map_3d(&m.y, p.out, bf, p.batch, p.seqlen, p.dim, kRowE, kTT, 0))
        return cudaErrorInvalidValue;
    auto kern = conv1d_tma_kernel<TIO, K, kFast>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kTmaSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    const int64_t ntiles = p.batch * ((p.seqlen + kTT - 1) / kTT) * ((p.dim + TD - 1) / TD);
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kBlockT, kTmaSmem);
    if (e != cudaSuccess) return e;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * (per_sm > 0 ? per_sm : 1);
    const unsigned grid = static_cast<unsigned>(ntiles < cap ? ntiles : cap);
    kern<<<grid, kBlockT, kTmaSmem, stream>>>(m, p);
    return cudaGetLastError();
}

template <typename TIO> cudaError_t launch_tma(const Conv1dParams &p, cudaStream_t st) {
    switch (p.width) {
        case 1: return launch_tma_k<TIO, 1>(p, st);
        case 2: return launch_tma_k<TIO, 2>(p, st);
        case 3: return launch_tma_k<TIO, 3>(p, st);
        case 4: return launch_tma_k<TIO, 4>(p, st);
        case 5: return launch_tma_k<TIO, 5>(p, st);
        case 6: return launch_tma_k<TIO, 6>(p, st);
        case 7: return launch_tma_k<TIO, 7>(p, st);
        case 8: return launch_tma_k<TIO, 8>(p, st);
        default: return cudaErrorInvalidValue;
    }
}

template <typename TIO, int VEC, int K>
cudaError_t launch_k(const Conv1dParams &p, cudaStream_t stream) {
    constexpr bool kFast = std::is_same<TIO, __nv_bfloat16>::value;
    const int64_t items = p.batch * ((p.seqlen + kT - 1) / kT) * ((p.dim + VEC - 1) / VEC);
    const int64_t blocks = (items + kBlock - 1) / kBlock;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    conv1d_kernel<TIO, VEC, K, kFast><<<static_cast<unsigned>(blocks), kBlock, 0, stream>>>(p);
    return cudaGetLastError();
}
template <typename TIO, int VEC> cudaError_t launch_vec(const Conv1dParams &p, cudaStream_t st) {
    switch (p.width) {
        case 1: return launch_k<TIO, VEC, 1>(p, st);
        case 2: return launch_k<TIO, VEC, 2>(p, st);
        case 3: return launch_k<TIO, VEC, 3>(p, st);
        case 4: return launch_k<TIO, VEC, 4>(p, st);
        case 5: return launch_k<TIO, VEC, 5>(p, st);
        case 6: return launch_k<TIO, VEC, 6>(p, st);
        case 7: return launch_k<TIO, VEC, 7>(p, st);
        case 8: return launch_k<TIO, VEC, 8>(p, st);
        default: return cudaErrorInvalidValue;
    }
}

template <typename TIO> cudaError_t launch_typed(const Conv1dParams &p, cudaStream_t stream) {
    constexpr int kVec = 16 / sizeof(TIO);
    if (conv1d_tma_ok(p)) return launch_tma<TIO>(p, stream);
    const bool vec = p.dim % kVec == 0 &&
                     reinterpret_cast<uintptr_t>(p.x) % 16 == 0 &&
                     reinterpret_cast<uintptr_t>(p.out) % 16 == 0 &&
                     (!p.x_prev || reinterpret_cast<uintptr_t>(p.x_prev) % 16 == 0);
    return vec ? launch_vec<TIO, kVec>(p, stream) : launch_vec<TIO, 1>(p, stream);
}

}  // namespace

int conv1d_max_width() { return kMaxK; }

bool conv1d_tma_ok(const Conv1dParams &p) {
    const size_t e = p.io_bf16 ? 2 : 4;
    auto a16 = [](const void *q) { return reinterpret_cast<uintptr_t>(q) % 16 == 0; };
    if (p.seqlen >= (int64_t(1) << 31) || p.batch >= (int64_t(1) << 31) ||
        p.dim >= (int64_t(1) << 31))
        return false;
    // the kernel indexes its tiles in 32 bits
    const int64_t tiles = p.batch * ((p.seqlen + kTT - 1) / kTT) *
                          ((p.dim * static_cast<int64_t>(e) + kRowB - 1) / kRowB);
    return (p.dim * e) % 16 == 0 && a16(p.x) && a16(p.out) && a16(p.x_prev) && a16(p.weight) &&
           a16(p.bias) && tiles < (int64_t(1) << 31) && tma_encoder() != nullptr;
}

cudaError_t launch_conv1d(const Conv1dParams &p, cudaStream_t stream) {
    return p.io_bf16 ? launch_typed<__nv_bfloat16>(p, stream) : launch_typed<float>(p, stream);
}

}  // namespace ssm
