// One recurrent decode step (tildalice.io Mamba review, section "추론 속도": the
// state has a fixed O(D x N) size and no cache grows with the sequence).  For
// every sequence b and channel d, with one new token:
//   dl = softplus(delta + bias_d)
//   h  = exp(dl A_d) (.) h + (dl x) B          (state read and written in place)
//   y  = (C . h + D_d x) * silu(z)
//
// B300 mapping: the step is a pure fp32 read-modify-write of the (B, D, N)
// state plus a few bytes per token, so it is HBM bound (or L2 bound when the
// state fits in the 126 MB L2).
//   * Fast path (decode_tma_kernel): a persistent grid of blocks that stream tiles of
//     R consecutive (b, d) rows through shared memory.  One thread issues bulk copies
//     (cp.async.bulk) of a tile's state and its x, delta and z into a two-stage
//     buffer; the block updates the state in shared memory (each thread eight states
//     of one row), and one bulk copy writes the tile's state back while the next
//     tile is already arriving.  A block keeps two tiles in flight, so an SM holds
//     about 100 KB of outstanding HBM traffic instead of the 32 bytes per resident
//     thread that register loads give; that is what brings the step near the speed
//     of a plain copy of the state.
//   * Other shapes and unaligned pointers: each thread owns eight (or four)
//     consecutive states of one (b, d) row and moves them with 16-byte loads and
//     stores; the lanes of a row are adjacent, so a warp touches a contiguous 1 KB
//     span, and the readout is reduced with xor shuffles inside those lanes.
#include "../../include/ssm.h"

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace ssm {
namespace {

constexpr int kBlock = 256;

// Four consecutive I/O values (B or C of one lane's states) as floats.
template <typename TIO> __device__ __forceinline__ void load4(const TIO *p, float (&v)[4]);
template <> __device__ __forceinline__ void load4<float>(const float *p, float (&v)[4]) {
    const float4 q = __ldg(reinterpret_cast<const float4 *>(p));
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16 *p, float (&v)[4]) {
    const uint2 q = __ldg(reinterpret_cast<const uint2 *>(p));
    v[0] = __uint_as_float(q.x << 16); v[1] = __uint_as_float(q.x & 0xffff0000u);
    v[2] = __uint_as_float(q.y << 16); v[3] = __uint_as_float(q.y & 0xffff0000u);
}

template <typename TIO, int NS, int LPC, bool kFast, bool kVec>
__global__ void __launch_bounds__(kBlock) decode_kernel(DecodeParams p) {
    const TIO *__restrict__ gx = static_cast<const TIO *>(p.x);
    const TIO *__restrict__ gdl = static_cast<const TIO *>(p.delta);
    const TIO *__restrict__ gz = static_cast<const TIO *>(p.z);
    const TIO *__restrict__ gB = static_cast<const TIO *>(p.Bm);
    const TIO *__restrict__ gC = static_cast<const TIO *>(p.Cm);
    TIO *__restrict__ gy = static_cast<TIO *>(p.y);

    const int64_t D = p.dim;
    const int N = static_cast<int>(p.dstate);
    const int64_t gid = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    const int64_t row = gid / LPC;   // b * D + d
    const int j = static_cast<int>(gid % LPC);
    const bool valid = row < p.batch * D;
    const int64_t b = valid ? row / D : 0;
    const int64_t d = valid ? row % D : 0;

    float acc = 0.f, xv = 0.f;
    if (valid) {
        const int n0 = j * NS;
        float *st = p.state + row * N + n0;
        float h[NS], a[NS], bv[NS], cv[NS];
        // issue the state loads first: they are the long-latency HBM traffic
        if (kVec) {
#pragma unroll
            for (int k = 0; k < NS; k += 4) {
                const float4 s4 = *reinterpret_cast<const float4 *>(st + k);
                h[k] = s4.x; h[k + 1] = s4.y; h[k + 2] = s4.z; h[k + 3] = s4.w;
            }
#pragma unroll
            for (int k = 0; k < NS; k += 4) {
                const float4 a4 = __ldg(reinterpret_cast<const float4 *>(p.A + d * N + n0 + k));
                a[k] = a4.x; a[k + 1] = a4.y; a[k + 2] = a4.z; a[k + 3] = a4.w;
                float t4[4];
                load4<TIO>(gB + b * N + n0 + k, t4);
                bv[k] = t4[0]; bv[k + 1] = t4[1]; bv[k + 2] = t4[2]; bv[k + 3] = t4[3];
                load4<TIO>(gC + b * N + n0 + k, t4);
                cv[k] = t4[0]; cv[k + 1] = t4[1]; cv[k + 2] = t4[2]; cv[k + 3] = t4[3];
            }
        } else {
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                const bool in = n0 + k < N;
                h[k] = in ? st[k] : 0.f;
                a[k] = in ? __ldg(p.A + d * N + n0 + k) : 0.f;
                bv[k] = in ? Io<TIO>::load(gB + b * N + n0 + k) : 0.f;
                cv[k] = in ? Io<TIO>::load(gC + b * N + n0 + k) : 0.f;
            }
        }
        xv = Io<TIO>::load(gx + row);
        const float bias = p.bias ? __ldg(p.bias + d) : 0.f;
        const float dl = step_size<kFast>(Io<TIO>::load(gdl + row), bias, p.softplus);
        const float dx = dl * xv;
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            const float da = decay<kFast>(dl, scale_A<kFast>(a[k]));
            float w = dx * bv[k];
            if (p.zoh)  // zero-order hold: ((exp(dl A) - 1) / A) B x
                w = zoh_coef<kFast>(dl, dl * a[k], da, a[k] != 0.f ? 1.f / a[k] : 0.f) * xv * bv[k];
            h[k] = fmaf(da, h[k], w);
            acc = fmaf(cv[k], h[k], acc);
        }
        if (kVec) {
#pragma unroll
            for (int k = 0; k < NS; k += 4)
                *reinterpret_cast<float4 *>(st + k) = make_float4(h[k], h[k + 1], h[k + 2], h[k + 3]);
        } else {
#pragma unroll
            for (int k = 0; k < NS; ++k)
                if (n0 + k < N) st[k] = h[k];
        }
    }
#pragma unroll
    for (int off = LPC / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (valid && j == 0) {
        float out = acc + (p.Dv ? __ldg(p.Dv + d) * xv : 0.f);
        if (gz) out *= silu<kFast>(Io<TIO>::load(gz + row));
        gy[row] = Io<TIO>::from_f(out);
    }
}


// ---------------------------------------------------------------- bulk-copy fast path
constexpr int kTmaThreads = 256;
constexpr int kTmaStages = 2;

// Shared-memory stage of one tile of R rows: the fp32 state (R x N), then x, delta and
// z of the tile (R values each, I/O type), each part a multiple of 16 bytes.
template <typename TIO, int N> struct TmaTile {
    static constexpr int LPC = N / 8;                 // threads per row, eight states each
    static constexpr int R = kTmaThreads / LPC;       // rows per tile
    static constexpr int E = sizeof(TIO);
    static constexpr int o_x = R * N * 4;
    static constexpr int o_dl = o_x + R * E;
    static constexpr int o_z = o_dl + R * E;
    static constexpr int stage = o_z + R * E;
    static constexpr int bytes = kTmaStages * stage + kTmaStages * 8 + 128;
};

__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(ptx::smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(ptx::smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void bulk_store(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(ptx::smem_u32(src)), "r"(bytes)
                 : "memory");
}

template <typename TIO> __device__ __forceinline__ float io_at(const unsigned char *base, int i) {
    return Io<TIO>::to_f(reinterpret_cast<const TIO *>(base)[i]);
}

// Eight consecutive values of B or C (I/O type) as floats.
template <typename TIO> __device__ __forceinline__ void load8(const TIO *p, float (&v)[8]) {
    float t[4];
    load4<TIO>(p, t);
    v[0] = t[0]; v[1] = t[1]; v[2] = t[2]; v[3] = t[3];
    load4<TIO>(p + 4, t);
    v[4] = t[0]; v[5] = t[1]; v[6] = t[2]; v[7] = t[3];
}

template <typename TIO, int N, bool kFast, bool kGate, bool kZoh>
__global__ void __launch_bounds__(kTmaThreads, 5) decode_tma_kernel(DecodeParams p, int ntiles) {
    using TT = TmaTile<TIO, N>;
    constexpr int R = TT::R, LPC = TT::LPC;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kTmaStages * TT::stage);
    const TIO *gx = static_cast<const TIO *>(p.x);
    const TIO *gdl = static_cast<const TIO *>(p.delta);
    const TIO *gz = static_cast<const TIO *>(p.z);
    const TIO *gB = static_cast<const TIO *>(p.Bm);
    const TIO *gC = static_cast<const TIO *>(p.Cm);
    TIO *gy = static_cast<TIO *>(p.y);
    DeviceStatus *status = static_cast<DeviceStatus *>(p.status);
    const int tid = threadIdx.x;
    // 32-bit indexing: the host takes this path only when B * D * N < 2^31
    const int D = static_cast<int>(p.dim), rows = static_cast<int>(p.batch * p.dim);

    if (tid == 0) {
        for (int s = 0; s < kTmaStages; ++s) ptx::mbar_init(&bars[s], 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    // tiles blockIdx.x, blockIdx.x + gridDim.x, ...; the last one may be short
    const int my = (ntiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                   static_cast<int>(gridDim.x);
    auto tile_row = [&](int i) { return (static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x)) * R; };
    auto tile_rows = [&](int i) {
        const int r0 = tile_row(i);
        return static_cast<uint32_t>(rows - r0 < R ? rows - r0 : R);
    };
    auto issue = [&](int i) {  // thread 0 only
        unsigned char *st = smem + (i % kTmaStages) * TT::stage;
        uint64_t *bar = &bars[i % kTmaStages];
        const int r0 = tile_row(i);
        const uint32_t nr = tile_rows(i);
        // bulk copies need 16-byte aligned, whole 16-byte spans inside the tensors; a
        // debug-bounds build records a tile that breaks this and completes its stage empty
        if (!in_bounds(r0 >= 0 && nr > 0 && nr <= static_cast<uint32_t>(R) && r0 + nr <= rows &&
                           (r0 * TT::E) % 16 == 0 && (nr * TT::E) % 16 == 0, status, 131)) {
            ptx::mbar_arrive_expect_tx(bar, 0);
            return;
        }
        ptx::mbar_arrive_expect_tx(bar, nr * (N * 4 + (kGate ? 3 : 2) * TT::E));
        bulk_load(st, p.state + static_cast<int64_t>(r0) * N, nr * N * 4, bar);
        bulk_load(st + TT::o_x, gx + r0, nr * TT::E, bar);
        bulk_load(st + TT::o_dl, gdl + r0, nr * TT::E, bar);
        if (kGate) bulk_load(st + TT::o_z, gz + r0, nr * TT::E, bar);
    };
    if (tid == 0)
        for (int i = 0; i < kTmaStages && i < my; ++i) issue(i);

    const int rr = tid / LPC, j = tid % LPC;
    bool ok = true;
    for (int i = 0; i < my; ++i) {
        const int s = i % kTmaStages;
        unsigned char *stg = smem + s * TT::stage;
        const int row = tile_row(i) + rr;
        const bool valid = row < rows;
        const int b = valid ? row / D : 0, d = valid ? row - b * D : 0;
        // inputs that do not come through the stage are fetched before waiting on it
        float a[8], bv[8], cv[8];
        float bias = 0.f, Dd = 0.f;
        if (valid) {
            const float4 a0 = __ldg(reinterpret_cast<const float4 *>(p.A + d * N + 8 * j));
            const float4 a1 = __ldg(reinterpret_cast<const float4 *>(p.A + d * N + 8 * j + 4));
            a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
            a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
            load8<TIO>(gB + b * N + 8 * j, bv);
            load8<TIO>(gC + b * N + 8 * j, cv);
            bias = p.bias ? __ldg(p.bias + d) : 0.f;
            Dd = p.Dv ? __ldg(p.Dv + d) : 0.f;
        }
        // the block agrees on the wait's outcome so that it never splits
        ok = __syncthreads_and(ptx::mbar_wait(&bars[s], static_cast<uint32_t>(i / kTmaStages) & 1u) ? 1 : 0) != 0;
        if (!ok) {
            if (tid == 0) report_status(status, SSM_ERR_TIMEOUT, 41);
            break;
        }
        float acc = 0.f, xv = 0.f;
        float *st = reinterpret_cast<float *>(stg) + rr * N + 8 * j;
        if (valid) {
            xv = io_at<TIO>(stg + TT::o_x, rr);
            const float dl = step_size<kFast>(io_at<TIO>(stg + TT::o_dl, rr), bias, p.softplus);
            const float dx = dl * xv;
            const float4 s0 = *reinterpret_cast<const float4 *>(st);
            const float4 s1 = *reinterpret_cast<const float4 *>(st + 4);
            float h[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float da = decay<kFast>(dl, scale_A<kFast>(a[k]));
                float w = dx * bv[k];
                if (kZoh)  // zero-order hold: ((exp(dl A) - 1) / A) B x
                    w = zoh_coef<kFast>(dl, dl * a[k], da, a[k] != 0.f ? 1.f / a[k] : 0.f) * xv *
                        bv[k];
                h[k] = fmaf(da, h[k], w);
                acc = fmaf(cv[k], h[k], acc);
            }
            *reinterpret_cast<float4 *>(st) = make_float4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<float4 *>(st + 4) = make_float4(h[4], h[5], h[6], h[7]);
        }
#pragma unroll
        for (int off = LPC / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (valid && j == 0) {
            float out = acc + Dd * xv;
            if (kGate) out *= silu<kFast>(io_at<TIO>(stg + TT::o_z, rr));
            gy[row] = Io<TIO>::from_f(out);
        }
        ptx::fence_proxy_async_smem();  // the state written here is read by the bulk store
        __syncthreads();
        if (tid == 0) {
            if (in_bounds(tile_row(i) + tile_rows(i) <= rows, status, 132))
                bulk_store(p.state + static_cast<int64_t>(tile_row(i)) * N, stg, tile_rows(i) * N * 4);
            ptx::bulk_commit();
            if (i + kTmaStages < my) {
                ptx::bulk_wait_read<0>();  // the stage's bytes have left shared memory
                issue(i + kTmaStages);
            }
        }
    }
    if (!ok && tid == 0) {
        // let the loads still in flight land before the block's shared memory is released
        // (each wait again bounded)
        for (int s = 0; s < kTmaStages; ++s)
            if (!ptx::mbar_wait(&bars[s], 0) && !ptx::mbar_wait(&bars[s], 1)) break;
    }
    if (tid == 0) ptx::bulk_wait<0>();
}

template <typename TIO, int NS, int LPC>
cudaError_t launch_lpc(const DecodeParams &p, cudaStream_t stream) {
    constexpr bool kFast = std::is_same<TIO, __nv_bfloat16>::value;
    // the vector path needs whole rows of NS-state slots and aligned row starts
    const size_t e = sizeof(TIO);
    const bool vec = (p.dstate == NS * LPC) &&
                     (reinterpret_cast<uintptr_t>(p.state) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(p.A) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(p.Bm) % (4 * e) == 0) &&
                     (reinterpret_cast<uintptr_t>(p.Cm) % (4 * e) == 0);
    const int64_t threads = p.batch * p.dim * LPC;
    const unsigned grid = static_cast<unsigned>((threads + kBlock - 1) / kBlock);
    if (vec)
        decode_kernel<TIO, NS, LPC, kFast, true><<<grid, kBlock, 0, stream>>>(p);
    else
        decode_kernel<TIO, NS, LPC, kFast, false><<<grid, kBlock, 0, stream>>>(p);
    return cudaGetLastError();
}


// The bulk-copy path needs N a multiple of 8 (8 .. 64), 16-byte aligned state, A, B, C
// and token rows, and a row count whose token bytes stay on 16-byte boundaries.
template <typename TIO, int N, bool kGate, bool kZoh>
cudaError_t launch_tma_k(const DecodeParams &p, int ntiles, cudaStream_t stream) {
    using TT = TmaTile<TIO, N>;
    constexpr bool kFast = std::is_same<TIO, __nv_bfloat16>::value;
    auto kern = decode_tma_kernel<TIO, N, kFast, kGate, kZoh>;
    static int per_sm = 0;  // resident blocks per SM, found once per instantiation
    if (per_sm == 0) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TT::bytes);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kTmaThreads, TT::bytes);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) per_sm = 1;
    }
    const int64_t slots = static_cast<int64_t>(device_sm_count()) * per_sm;
    const unsigned grid = static_cast<unsigned>(ntiles < slots ? ntiles : slots);
    kern<<<grid, kTmaThreads, TT::bytes, stream>>>(p, ntiles);
    return cudaGetLastError();
}

// The bulk-copy path needs N a multiple of 8 (8 .. 64), 16-byte aligned state, A, B, C
// and token rows, and a row count whose token bytes stay on 16-byte boundaries.
template <typename TIO, int N>
cudaError_t launch_tma_n(const DecodeParams &p, cudaStream_t stream, bool *taken) {
    using TT = TmaTile<TIO, N>;
    const int64_t rows = p.batch * p.dim;
    const int ntiles = static_cast<int>((rows + TT::R - 1) / TT::R);
    auto a16 = [](const void *q) { return reinterpret_cast<uintptr_t>(q) % 16 == 0; };
    const bool ok = rows * N < (int64_t(1) << 31) && (rows * TT::E) % 16 == 0 && a16(p.state) && a16(p.A) && a16(p.x) &&
                    a16(p.delta) && (!p.z || a16(p.z)) && a16(p.Bm) && a16(p.Cm);
    *taken = ok;
    if (!ok) return cudaSuccess;
    if (p.z)
        return p.zoh ? launch_tma_k<TIO, N, true, true>(p, ntiles, stream)
                     : launch_tma_k<TIO, N, true, false>(p, ntiles, stream);
    return p.zoh ? launch_tma_k<TIO, N, false, true>(p, ntiles, stream)
                 : launch_tma_k<TIO, N, false, false>(p, ntiles, stream);
}

template <typename TIO>
cudaError_t launch_tma(const DecodeParams &p, cudaStream_t stream, bool *taken) {
    *taken = false;
    switch (p.dstate) {
        case 8: return launch_tma_n<TIO, 8>(p, stream, taken);
        case 16: return launch_tma_n<TIO, 16>(p, stream, taken);
        case 32: return launch_tma_n<TIO, 32>(p, stream, taken);
        case 64: return launch_tma_n<TIO, 64>(p, stream, taken);
        default: return cudaSuccess;
    }
}

// Eight states per thread where N allows (two 16-byte state accesses in flight per
// thread keep more HBM traffic outstanding), four otherwise.
template <typename TIO> cudaError_t launch_typed(const DecodeParams &p, cudaStream_t stream) {
    const int64_t N = p.dstate;
    if (N <= 4) return launch_lpc<TIO, 4, 1>(p, stream);
    if (N <= 8) return launch_lpc<TIO, 8, 1>(p, stream);
    if (N <= 16) return launch_lpc<TIO, 8, 2>(p, stream);
    if (N <= 32) return launch_lpc<TIO, 8, 4>(p, stream);
    return launch_lpc<TIO, 8, 8>(p, stream);
}

}  // namespace

cudaError_t launch_decode(const DecodeParams &p, cudaStream_t stream) {
    bool taken = false;
    cudaError_t e = p.io_bf16 ? launch_tma<__nv_bfloat16>(p, stream, &taken)
                              : launch_tma<float>(p, stream, &taken);
    if (e != cudaSuccess || taken) return e;
    return p.io_bf16 ? launch_typed<__nv_bfloat16>(p, stream) : launch_typed<float>(p, stream);
}

}  // namespace ssm
