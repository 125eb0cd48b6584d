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
#include "common.cuh"
#include "internal.h"

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
    const bool vec = p.dim % kVec == 0 &&
                     reinterpret_cast<uintptr_t>(p.x) % 16 == 0 &&
                     reinterpret_cast<uintptr_t>(p.out) % 16 == 0 &&
                     (!p.x_prev || reinterpret_cast<uintptr_t>(p.x_prev) % 16 == 0);
    return vec ? launch_vec<TIO, kVec>(p, stream) : launch_vec<TIO, 1>(p, stream);
}

}  // namespace

int conv1d_max_width() { return kMaxK; }

cudaError_t launch_conv1d(const Conv1dParams &p, cudaStream_t stream) {
    return p.io_bf16 ? launch_typed<__nv_bfloat16>(p, stream) : launch_typed<float>(p, stream);
}

}  // namespace ssm
