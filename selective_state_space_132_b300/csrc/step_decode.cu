// One recurrent decode step (tildalice.io Mamba review, section "추론 속도": the
// state has a fixed O(D x N) size and no cache grows with the sequence).  For
// every sequence b and channel d, with one new token:
//   dl = softplus(delta + bias_d)
//   h  = exp(dl A_d) (.) h + (dl x) B          (state read and written in place)
//   y  = (C . h + D_d x) * silu(z)
//
// B300 mapping: the step is a pure fp32 read-modify-write of the (B, D, N)
// state plus a few bytes per token, so it is HBM bound (or L2 bound when the
// state fits in the 126 MB L2).  Each thread owns eight (or four) consecutive states
// of one (b, d) row and moves them with 16-byte loads and stores; the lanes of a row
// are adjacent, so a warp touches a contiguous 1 KB span, and the readout is reduced
// with xor shuffles inside those lanes.
#include "common.cuh"
#include "internal.h"

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
    return p.io_bf16 ? launch_typed<__nv_bfloat16>(p, stream) : launch_typed<float>(p, stream);
}

}  // namespace ssm
