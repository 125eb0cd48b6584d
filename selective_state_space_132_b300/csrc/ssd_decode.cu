// One recurrent decode step of the multi-head scalar-A SSM (Mamba-2 form): the
// single-token counterpart of the chunked SSD kernel ("Mamba-2: 상태 공간 기반 시퀀스
// 모델", section "멀티-헤드 구조"; tildalice review, section "추론 속도" for the fixed-size
// state).  For every sequence b and head h (group g = h / (H / G)):
//   dl = softplus(delta_h + bias_h),   S[p, :] <- exp(dl A_h) S[p, :] + dl x_p B
//   y_p = S[p, :] . C + D_h x_p       (times silu(z_p) with a gate)
// The (B, H, P, N) fp32 state is read and written in place.
//
// B300 mapping: a pure read-modify-write of the state, HBM bound.  Each thread owns
// NS = 8 consecutive states of one (b, h, p) row (two 16-byte loads and stores in
// flight per thread), the N / 8 lanes of a row are adjacent (a warp covers a
// contiguous 1 KB), B and C arrive as one 16-byte load each (bf16) and the readout
// is reduced with xor shuffles inside the row's lanes.
#include "common.cuh"
#include "internal.h"

namespace ssm {
namespace {

constexpr int kBlock = 256;
constexpr int kNS = 8;

template <typename TIO> __device__ __forceinline__ void load8(const TIO *p, float (&v)[8]);
template <> __device__ __forceinline__ void load8<float>(const float *p, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p + 4));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16 *p, float (&v)[8]) {
    const uint4 q = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

template <typename TIO, int LPC, bool kFast, bool kVec>
__global__ void __launch_bounds__(kBlock) ssd_decode_kernel(SSDDecodeParams p) {
    const TIO *__restrict__ gx = static_cast<const TIO *>(p.x);
    const TIO *__restrict__ gdl = static_cast<const TIO *>(p.delta);
    const TIO *__restrict__ gz = static_cast<const TIO *>(p.z);
    const TIO *__restrict__ gB = static_cast<const TIO *>(p.Bm);
    const TIO *__restrict__ gC = static_cast<const TIO *>(p.Cm);
    TIO *__restrict__ gy = static_cast<TIO *>(p.y);

    const int64_t H = p.nheads, P = p.headdim, G = p.ngroups;
    const int N = static_cast<int>(p.dstate);
    const int64_t gid = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    const int64_t row = gid / LPC;  // (b * H + h) * P + pp
    const int j = static_cast<int>(gid % LPC);
    const bool valid = row < p.batch * H * P;
    const int64_t bh = valid ? row / P : 0;
    const int64_t b = bh / H, h = bh % H;
    const int64_t g = h / (H / G);

    float acc = 0.f, xv = 0.f;
    if (valid) {
        const int n0 = j * kNS;
        float *st = p.state + row * N + n0;
        float s[kNS], bv[kNS], cv[kNS];
        if (kVec) {
            const float4 s0 = *reinterpret_cast<const float4 *>(st);
            const float4 s1 = *reinterpret_cast<const float4 *>(st + 4);
            s[0] = s0.x; s[1] = s0.y; s[2] = s0.z; s[3] = s0.w;
            s[4] = s1.x; s[5] = s1.y; s[6] = s1.z; s[7] = s1.w;
            load8<TIO>(gB + (b * G + g) * N + n0, bv);
            load8<TIO>(gC + (b * G + g) * N + n0, cv);
        } else {
#pragma unroll
            for (int k = 0; k < kNS; ++k) {
                const bool in = n0 + k < N;
                s[k] = in ? st[k] : 0.f;
                bv[k] = in ? Io<TIO>::load(gB + (b * G + g) * N + n0 + k) : 0.f;
                cv[k] = in ? Io<TIO>::load(gC + (b * G + g) * N + n0 + k) : 0.f;
            }
        }
        xv = Io<TIO>::load(gx + row);
        const float bias = p.bias ? __ldg(p.bias + h) : 0.f;
        const float dl = step_size<kFast>(Io<TIO>::load(gdl + bh), bias, p.softplus);
        const float a = decay<kFast>(dl, scale_A<kFast>(__ldg(p.A + h)));
        const float dx = dl * xv;
#pragma unroll
        for (int k = 0; k < kNS; ++k) {
            s[k] = fmaf(a, s[k], dx * bv[k]);
            acc = fmaf(cv[k], s[k], acc);
        }
        if (kVec) {
            *reinterpret_cast<float4 *>(st) = make_float4(s[0], s[1], s[2], s[3]);
            *reinterpret_cast<float4 *>(st + 4) = make_float4(s[4], s[5], s[6], s[7]);
        } else {
#pragma unroll
            for (int k = 0; k < kNS; ++k)
                if (n0 + k < N) st[k] = s[k];
        }
    }
#pragma unroll
    for (int off = LPC / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (valid && j == 0) {
        float out = acc + (p.Dv ? __ldg(p.Dv + h) * xv : 0.f);
        if (gz) out *= silu<kFast>(Io<TIO>::load(gz + row));
        gy[row] = Io<TIO>::from_f(out);
    }
}

template <typename TIO, int LPC>
cudaError_t launch_lpc(const SSDDecodeParams &p, cudaStream_t stream) {
    constexpr bool kFast = std::is_same<TIO, __nv_bfloat16>::value;
    const size_t e = sizeof(TIO);
    const bool vec = (p.dstate == kNS * LPC) &&
                     (reinterpret_cast<uintptr_t>(p.state) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(p.Bm) % (8 * e) == 0) &&
                     (reinterpret_cast<uintptr_t>(p.Cm) % (8 * e) == 0);
    const int64_t threads = p.batch * p.nheads * p.headdim * LPC;
    const unsigned grid = static_cast<unsigned>((threads + kBlock - 1) / kBlock);
    if (vec)
        ssd_decode_kernel<TIO, LPC, kFast, true><<<grid, kBlock, 0, stream>>>(p);
    else
        ssd_decode_kernel<TIO, LPC, kFast, false><<<grid, kBlock, 0, stream>>>(p);
    return cudaGetLastError();
}

template <typename TIO>
cudaError_t launch_typed(const SSDDecodeParams &p, cudaStream_t stream) {
    const int64_t N = p.dstate;
    if (N <= 8) return launch_lpc<TIO, 1>(p, stream);
    if (N <= 16) return launch_lpc<TIO, 2>(p, stream);
    if (N <= 32) return launch_lpc<TIO, 4>(p, stream);
    if (N <= 64) return launch_lpc<TIO, 8>(p, stream);
    if (N <= 128) return launch_lpc<TIO, 16>(p, stream);
    return launch_lpc<TIO, 32>(p, stream);
}

}  // namespace

cudaError_t launch_ssd_decode(const SSDDecodeParams &p, cudaStream_t stream) {
    return p.io_bf16 ? launch_typed<__nv_bfloat16>(p, stream) : launch_typed<float>(p, stream);
}

}  // namespace ssm
