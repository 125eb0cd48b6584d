// Multi-head selective SSM with a scalar decay per head (Mamba-2 / SSD form).
//
// What it computes ("Mamba-2: 상태 공간 기반 시퀀스 모델", sections "1-세미분리
// 행렬", "멀티-헤드 구조"), per batch b and head h (group g = h / (H / G)):
//   dl_t = softplus(delta_t,h + bias_h),  a_t = exp(dl_t A_h)        (scalars)
//   S_t  = a_t S_{t-1} + dl_t x_t B_t^T        (P x N matrix state)
//   y_t  = S_t C_t + D_h x_t,  optionally * silu(z_t)
//
// This file holds the sequential-recurrence kernel: one lane group per (b, h, p)
// row of the state, N / NS lanes per row, walking time in order.  It is the
// general-shape path (any P, N <= 256, any G, fp32 or bf16); the chunked
// tensor-core form (ssd_tc.cu) runs where its shape rules hold.
#include "common.cuh"
#include "internal.h"

namespace ssm {
namespace {

constexpr int kBlock = 256;

template <typename TIO, int NS, int LPC, bool kFast>
__global__ void __launch_bounds__(kBlock) ssd_recurrent_kernel(SSDParams p) {
    const TIO *__restrict__ gx = static_cast<const TIO *>(p.x);
    const TIO *__restrict__ gdl = static_cast<const TIO *>(p.delta);
    const TIO *__restrict__ gz = static_cast<const TIO *>(p.z);
    const TIO *__restrict__ gB = static_cast<const TIO *>(p.Bm);
    const TIO *__restrict__ gC = static_cast<const TIO *>(p.Cm);
    TIO *__restrict__ gy = static_cast<TIO *>(p.y);

    const int64_t H = p.nheads, P = p.headdim, G = p.ngroups, L = p.seqlen;
    const int N = static_cast<int>(p.dstate);
    const int64_t gid = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    const int64_t row = gid / LPC;  // (b * H + h) * P + pp
    const int j = static_cast<int>(gid % LPC);
    const bool valid = row < p.batch * H * P;
    const int64_t b = valid ? row / (H * P) : 0;
    const int64_t hd = valid ? (row / P) % H : 0;
    const int64_t pp = valid ? row % P : 0;
    const int64_t g = hd / (H / G);

    const float a_s = scale_A<kFast>(p.A[hd]);
    const float bias = p.bias ? p.bias[hd] : 0.f;
    const float Dh = p.Dv ? p.Dv[hd] : 0.f;

    float h[NS];
#pragma unroll
    for (int k = 0; k < NS; ++k) {
        const int n = j * NS + k;
        h[k] = (valid && n < N && p.h0) ? p.h0[row * N + n] : 0.f;
    }
    for (int64_t t = 0; t < L; ++t) {
        const int64_t bt = b * L + t;
        float acc = 0.f, xv = 0.f;
        if (valid) {
            const float dl = step_size<kFast>(Io<TIO>::load(gdl + bt * H + hd), bias, p.softplus);
            const float a = decay<kFast>(dl, a_s);
            xv = Io<TIO>::load(gx + (bt * H + hd) * P + pp);
            const float dx = dl * xv;
            const TIO *Bt = gB + (bt * G + g) * N;
            const TIO *Ct = gC + (bt * G + g) * N;
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                const int n = j * NS + k;
                if (n < N) {
                    h[k] = fmaf(a, h[k], dx * Io<TIO>::load(Bt + n));
                    acc = fmaf(Io<TIO>::load(Ct + n), h[k], acc);
                }
            }
        }
#pragma unroll
        for (int off = LPC / 2; off > 0; off >>= 1)
            acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (valid && j == 0) {
            float out = fmaf(Dh, xv, acc);
            if (gz) out *= silu<kFast>(Io<TIO>::load(gz + (bt * H + hd) * P + pp));
            gy[(bt * H + hd) * P + pp] = Io<TIO>::from_f(out);
        }
    }
    if (valid && p.h_final) {
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            const int n = j * NS + k;
            if (n < N) p.h_final[row * N + n] = h[k];
        }
    }
}

template <typename TIO, int NS, int LPC>
cudaError_t launch_rec(const SSDParams &p, cudaStream_t stream) {
    constexpr bool kFast = std::is_same<TIO, __nv_bfloat16>::value;
    const int64_t threads = p.batch * p.nheads * p.headdim * LPC;
    const unsigned grid = static_cast<unsigned>((threads + kBlock - 1) / kBlock);
    ssd_recurrent_kernel<TIO, NS, LPC, kFast><<<grid, kBlock, 0, stream>>>(p);
    return cudaGetLastError();
}

template <typename TIO> cudaError_t launch_rec_typed(const SSDParams &p, cudaStream_t stream) {
    const int64_t N = p.dstate;
    if (N <= 8) return launch_rec<TIO, 8, 1>(p, stream);
    if (N <= 16) return launch_rec<TIO, 8, 2>(p, stream);
    if (N <= 32) return launch_rec<TIO, 8, 4>(p, stream);
    if (N <= 64) return launch_rec<TIO, 8, 8>(p, stream);
    if (N <= 128) return launch_rec<TIO, 8, 16>(p, stream);
    return launch_rec<TIO, 16, 16>(p, stream);
}

}  // namespace

cudaError_t launch_ssd_recurrent(const SSDParams &p, cudaStream_t stream) {
    return p.io_bf16 ? launch_rec_typed<__nv_bfloat16>(p, stream)
                     : launch_rec_typed<float>(p, stream);
}


cudaError_t launch_ssd(const SSDParams &p, cudaStream_t stream) {
    if (ssd_tc_eligible(p)) return launch_ssd_tc(p, stream);
    return launch_ssd_recurrent(p, stream);
}

}  // namespace ssm
