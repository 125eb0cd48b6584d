// Backward pass of the selective scan: gradients of x, the raw step, A, B, C, D,
// the step bias, z and the initial state, from the gradient of y (and of the final
// state).  The pages ask that the backward pass rebuild the hidden states from the
// inputs instead of keeping them from the forward pass (tildalice review, section
// "Hardware-Aware 병렬 알고리즘", item "역전파 시 재계산"; yongggg review, section
// "하드웨어 인식 알고리즘").  The arithmetic is the adjoint of the recurrence
//   h_t = exp(dl_t A) h_{t-1} + c_t B_t x_t,  c_t = dl_t (Euler) or (exp(dl_t A) - 1)/A
//   y_t = (C_t . h_t + D x_t) silu(z_t):
// with lam = dLoss/dh_t walking back in time,
//   g_t    = dy_t silu(z_t)                  (gradient of C.h + D x)
//   dz_t   = dy_t (C_t.h_t + D x_t) silu'(z_t)
//   dC_t  += g_t h_t          lam += g_t C_t
//   dB_t  += lam c_t x_t      dx_t = g_t D + sum_n lam c_t B_t
//   ddl_t  = sum_n lam (h_{t-1} a A + B_t x_t dc/ddl)
//   dA    += lam (h_{t-1} a dl_t + B_t x_t dc/dA)
//   lam   *= a                (now dLoss/dh_{t-1})
//   ddelta_t = ddl_t softplus'(delta_t + bias), dbias += ddelta_t, dh0 = lam at the start.
//
// B300 mapping.  A block owns 32 channels of one batch row (4 warps x 8 channels x
// 4 lanes, each lane NS = ceil(N/4) states), the same split as the forward kernel.
//   1. Checkpoint pass: the forward recurrence over the whole sequence, storing the
//      state at the start of every T-step tile in the workspace (B, ntiles, D, N).
//   2. Reverse pass, tile by tile from the last: stage the tile's rows (x, step, z, dy)
//      and B, C in shared memory; recompute the tile's states from its checkpoint into
//      shared memory; walk the tile backwards carrying lam in registers.
//   Row quantities (dx, ddl) are summed over a channel's 4 lanes with shuffles.  dB
//   and dC are sums over channels: a reduce-scatter over the 8 channels of a warp
//   (shuffles), a sum over the 4 warps in shared memory, then one fp32 atomic add per
//   (t, n) and block into the output.  dA, dD and dbias are summed in registers over
//   the sequence and added atomically at the end.
#include "../../include/ssm.h"
#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"
#include "internal.h"

namespace ssm {
namespace {

constexpr int kCB = 32;          // channels per block
constexpr int kThreads = 128;

#ifndef SSM_BWD_TILE_NS4
#define SSM_BWD_TILE_NS4 16
#endif
template <int NS> struct BwdShape {
    static constexpr int NP = 4 * NS;                            // padded state count
    // steps per tile (and between checkpoints)
    static constexpr int T = NS <= 2 ? 32 : (NS == 4 ? SSM_BWD_TILE_NS4 : 64 / NS);
    static_assert(NS % 2 == 0, "states are processed in packed pairs");
    // the forward kernels' 32-step tiles hold whole checkpoint intervals, and their 4-step
    // blocks start at every checkpoint
    static_assert(T >= 4 && T <= 32 && (T & (T - 1)) == 0, "T must be a power of two in [4, 32]");
    static constexpr int kRows = 9;                              // per-(t, channel) arrays
    static constexpr size_t floats = static_cast<size_t>(T) * kCB * NP   // states
                                     + 2 * T * NP                        // B, C
                                     + kRows * T * kCB                   // rows
                                     + T * 4 * 2 * NP;                   // dB/dC partials
    static constexpr size_t bytes = floats * sizeof(float);
};

__device__ __forceinline__ float sigmoid_f(float v, bool fast) {
    return fast ? __fdividef(1.f, 1.f + ex2_approx(-v * kLog2e)) : 1.f / (1.f + expf(-v));
}

// dc/dA of the zero-order-hold coefficient c = (exp(v) - 1) / A, v = dl A:
// dl^2 f(v), f(v) = (v e^v - e^v + 1) / v^2 = sum_j (j + 1) v^j / (j + 2)!.  The
// series (seven terms, error < 2e-9 relative) below |v| = 1/4; the closed form, with
// a = e^v and invA = 1 / A, above.
template <bool kFast>
__device__ __forceinline__ float zoh_dc_dA(float dl, float v, float a, float invA) {
    float f = 1.f / 5760.f;
    f = fmaf(f, v, 1.f / 840.f);
    f = fmaf(f, v, 1.f / 144.f);
    f = fmaf(f, v, 1.f / 30.f);
    f = fmaf(f, v, 1.f / 8.f);
    f = fmaf(f, v, 1.f / 3.f);
    f = fmaf(f, v, 0.5f);
    const float em1 = kFast ? a - 1.f : expm1f(v);
    const float direct = (dl * a - em1 * invA) * invA;
    return fabsf(v) < 0.25f ? dl * dl * f : direct;
}

// One level of a reduce-scatter over a lane mask: each lane keeps half of its 2H
// values (the upper half when `upper`) and adds the partner's copy of that half.
template <int H>
__device__ __forceinline__ void halve(const float *v, float *o, int mask, bool upper) {
#pragma unroll
    for (int i = 0; i < H; ++i) {
        const float send = upper ? v[i] : v[i + H];
        const float keep = upper ? v[i + H] : v[i];
        o[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
    }
}

using ptx::f2;
using ptx::fma2;
using ptx::mul2;

template <bool kFast> __device__ __forceinline__ f2 decay2(f2 dl2, f2 a2) {
    const f2 e = mul2(dl2, a2);
    if (kFast) return f2{ex2_approx(e.x), ex2_approx(e.y)};
    return f2{expf(e.x), expf(e.y)};
}

// NH pairs of consecutive floats from shared memory (8- or 16-byte aligned).
template <int NH> __device__ __forceinline__ void ld_pairs(const float *p, f2 (&o)[NH]) {
    if constexpr (NH == 1) {
        const float2 v = *reinterpret_cast<const float2 *>(p);
        o[0] = f2{v.x, v.y};
    } else {
#pragma unroll
        for (int i = 0; i < NH / 2; ++i) {
            const float4 v = reinterpret_cast<const float4 *>(p)[i];
            o[2 * i] = f2{v.x, v.y};
            o[2 * i + 1] = f2{v.z, v.w};
        }
    }
}
template <int NH> __device__ __forceinline__ void st_pairs(float *p, const f2 (&o)[NH]) {
    if constexpr (NH == 1) {
        *reinterpret_cast<float2 *>(p) = make_float2(o[0].x, o[0].y);
    } else {
#pragma unroll
        for (int i = 0; i < NH / 2; ++i)
            reinterpret_cast<float4 *>(p)[i] = make_float4(o[2 * i].x, o[2 * i].y,
                                                           o[2 * i + 1].x, o[2 * i + 1].y);
    }
}

template <typename TIO> __device__ __forceinline__ float ld_io(const void *p, int64_t i) {
    return Io<TIO>::load(static_cast<const TIO *>(p) + i);
}

template <typename TIO, int NS, bool kZoh>
__device__ __forceinline__ void scan_bwd_body(const ScanBwdParams &p) {
    using S = BwdShape<NS>;
    constexpr int NP = S::NP, T = S::T;
    constexpr bool kFast = std::is_same<TIO, __nv_bfloat16>::value;
    extern __shared__ __align__(16) float sm[];
    float *hs = sm;                       // [T][kCB][NP] states h_t of the tile
    float *sB = hs + T * kCB * NP;        // [T][NP]
    float *sC = sB + T * NP;              // [T][NP]
    float *sx = sC + T * NP;              // [T][kCB] x
    float *sdl = sx + T * kCB;            // step size dl
    float *sv = sdl + T * kCB;            // delta + bias (before softplus)
    float *sz = sv + T * kCB;             // z
    float *sgy = sz + T * kCB;            // dy
    float *sg = sgy + T * kCB;            // dy silu(z)
    float *syr = sg + T * kCB;            // C.h + D x
    float *sgx = syr + T * kCB;           // dx
    float *sgdl = sgx + T * kCB;          // d loss / d dl
    float *sred = sgdl + T * kCB;         // [T][4][2][NP] per-warp dB, dC

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c8 = lane >> 2, k = lane & 3;
    DeviceStatus *status = static_cast<DeviceStatus *>(p.status);
    (void)status;
    const int c = warp * 8 + c8;                       // channel within the block
    const int64_t Dm = p.dim, L = p.seqlen, N = p.dstate;
    const int64_t b = blockIdx.y;
    const int64_t dbase = static_cast<int64_t>(blockIdx.x) * kCB;
    const int64_t d = dbase + c;
    const bool dvalid = d < Dm;
    const int64_t nt = (L + T - 1) / T;

    constexpr int NH = NS / 2;           // state pairs of a lane
    f2 A2[NH], An[NH], ia[NH];
    bool nval[NS];
#pragma unroll
    for (int q = 0; q < NH; ++q) {
        float av[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int j = 2 * q + e;
            const int64_t n = k * NS + j;
            nval[j] = dvalid && n < N;
            av[e] = nval[j] ? p.A[d * N + n] : 0.f;
        }
        An[q] = f2{av[0], av[1]};
        A2[q] = f2{scale_A<kFast>(av[0]), scale_A<kFast>(av[1])};
        ia[q] = f2{av[0] != 0.f ? 1.f / av[0] : 0.f, av[1] != 0.f ? 1.f / av[1] : 0.f};
    }
    const float Dd = (dvalid && p.D) ? p.D[d] : 0.f;

    // ---- staging of a tile's rows and of B, C, software-pipelined: the raw values of
    // the next tile are loaded into registers before the current tile is computed and
    // written to shared memory after it.
    // row element e = tid + 128 r: t = e / 32, channel cc = e % 32 = tid % 32
    const int cc = tid & 31;
    const int64_t dcc = dbase + cc;
    const bool ccvalid = dcc < Dm;
    const float bias_cc = (ccvalid && p.bias) ? p.bias[dcc] : 0.f;
    constexpr int kRowsPer = T / (kThreads / kCB);                 // rows per thread
    constexpr int kBCPer = (T * NP + kThreads - 1) / kThreads;     // B/C elements per thread
    const TIO zero_io = Io<TIO>::from_f(0.f);
    struct Pre {
        TIO x[kRowsPer], dt[kRowsPer], z[kRowsPer], gy[kRowsPer], B[kBCPer], C[kBCPer];
    } pre;
    auto prefetch = [&](int64_t t0, int Ts, bool full) {
        const TIO *gx = static_cast<const TIO *>(p.x), *gd = static_cast<const TIO *>(p.delta);
        const TIO *gz = static_cast<const TIO *>(p.z), *ggy = static_cast<const TIO *>(p.dy);
        const TIO *gB = static_cast<const TIO *>(p.B), *gC = static_cast<const TIO *>(p.C);
#pragma unroll
        for (int r = 0; r < kRowsPer; ++r) {
            const int t = (tid >> 5) + r * (kThreads / kCB);
            const bool in = t < Ts && ccvalid;
            const int64_t i = (b * L + t0 + t) * Dm + dcc;
            pre.x[r] = in ? __ldg(gx + i) : zero_io;
            pre.dt[r] = in ? __ldg(gd + i) : zero_io;
            if (full) {
                pre.z[r] = (in && gz) ? __ldg(gz + i) : zero_io;
                pre.gy[r] = in ? __ldg(ggy + i) : zero_io;
            }
        }
#pragma unroll
        for (int q = 0; q < kBCPer; ++q) {
            const int e = tid + q * kThreads;
            const int t = e / NP, n = e % NP;
            const bool in = e < T * NP && t < Ts && n < N;
            const int64_t i = (b * L + t0 + t) * N + n;
            pre.B[q] = in ? __ldg(gB + i) : zero_io;
            if (full) pre.C[q] = in ? __ldg(gC + i) : zero_io;
        }
    };
    auto commit = [&](bool full) {
#pragma unroll
        for (int r = 0; r < kRowsPer; ++r) {
            const int t = (tid >> 5) + r * (kThreads / kCB);
            const float xv = Io<TIO>::to_f(pre.x[r]);
            const float v = Io<TIO>::to_f(pre.dt[r]) + bias_cc;
            sx[t * kCB + cc] = xv;
            sdl[t * kCB + cc] = ccvalid ? (p.softplus ? softplus<kFast>(v) : v) : 0.f;
            if (full) {
                const float zv = Io<TIO>::to_f(pre.z[r]);
                const float gy = Io<TIO>::to_f(pre.gy[r]);
                sv[t * kCB + cc] = v;
                sz[t * kCB + cc] = zv;
                sgy[t * kCB + cc] = gy;
                sg[t * kCB + cc] = p.z ? gy * silu<kFast>(zv) : gy;
            }
        }
#pragma unroll
        for (int q = 0; q < kBCPer; ++q) {
            const int e = tid + q * kThreads;
            if (e < T * NP) {
                sB[e] = Io<TIO>::to_f(pre.B[q]);
                if (full) sC[e] = Io<TIO>::to_f(pre.C[q]);
            }
        }
    };

    // ---- 1. checkpoint pass
    // input term of the update for a pair: coefficient (dl or the ZOH one) x B x
    auto input2 = [&](int q, f2 a, f2 Bp, float dl, float xv) -> f2 {
        if (kZoh) {
            const f2 cf{zoh_coef<kFast>(dl, dl * An[q].x, a.x, ia[q].x),
                        zoh_coef<kFast>(dl, dl * An[q].y, a.y, ia[q].y)};
            return mul2(mul2(cf, Bp), f2{xv, xv});
        }
        const float u = dl * xv;
        return mul2(Bp, f2{u, u});
    };
    f2 h[NH];
#pragma unroll
    for (int q = 0; q < NH; ++q) {
        const float *h0 = p.h0 + (b * Dm + d) * N + k * NS + 2 * q;
        h[q] = f2{(nval[2 * q] && p.h0) ? h0[0] : 0.f, (nval[2 * q + 1] && p.h0) ? h0[1] : 0.f};
    }
    // (skipped when the forward pass wrote the checkpoints)
    if (nt > 1 && !p.ckpt_given) prefetch(0, T, false);
    for (int64_t s = 0; s < nt && !p.ckpt_given; ++s) {
        float *ck = p.ckpt + ((b * nt + s) * Dm + d) * N + k * NS;
        if (in_bounds(b < p.batch && s < nt, status, 151)) {
#pragma unroll
            for (int q = 0; q < NH; ++q) {
                if (nval[2 * q]) ck[2 * q] = h[q].x;
                if (nval[2 * q + 1]) ck[2 * q + 1] = h[q].y;
            }
        }
        if (s == nt - 1) break;                 // the last tile starts from this state
        __syncthreads();
        commit(false);
        if (s + 2 < nt) prefetch((s + 1) * T, T, false);
        __syncthreads();
#pragma unroll 8
        for (int t = 0; t < T; ++t) {
            const float dl = sdl[t * kCB + c], xv = sx[t * kCB + c];
            f2 Bp[NH];
            ld_pairs<NH>(sB + t * NP + k * NS, Bp);
#pragma unroll
            for (int q = 0; q < NH; ++q) {
                const f2 a = decay2<kFast>(f2{dl, dl}, A2[q]);
                h[q] = fma2(a, h[q], input2(q, a, Bp[q], dl, xv));
            }
        }
    }
    // the checkpoint stores of this block are read back by the same threads below; the
    // forward pass's are visible to this launch

    // ---- 2. reverse pass
    f2 lam[NH], gA[NH];
#pragma unroll
    for (int q = 0; q < NH; ++q) {
        const float *hf = p.dh_final + (b * Dm + d) * N + k * NS + 2 * q;
        lam[q] = f2{(nval[2 * q] && p.dh_final) ? hf[0] : 0.f,
                    (nval[2 * q + 1] && p.dh_final) ? hf[1] : 0.f};
        gA[q] = f2{0.f, 0.f};
    }
    float gD_acc = 0.f, gbias_acc = 0.f;     // channel cc, rows of this thread
    auto tile_len = [&](int64_t s) { return static_cast<int>(L - s * T < T ? L - s * T : T); };
    f2 hst[NH], hst_next[NH];
    auto load_ckpt = [&](int64_t s) {
        const float *ck = p.ckpt + ((b * nt + s) * Dm + d) * N + k * NS;
#pragma unroll
        for (int q = 0; q < NH; ++q)
            hst_next[q] = f2{nval[2 * q] ? __ldcg(ck + 2 * q) : 0.f,
                             nval[2 * q + 1] ? __ldcg(ck + 2 * q + 1) : 0.f};
    };
    prefetch((nt - 1) * T, tile_len(nt - 1), true);
    load_ckpt(nt - 1);
    for (int64_t s = nt - 1; s >= 0; --s) {
        const int64_t t0 = s * T;
        const int Ts = tile_len(s);
        __syncthreads();
        commit(true);
#pragma unroll
        for (int q = 0; q < NH; ++q) hst[q] = hst_next[q];
        if (s > 0) {
            prefetch((s - 1) * T, T, true);
            load_ckpt(s - 1);
        }
        __syncthreads();
        // the tile's recompute and walk, with a compile-time step count for whole tiles
        // (1106 -> 1073 us, from forward checkpoints 973 -> 940 us, at the 130M-layer shape)
        auto tile_work = [&](auto ts) {
        // recompute h_t of the tile (and C.h + D x for the gate's gradient)
#pragma unroll
        for (int q = 0; q < NH; ++q) h[q] = hst[q];
#pragma unroll 8
        for (int t = 0; t < ts; ++t) {
            const float dl = sdl[t * kCB + c], xv = sx[t * kCB + c];
            f2 Bp[NH], Cp[NH];
            ld_pairs<NH>(sB + t * NP + k * NS, Bp);
            ld_pairs<NH>(sC + t * NP + k * NS, Cp);
            f2 part2{0.f, 0.f};
#pragma unroll
            for (int q = 0; q < NH; ++q) {
                const f2 a = decay2<kFast>(f2{dl, dl}, A2[q]);
                h[q] = fma2(a, h[q], input2(q, a, Bp[q], dl, xv));
                part2 = fma2(Cp[q], h[q], part2);
            }
            st_pairs<NH>(hs + (t * kCB + c) * NP + k * NS, h);
            float part = part2.x + part2.y;
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            part += __shfl_xor_sync(0xffffffffu, part, 2);
            if (k == 0) syr[t * kCB + c] = fmaf(Dd, xv, part);
        }
        // walk the tile backwards; h holds h_t, hp is h_{t-1}
#pragma unroll 8
        for (int t = ts - 1; t >= 0; --t) {
            f2 hp[NH];
            if (t > 0) {
                ld_pairs<NH>(hs + ((t - 1) * kCB + c) * NP + k * NS, hp);
            } else {
#pragma unroll
                for (int q = 0; q < NH; ++q) hp[q] = hst[q];
            }
            const float g = sg[t * kCB + c], xv = sx[t * kCB + c], dl = sdl[t * kCB + c];
            const f2 g2{g, g}, dl2{dl, dl};
            f2 Bp[NH], Cp[NH];
            ld_pairs<NH>(sB + t * NP + k * NS, Bp);
            ld_pairs<NH>(sC + t * NP + k * NS, Cp);
            float pv[2 * NS];          // [0, NS): dB parts, [NS, 2NS): dC parts
            f2 sLB2{0.f, 0.f}, gx2{0.f, 0.f}, gdl2{0.f, 0.f};
#pragma unroll
            for (int q = 0; q < NH; ++q) {
                const f2 pc = mul2(g2, h[q]);
                pv[NS + 2 * q] = pc.x;
                pv[NS + 2 * q + 1] = pc.y;
                lam[q] = fma2(g2, Cp[q], lam[q]);
                const f2 a = decay2<kFast>(dl2, A2[q]);
                const f2 qq = mul2(mul2(lam[q], hp[q]), a);
                gdl2 = fma2(qq, An[q], gdl2);
                f2 pb;
                if (kZoh) {
                    const f2 v{dl * An[q].x, dl * An[q].y};
                    const f2 cf{zoh_coef<kFast>(dl, v.x, a.x, ia[q].x),
                                zoh_coef<kFast>(dl, v.y, a.y, ia[q].y)};
                    const f2 lc = mul2(lam[q], cf);
                    pb = mul2(lc, f2{xv, xv});
                    gx2 = fma2(lc, Bp[q], gx2);
                    const f2 lbx = mul2(mul2(lam[q], Bp[q]), f2{xv, xv});
                    gdl2 = fma2(lbx, a, gdl2);
                    const f2 dcda{zoh_dc_dA<kFast>(dl, v.x, a.x, ia[q].x),
                                  zoh_dc_dA<kFast>(dl, v.y, a.y, ia[q].y)};
                    gA[q] = fma2(qq, dl2, fma2(lbx, dcda, gA[q]));
                } else {
                    const float u = dl * xv;
                    pb = mul2(lam[q], f2{u, u});
                    sLB2 = fma2(lam[q], Bp[q], sLB2);
                    gA[q] = fma2(qq, dl2, gA[q]);
                }
                pv[2 * q] = pb.x;
                pv[2 * q + 1] = pb.y;
                lam[q] = mul2(lam[q], a);
                h[q] = hp[q];
            }
            float gxp, gdlp = gdl2.x + gdl2.y;
            if (kZoh) {
                gxp = gx2.x + gx2.y;
            } else {
                const float sLB = sLB2.x + sLB2.y;
                gxp = dl * sLB;
                gdlp = fmaf(xv, sLB, gdlp);
            }
            gxp += __shfl_xor_sync(0xffffffffu, gxp, 1);
            gxp += __shfl_xor_sync(0xffffffffu, gxp, 2);
            gdlp += __shfl_xor_sync(0xffffffffu, gdlp, 1);
            gdlp += __shfl_xor_sync(0xffffffffu, gdlp, 2);
            if (k == 0) {
                sgx[t * kCB + c] = fmaf(g, Dd, gxp);
                sgdl[t * kCB + c] = gdlp;
            }
            // dB, dC: sum over the warp's 8 channels (lane bits 2..4)
            float *red = sred + ((t * 4 + warp) * 2) * NP;
            constexpr int M = 2 * NS;
            if constexpr (M >= 8) {
                float r1[M / 2], r2[M / 4], r3[M / 8];
                halve<M / 2>(pv, r1, 16, lane & 16);
                halve<M / 4>(r1, r2, 8, lane & 8);
                halve<M / 8>(r2, r3, 4, lane & 4);
#pragma unroll
                for (int i = 0; i < M / 8; ++i) {
                    const int m = c8 * (M / 8) + i;
                    red[(m / NS) * NP + k * NS + m % NS] = r3[i];
                }
            } else if constexpr (M == 4) {
                float r1[2], r2[1];
                halve<2>(pv, r1, 16, lane & 16);
                halve<1>(r1, r2, 8, lane & 8);
                r2[0] += __shfl_xor_sync(0xffffffffu, r2[0], 4);
                if (!(lane & 4)) {
                    const int m = (c8 >> 1);             // 2 b4 + b3
                    red[(m / NS) * NP + k * NS + m % NS] = r2[0];
                }
            }
        }
        };
        // (more states per lane, or the zero-order-hold terms, would spill: runtime count)
        if constexpr (NS <= 4 && !kZoh) {
            if (Ts == T) tile_work(std::integral_constant<int, T>{});
            else tile_work(Ts);
        } else {
            tile_work(Ts);
        }
        __syncthreads();
        // rows of the tile: dx, ddelta, dz; dD and dbias partial sums
        for (int t = tid >> 5; t < Ts; t += kThreads / kCB) {
            if (!ccvalid) continue;
            const int e = t * kCB + cc;
            const int64_t i = (b * L + t0 + t) * Dm + dcc;
            if (!in_bounds(t0 + t < L && b < p.batch, status, 152)) continue;
            const float gdl = sgdl[e];
            const float gdelta = p.softplus ? gdl * sigmoid_f(sv[e], kFast) : gdl;
            static_cast<TIO *>(p.dx)[i] = Io<TIO>::from_f(sgx[e]);
            static_cast<TIO *>(p.ddelta)[i] = Io<TIO>::from_f(gdelta);
            if (p.z) {
                const float zv = sz[e], sgm = sigmoid_f(zv, kFast);
                const float dsilu = sgm * fmaf(zv, 1.f - sgm, 1.f);
                static_cast<TIO *>(p.dz)[i] = Io<TIO>::from_f(sgy[e] * syr[e] * dsilu);
            }
            gD_acc = fmaf(sg[e], sx[e], gD_acc);
            gbias_acc += gdelta;
        }
        // dB, dC of the tile: sum the four warps, one atomic per (t, n)
        for (int e = tid; e < Ts * 2 * NP; e += kThreads) {
            const int t = e / (2 * NP), r = e % (2 * NP), kind = r / NP, n = r % NP;
            if (n >= N) continue;
            const float *src = sred + (t * 4 * 2 + kind) * NP + n;
            const float sum = src[0] + src[2 * NP] + src[4 * NP] + src[6 * NP];
            float *dst = kind ? p.dC : p.dB;
            if (in_bounds(t0 + t < L && b < p.batch, status, 153))
                atomicAdd(dst + (b * L + t0 + t) * N + n, sum);
        }
    }
    // ---- per-channel and per-state sums
#pragma unroll
    for (int q = 0; q < NH; ++q) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int j = 2 * q + e;
            if (!nval[j] || !in_bounds(d < Dm && b < p.batch, status, 154)) continue;
            atomicAdd(p.dA + d * N + k * NS + j, e ? gA[q].y : gA[q].x);
            if (p.dh0) p.dh0[(b * Dm + d) * N + k * NS + j] = e ? lam[q].y : lam[q].x;
        }
    }
    __syncthreads();
    float *sacc = sm;                  // [4][kCB][2]
    sacc[((tid >> 5) * kCB + cc) * 2] = gD_acc;
    sacc[((tid >> 5) * kCB + cc) * 2 + 1] = gbias_acc;
    __syncthreads();
    if (tid < kCB && ccvalid) {
        float s0 = 0.f, s1 = 0.f;
        for (int w = 0; w < 4; ++w) {
            s0 += sacc[(w * kCB + tid) * 2];
            s1 += sacc[(w * kCB + tid) * 2 + 1];
        }
        if (p.dD) atomicAdd(p.dD + dcc, s0);
        if (p.ddelta_bias) atomicAdd(p.ddelta_bias + dcc, s1);
    }
}

template <typename TIO, int NS, bool kZoh>
__global__ void __launch_bounds__(kThreads) scan_bwd_kernel(const ScanBwdParams p) {
    scan_bwd_body<TIO, NS, kZoh>(p);
}

// Up to four states per lane the kernel runs under a register budget instead of launch
// bounds: 168 registers is the most that keeps three 128-thread blocks per SM, and the
// compiler then schedules the unrolled loops without spills (96 registers under launch
// bounds at the 130M-layer shape; 1072 -> 1018 us, 938 -> 880 us from forward
// checkpoints, on B300).  More states per lane spill under the budget.
template <typename TIO, int NS, bool kZoh>
__global__ void __maxnreg__(168) scan_bwd_kernel_r168(const ScanBwdParams p) {
    scan_bwd_body<TIO, NS, kZoh>(p);
}

template <typename TIO, int NS, bool kZoh>
cudaError_t launch_ns(const ScanBwdParams &p, cudaStream_t stream) {
    using S = BwdShape<NS>;
    void (*kern)(const ScanBwdParams);
    if constexpr (NS <= 4)
        kern = scan_bwd_kernel_r168<TIO, NS, kZoh>;
    else
        kern = scan_bwd_kernel<TIO, NS, kZoh>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(S::bytes));
    if (e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>((p.dim + kCB - 1) / kCB), static_cast<unsigned>(p.batch));
    kern<<<grid, kThreads, S::bytes, stream>>>(p);
    return cudaGetLastError();
}

template <typename TIO, bool kZoh>
cudaError_t launch_typed(const ScanBwdParams &p, cudaStream_t stream) {
    if (p.dstate <= 8) return launch_ns<TIO, 2, kZoh>(p, stream);
    if (p.dstate <= 16) return launch_ns<TIO, 4, kZoh>(p, stream);
    if (p.dstate <= 32) return launch_ns<TIO, 8, kZoh>(p, stream);
    return launch_ns<TIO, 16, kZoh>(p, stream);
}

}  // namespace

int scan_ckpt_steps(int64_t dstate) {
    if (dstate <= 8) return BwdShape<2>::T;
    if (dstate <= 16) return BwdShape<4>::T;
    if (dstate <= 32) return BwdShape<8>::T;
    return BwdShape<16>::T;
}

size_t scan_bwd_ckpt_floats(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate) {
    const int64_t T = scan_ckpt_steps(dstate);
    const int64_t nt = (seqlen + T - 1) / T;
    return static_cast<size_t>(batch * nt * dim * dstate);
}

cudaError_t launch_scan_bwd(const ScanBwdParams &p, cudaStream_t stream) {
    if (p.io_bf16)
        return p.zoh ? launch_typed<__nv_bfloat16, true>(p, stream)
                     : launch_typed<__nv_bfloat16, false>(p, stream);
    return p.zoh ? launch_typed<float, true>(p, stream) : launch_typed<float, false>(p, stream);
}

}  // namespace ssm
