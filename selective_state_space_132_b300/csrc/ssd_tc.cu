// Multi-head selective SSM with a scalar decay per head (Mamba-2), computed in its
// chunked dual form on the tcgen05 tensor cores.
//
// What it computes ("Mamba-2: 상태 공간 기반 시퀀스 모델", sections "1-세미분리 행렬",
// "SSM-Attention 동치성", "멀티-헤드 구조" and "SSD 타일링 알고리즘"), per batch b and
// head h (group g = h / (H / G)), with dl_t = softplus(delta_t,h + bias_h):
//   S_t = exp(dl_t A_h) S_{t-1} + dl_t x_t B_t^T            (P x N state)
//   y_t = S_t C_t + D_h x_t            (optionally times silu(z_t))
// Inside a chunk of Q = 128 steps starting from state S_in, with the running
// log-decay Lam_t = sum_{r <= t} dl_r A_h (inclusive, from the chunk start):
//   G      = C B^T                                         (Q x Q, shared by heads)
//   M[t,s] = G[t,s] exp(Lam_t - Lam_s) dl_s   for s <= t, else 0
//   Y      = M X + diag(exp(Lam_t)) C S_in^T + D X         (the 1-semiseparable
//                                                           matrix applied blockwise)
//   S_out  = exp(Lam_end) S_in + (B^T Xw)^T,  Xw[s,:] = exp(Lam_end - Lam_s) dl_s x_s
// which is the pages' intra-chunk (L o C B^T) X plus inter-chunk state passing
// with the decay weights written out.  Chunk length: the pages' tiling uses 256
// steps (tuned for A100); on B300 the M = 128 tcgen05 tile and the 512-column TMEM
// make 128 the natural chunk.  A longer requested chunk is evaluated as 128-step
// tiles whose below-diagonal block goes through the state at the tile boundary,
// which is the same sum factored through rank N.
//
// B300 mapping (persistent blocks of 256 threads: two warps per TMEM lane quadrant,
// each thread one lane (row) and half of the columns):
//   * TMA (128-byte swizzle) brings C, B (Q x N), X (Q x P) and z of a chunk into
//     shared memory in the canonical UMMA layouts.
//   * Four bf16 MMAs per chunk with fp32 accumulators in TMEM:
//       G  = C B^T        (M=128, N=128, K=N)   A=C  K-major, B=B  K-major
//       Yo = C S_in^T     (M=128, N=P,   K=N)   A=C  K-major, B=S  MN-major
//       Sc = B^T Xw       (M=N=128, N=P, K=Q)   A=B  MN-major, B=Xw MN-major
//       Yd = M X          (M=128, N=P,   K=Q)   A=M  in TMEM,  B=X  MN-major
//   * CUDA cores build Xw (bf16, swizzled shared memory) and M (bf16 pairs written
//     to TMEM with tcgen05.st; pairwise exponentials on the diagonal 32 x 32 blocks,
//     a product of two factors <= 1 below them), update the fp32 state held in
//     registers (threads n and n + 128 own the two halves of row n of S^T) and finish
//     y = Yd + exp(Lam_t) Yo + D x,
//     which goes back to HBM through a TMA store.
// Two blocks share an SM: TMEM is cut to 256 columns by writing M (bf16 pairs) over
// the G accumulator and reading it as the A operand of the M X product straight from
// tensor memory, and shared memory stays under half of the SM by letting the bf16
// state tile and Xw take turns in one buffer.
// Shape rules of this kernel: bf16 I/O, P = 64, N = 128; other shapes run the
// sequential kernel (ssd_chunk.cu).
#include <cudaTypedefs.h>

#include <algorithm>

#include "../../include/ssm.h"
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tma_host.cuh"

namespace ssm {
namespace {

using ptx::f2;

constexpr int kQ = 128;   // chunk length (MMA M)
constexpr int kP = 64;    // head dim
constexpr int kN = 128;   // state size
constexpr int kThreads = 256;   // two warps per TMEM lane quadrant
constexpr int kPH = kP / 2;     // columns of P (or of a state row) one thread handles
constexpr int kTmemCols = 256;  // two blocks per SM share the 512 columns
// TMEM columns: G (fp32, 128) whose first 64 columns are then overwritten by M
// (bf16 pairs) and whose last 64 by the chunk state Sc; Yd and Yo (fp32, 64 each).
constexpr uint32_t kColG = 0, kColM = 0, kColSc = 64, kColYd = 128, kColYo = 192;

// Shared-memory layout (bytes); every operand tile starts on a 1024-byte boundary.
constexpr int kTile = kQ * 128;                 // 128 rows x 128 bytes = 16 KB
constexpr int o_C = 0;                          // 2 k-blocks of 64 states
constexpr int o_B = o_C + 2 * kTile;
constexpr int o_X = o_B + 2 * kTile;            // also the y staging tile
constexpr int o_W = o_X + kTile;                // S_in^T (bf16) and, once Yo is done, Xw
constexpr int o_Z = o_W + kTile;                // gate input (only with a gate)
template <bool kGate> struct Smem {
    static constexpr int o_dl = o_Z + (kGate ? kTile : 0);  // float[128]
    static constexpr int o_lam = o_dl + kQ * 4;             // float[128]
    static constexpr int o_v = o_lam + kQ * 4;              // float[128] column factors
    static constexpr int o_red = o_v + kQ * 4;              // float[4] warp totals
    static constexpr int o_bar = o_red + 16;                // 2 mbarriers
    static constexpr int o_tmem = o_bar + 16;
    static constexpr int bytes = o_tmem + 16;
};

struct Maps {
    CUtensorMap C, B, X, Z, Y;
};

// 16-byte chunk `chunk` of row `row` in a tile of 128-byte rows stored with the
// 128-byte swizzle (chunk index XOR row % 8), the layout TMA writes and UMMA reads.
__device__ __forceinline__ uint4 ld_chunk(const unsigned char *tile, uint32_t row, uint32_t chunk) {
    return *reinterpret_cast<const uint4 *>(tile + row * 128u + ((chunk ^ (row & 7u)) << 4));
}
__device__ __forceinline__ void st_chunk(unsigned char *tile, uint32_t row, uint32_t chunk, uint4 v) {
    *reinterpret_cast<uint4 *>(tile + row * 128u + ((chunk ^ (row & 7u)) << 4)) = v;
}
__device__ __forceinline__ uint4 pack8(const float *v) {
    return make_uint4(ptx::f2_to_bf2(v[0], v[1]), ptx::f2_to_bf2(v[2], v[3]),
                      ptx::f2_to_bf2(v[4], v[5]), ptx::f2_to_bf2(v[6], v[7]));
}

// Work split over a persistent grid (stream-K): the B * H chains of nch chunks each
// form units = B * H * nch chunk steps; block k takes steps [u0, u1).  A chain cut
// between blocks k and k + 1 hands its state over through the workspace: block k
// runs that chain's head first and publishes the state (flag[k] = 1, release);
// block k + 1 runs its other work first and that chain's tail last, after
// acquiring the flag.  With at least one chain per block a chain is cut at most
// once and, since head + tail = nch <= the steps of a block, no block waits in
// steady state.  A block takes its range index k from an atomic ticket, i.e. in the
// order blocks actually start, so the block it may wait for (k - 1) has always started
// already and the wait cannot depend on a block that is not yet resident.
struct Split {
    int nctas;
    int nch;           // chunks per chain
    int64_t units;
    uint32_t *ticket;  // block-order counter, zeroed before the launch
    uint32_t *flags;   // nctas flags, zeroed before the launch
    float *states;     // nctas states of P x N fp32
};

template <bool kGate>
__global__ void __launch_bounds__(kThreads, 2) ssd_tc_kernel(const __grid_constant__ Maps maps,
                                                             SSDParams p, Split sk) {
    using SM = Smem<kGate>;
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char *sC = smem + o_C, *sB = smem + o_B, *sX = smem + o_X, *sW = smem + o_W;
    unsigned char *sZ = smem + o_Z;
    float *s_dl = reinterpret_cast<float *>(smem + SM::o_dl);
    float *s_lam = reinterpret_cast<float *>(smem + SM::o_lam);
    float *s_v = reinterpret_cast<float *>(smem + SM::o_v);
    float *s_red = reinterpret_cast<float *>(smem + SM::o_red);
    uint64_t *bar_load = reinterpret_cast<uint64_t *>(smem + SM::o_bar);
    uint64_t *bar_mma = bar_load + 1;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + SM::o_tmem);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    // row = TMEM lane (chunk step t, or state n) of this thread; hh = which half of the
    // P columns it handles; q4 = its lane quadrant (warps q4 and q4 + 4 share it)
    const int row = tid & 127, hh = tid >> 7, q4 = warp & 3;
    const int64_t H = p.nheads, L = p.seqlen;
    const __nv_bfloat16 *gdt = static_cast<const __nv_bfloat16 *>(p.delta);
    DeviceStatus *status = static_cast<DeviceStatus *>(p.status);

    // The swizzled operand tiles need a 1024-byte aligned base.
    if (ptx::smem_u32(smem) & 1023u) {
        if (tid == 0) report_status(status, SSM_ERR_UNSUPPORTED, 29);
        return;
    }

    if (tid == 0) {
        ptx::mbar_init(bar_load, 1);
        ptx::mbar_init(bar_mma, 1);
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(s_tmem, kTmemCols);
        ptx::tmem_relinquish();
    }
    if (tid == 0) reinterpret_cast<volatile uint32_t *>(s_red)[0] = atomicAdd(sk.ticket, 1u);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const int k = static_cast<int>(reinterpret_cast<volatile uint32_t *>(s_red)[0]);
    __syncthreads();  // s_red is reused for the warp totals

    const uint32_t id_G = ptx::idesc_bf16(128, 128, 0, 0);
    const uint32_t id_Yo = ptx::idesc_bf16(128, kP, 0, 1);
    const uint32_t id_Sc = ptx::idesc_bf16(128, kP, 1, 1);
    const uint32_t id_Yd = ptx::idesc_bf16(128, kP, 0, 1);
    const uint32_t aC = ptx::smem_u32(sC), aB = ptx::smem_u32(sB), aX = ptx::smem_u32(sX);
    const uint32_t aW = ptx::smem_u32(sW);
    constexpr uint32_t kLoadBytes = 4 * kTile + (kGate ? 2 : 1) * kTile;

    uint32_t ph_load = 0, ph_mma = 0;
    bool ok = true;
    int pending = 0;  // 1: a TMA load, 2: an MMA commit, 3: a state hand-over that timed out
    // Every thread waits; the block agrees on the outcome so that it never splits.
    auto wait_all = [&](uint64_t *bar, uint32_t ph) -> bool {
        const int mine = ptx::mbar_wait(bar, ph) ? 1 : 0;
        return __syncthreads_and(mine) != 0;
    };

    // ---- this block's steps: head of the last chain, whole chains, tail of the first
    const int nch = sk.nch;
    const int64_t u0 = static_cast<int64_t>(k) * sk.units / sk.nctas;
    const int64_t u1 = static_cast<int64_t>(k + 1) * sk.units / sk.nctas;
    const int64_t first = u0 / nch, last = (u1 - 1) / nch;
    const int first_off = static_cast<int>(u0 - first * nch);
    const int last_end = static_cast<int>(u1 - last * nch);
    const bool has_tail = u1 > u0 && first_off > 0;
    const bool has_head = u1 > u0 && last_end < nch && !(has_tail && first == last);
    const int64_t full_lo = has_tail ? first + 1 : first;
    const int64_t full_hi = has_head ? last : last + 1;  // exclusive
    const int64_t nfull = full_hi > full_lo ? full_hi - full_lo : 0;
    const int nseg = (u1 > u0) ? (has_head ? 1 : 0) + static_cast<int>(nfull) + (has_tail ? 1 : 0)
                               : 0;

    float S[kPH];
    for (int seg = 0; seg < nseg && ok; ++seg) {
        // kind: 1 head (publishes), 0 whole chain, 2 tail (acquires)
        int kind;
        int64_t chain;
        int c_lo, c_hi;
        if (has_head && seg == 0) {
            kind = 1; chain = last; c_lo = 0; c_hi = last_end;
        } else if (has_tail && seg == nseg - 1) {
            kind = 2; chain = first; c_lo = first_off; c_hi = nch;
        } else {
            kind = 0; chain = full_lo + (seg - (has_head ? 1 : 0)); c_lo = 0; c_hi = nch;
        }
        const int b = static_cast<int>(chain / H), h = static_cast<int>(chain % H);
        const int g = static_cast<int>(h / (H / p.ngroups));
        const float a_l2 = p.A[h] * kLog2e;  // decay exponent per unit step, base 2
        const float bias = p.bias ? p.bias[h] : 0.f;
        const float Dh = p.Dv ? p.Dv[h] : 0.f;

        // ---- initial state: h0 (or zero), or the state the previous block handed over
        const float *src;
        if (kind == 2) {
            int got = 1;
            if (tid == 0)
                got = in_bounds(k >= 1 && k - 1 < sk.nctas, status, 123) &&
                              ptx::wait_flag(sk.flags + (k - 1), ptx::kWaitCycles)
                          ? 1 : 0;
            if (__syncthreads_or(tid == 0 && !got)) {
                ok = false;
                pending = 3;
                break;
            }
            src = sk.states + static_cast<int64_t>(k - 1) * kP * kN;
        } else {
            src = p.h0 ? p.h0 + (static_cast<int64_t>(b) * H + h) * kP * kN : nullptr;
        }
#pragma unroll
        for (int pp = 0; pp < kPH; ++pp) S[pp] = src ? __ldcg(src + (kPH * hh + pp) * kN + row) : 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) st_chunk(sW, row, 4 * hh + q, pack8(S + 8 * q));
        ptx::fence_proxy_async_smem();  // the first Yo MMA reads sW

        float raw_next = 0.f;
        {
            const int64_t t = static_cast<int64_t>(c_lo) * kQ + row;
            if (t < L) raw_next = __bfloat162float(gdt[(static_cast<int64_t>(b) * L + t) * H + h]);
        }

        for (int c = c_lo; c < c_hi; ++c) {
            const int t0 = c * kQ;
            // ---- (a) loads of this chunk (the previous chunk released every tile) and an
            //      L2 prefetch of the next one
            if (tid == 0) {
                ptx::bulk_wait_read<0>();  // y store of the previous chunk has left sX
                (void)in_bounds(g < p.ngroups && h < H && t0 < L && b < p.batch, status, 121);
                ptx::mbar_arrive_expect_tx(bar_load, kLoadBytes);
                for (int kb = 0; kb < 2; ++kb) {
                    ptx::tma_load_3d(sC + kb * kTile, &maps.C, bar_load, g * kN + 64 * kb, t0, b);
                    ptx::tma_load_3d(sB + kb * kTile, &maps.B, bar_load, g * kN + 64 * kb, t0, b);
                }
                ptx::tma_load_3d(sX, &maps.X, bar_load, h * kP, t0, b);
                if (kGate) ptx::tma_load_3d(sZ, &maps.Z, bar_load, h * kP, t0, b);
                if (c + 1 < c_hi) {
                    for (int kb = 0; kb < 2; ++kb) {
                        ptx::tma_prefetch_3d(&maps.C, g * kN + 64 * kb, t0 + kQ, b);
                        ptx::tma_prefetch_3d(&maps.B, g * kN + 64 * kb, t0 + kQ, b);
                    }
                    ptx::tma_prefetch_3d(&maps.X, h * kP, t0 + kQ, b);
                    if (kGate) ptx::tma_prefetch_3d(&maps.Z, h * kP, t0 + kQ, b);
                }
            }
            // ---- (b) step sizes (the raw value was fetched one chunk ahead), the running
            //      log2-decay and the column factors of the mask
            const int64_t t = t0 + row;
            const float raw = raw_next;
            if (c + 1 < c_hi && t + kQ < L)
                raw_next = __bfloat162float(gdt[(static_cast<int64_t>(b) * L + t + kQ) * H + h]);
            const float dl = t < L ? step_size<true>(raw, bias, p.softplus) : 0.f;
            float lam = dl * a_l2;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float v = __shfl_up_sync(0xffffffffu, lam, off);
                if (lane >= off) lam += v;
            }
            // lam of the last step of this warp's 32-step block (before adding earlier warps)
            const float lam_blk = __shfl_sync(0xffffffffu, lam, 31);
            // (both halves compute the same values; the first half publishes them)
            if (lane == 31 && hh == 0) s_red[warp] = lam;
            __syncthreads();
            float base = 0.f;
            for (int w = 0; w < q4; ++w) base += s_red[w];
            lam += base;
            if (hh == 0) {
                // v_s = exp(Lam_e - Lam_s) dl_s with e the last step of the block holding s
                s_v[row] = ex2_approx((base + lam_blk) - lam) * dl;
                s_dl[row] = dl;
                s_lam[row] = lam;
            }

            if (!wait_all(bar_load, ph_load)) {
                ok = false;
                pending = 1;
                break;
            }
            ph_load ^= 1;
            const float lam_tot = s_red[0] + s_red[1] + s_red[2] + s_red[3];

            // ---- (c) G = C B^T and Yo = C S_in^T
            if (tid == 0) {
                ptx::tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kN / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kTile + (kk & 3) * 32;
                    const uint64_t da = ptx::sdesc_sw128(aC + off, 16, 1024);
                    const uint64_t db = ptx::sdesc_sw128(aB + off, 16, 1024);
                    ptx::mma_bf16(tmem + kColG, da, db, id_G, kk > 0);
                }
#pragma unroll
                for (int kk = 0; kk < kN / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kTile + (kk & 3) * 32;
                    const uint64_t da = ptx::sdesc_sw128(aC + off, 16, 1024);
                    const uint64_t db = ptx::sdesc_sw128(aW + kk * 2048, 1024, 1024);
                    ptx::mma_bf16(tmem + kColYo, da, db, id_Yo, kk > 0);
                }
                ptx::mma_commit(bar_mma);
            }
            if (!wait_all(bar_mma, ph_mma)) {
                ok = false;
                pending = 2;
                break;
            }
            ph_mma ^= 1;
            ptx::tc_fence_after();

            // ---- (d) Xw[s, :] = exp(Lam_end - Lam_s) dl_s x_s into sW (S_in is consumed)
            {
                const float w = ex2_approx(lam_tot - lam) * dl;
                const f2 w2{w, w};
#pragma unroll
                for (int q = 4 * hh; q < 4 * hh + 4; ++q) {
                    const uint4 v = ld_chunk(sX, row, q);
                    const uint32_t in[4] = {v.x, v.y, v.z, v.w};
                    uint32_t out[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const f2 e = ptx::mul2(ptx::bf2_to_f2(in[i]), w2);
                        out[i] = ptx::f2_to_bf2(e.x, e.y);
                    }
                    st_chunk(sW, row, q, make_uint4(out[0], out[1], out[2], out[3]));
                }
            }
            // ---- (e) M[t, s] = G[t, s] exp(Lam_t - Lam_s) dl_s, s <= t, as bf16 pairs over
            //      G's first 64 columns (row t).  Blocks of 32 columns: below the diagonal
            //      block exp(Lam_t - Lam_s) = u_t v_s / dl_s with u_t = exp(Lam_t - Lam_e),
            //      both factors <= 1; on it, pairwise exponentials.  This thread builds the
            //      column blocks hh and hh + 2; M overwrites G, so every warp first reads
            //      what it needs of G, then the block synchronises, then M is stored.
            {
                uint32_t packed[2][16];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int i = hh + 2 * r;
                    if (i < q4) {
                        float gv[32];
                        ptx::tmem_ld32(tmem + lane_base + kColG + 32 * i, gv);
                        const float u = ex2_approx(lam - s_lam[32 * i + 31]);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float2 vv = *reinterpret_cast<const float2 *>(s_v + 32 * i + 2 * e);
                            const f2 m = ptx::mul2(ptx::mul2(f2{gv[2 * e], gv[2 * e + 1]}, f2{u, u}),
                                                   f2{vv.x, vv.y});
                            packed[r][e] = ptx::f2_to_bf2(m.x, m.y);
                        }
                    } else if (i == q4) {
                        float gv[32];
                        ptx::tmem_ld32(tmem + lane_base + kColG + 32 * i, gv);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            float m2[2];
#pragma unroll
                            for (int u2 = 0; u2 < 2; ++u2) {
                                const int sc = 32 * i + 2 * e + u2;
                                const float val = gv[2 * e + u2] * ex2_approx(lam - s_lam[sc]) * s_dl[sc];
                                m2[u2] = sc <= row ? val : 0.f;
                            }
                            packed[r][e] = ptx::f2_to_bf2(m2[0], m2[1]);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) packed[r][e] = 0u;
                    }
                }
                ptx::tc_fence_before();
                __syncthreads();  // every read of G is done
                ptx::tc_fence_after();
#pragma unroll
                for (int r = 0; r < 2; ++r)
                    ptx::tmem_st16(tmem + lane_base + kColM + 16 * (hh + 2 * r), packed[r]);
            }
            ptx::tmem_wait_st();
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            __syncthreads();
            // ---- (f) Yd = M X (A from TMEM) and Sc = B^T Xw
            if (tid == 0) {
                ptx::tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kQ / 16; ++kk) {
                    const uint64_t db = ptx::sdesc_sw128(aX + kk * 2048, 1024, 1024);
                    ptx::mma_bf16_ts(tmem + kColYd, tmem + kColM + 8 * kk, db, id_Yd, kk > 0);
                }
#pragma unroll
                for (int kk = 0; kk < kQ / 16; ++kk) {
                    const uint64_t da = ptx::sdesc_sw128(aB + kk * 2048, kTile, 1024);
                    const uint64_t db = ptx::sdesc_sw128(aW + kk * 2048, 1024, 1024);
                    ptx::mma_bf16(tmem + kColSc, da, db, id_Sc, kk > 0);
                }
                ptx::mma_commit(bar_mma);
            }
            if (!wait_all(bar_mma, ph_mma)) {
                ok = false;
                pending = 2;
                break;
            }
            ph_mma ^= 1;
            ptx::tc_fence_after();
            // ---- (g) state: S <- exp(Lam_end) S + Sc (row n, columns of this half), bf16
            //      copy into sW
            {
                const float dec = ex2_approx(lam_tot);
                float sc[32];
                ptx::tmem_ld32(tmem + lane_base + kColSc + kPH * hh, sc);
#pragma unroll
                for (int pp = 0; pp < kPH; ++pp) S[pp] = fmaf(dec, S[pp], sc[pp]);
#pragma unroll
                for (int q = 0; q < 4; ++q) st_chunk(sW, row, 4 * hh + q, pack8(S + 8 * q));
            }
            // ---- (h) y = Yd + exp(Lam_t) Yo + D x (x gate), written over X in place
            {
                const float et = ex2_approx(lam);
                {
                    const int half = hh;
                    float yd[32], yo[32];
                    ptx::tmem_ld32(tmem + lane_base + kColYd + 32 * half, yd);
                    ptx::tmem_ld32(tmem + lane_base + kColYo + 32 * half, yo);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int qq = half * 4 + q;
                        const uint4 xv = ld_chunk(sX, row, qq);
                        const uint32_t xin[4] = {xv.x, xv.y, xv.z, xv.w};
                        uint32_t zin[4] = {0, 0, 0, 0};
                        if (kGate) {
                            const uint4 zv = ld_chunk(sZ, row, qq);
                            zin[0] = zv.x; zin[1] = zv.y; zin[2] = zv.z; zin[3] = zv.w;
                        }
                        uint32_t out[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const f2 xf = ptx::bf2_to_f2(xin[e]);
                            const int jj = 8 * q + 2 * e;
                            f2 y = ptx::fma2(f2{et, et}, f2{yo[jj], yo[jj + 1]},
                                             f2{yd[jj], yd[jj + 1]});
                            y = ptx::fma2(f2{Dh, Dh}, xf, y);
                            if (kGate) {
                                const f2 zf = ptx::bf2_to_f2(zin[e]);
                                y.x *= silu<true>(zf.x);
                                y.y *= silu<true>(zf.y);
                            }
                            out[e] = ptx::f2_to_bf2(y.x, y.y);
                        }
                        st_chunk(sX, row, qq, make_uint4(out[0], out[1], out[2], out[3]));
                    }
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            __syncthreads();
            if (tid == 0) {
                if (in_bounds(h < H && t0 < L && b < p.batch, status, 122))
                    ptx::tma_store_3d(&maps.Y, sX, h * kP, t0, b);
                ptx::bulk_commit();
            }
        }
        if (!ok) break;

        // ---- the segment's final state: hand it over (head) or write h_final
        if (kind == 1 && in_bounds(k < sk.nctas, status, 124)) {
            float *dst = sk.states + static_cast<int64_t>(k) * kP * kN;
#pragma unroll
            for (int pp = 0; pp < kPH; ++pp) __stcg(dst + (kPH * hh + pp) * kN + row, S[pp]);
            __threadfence();
            __syncthreads();
            if (tid == 0) ptx::st_release_u32(sk.flags + k, 1u);
        } else if (p.h_final && in_bounds(b < p.batch && h < H, status, 125)) {
            float *hf = p.h_final + (static_cast<int64_t>(b) * H + h) * kP * kN;
#pragma unroll
            for (int pp = 0; pp < kPH; ++pp) hf[(kPH * hh + pp) * kN + row] = S[pp];
        }
    }

    if (!ok) {
        if (tid == 0) report_status(status, SSM_ERR_TIMEOUT, 20 + pending);
        // give the late operation one more bounded wait before TMEM and shared
        // memory are released
        if (pending == 1) (void)ptx::mbar_wait(bar_load, ph_load);
        if (pending == 2) (void)ptx::mbar_wait(bar_mma, ph_mma);
    }
    if (tid == 0) ptx::bulk_wait<0>();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- host side
}  // namespace

bool ssd_tc_sizes_ok(const SSDParams &p) {
    if (!p.io_bf16 || p.headdim != kP || p.dstate != kN) return false;
    if (p.seqlen <= 0 || p.seqlen >= (int64_t(1) << 31)) return false;
    return p.batch * p.nheads < (int64_t(1) << 31);
}

bool ssd_tc_eligible(const SSDParams &p) {
    if (!ssd_tc_sizes_ok(p)) return false;
    const void *ptrs[] = {p.x, p.Bm, p.Cm, p.z, p.y};
    for (const void *q : ptrs)
        if (q && reinterpret_cast<uintptr_t>(q) % 16 != 0) return false;
    return tma_encoder() != nullptr;
}

// Persistent grid: two blocks per SM (their TMEM and shared memory fill an SM), but
// never more blocks than chains.
int ssd_tc_ctas(const SSDParams &p) {
    const int64_t chains = p.batch * p.nheads;
    const int64_t slots = 2 * static_cast<int64_t>(device_sm_count());
    return static_cast<int>(std::min(chains, slots));
}

// ticket + one hand-over flag per block
size_t ssd_tc_flag_bytes(const SSDParams &p) {
    return (static_cast<size_t>(ssd_tc_ctas(p) + 1) * 4 + 255) / 256 * 256;
}

size_t ssd_workspace_bytes(const SSDParams &p) {
    size_t bytes = kStatusBytes;
    if (ssd_tc_sizes_ok(p))
        bytes += ssd_tc_flag_bytes(p) + static_cast<size_t>(ssd_tc_ctas(p)) * kP * kN * 4;
    return bytes;
}

size_t ssd_clear_bytes(const SSDParams &p) {
    return kStatusBytes + (ssd_tc_sizes_ok(p) ? ssd_tc_flag_bytes(p) : 0);
}

cudaError_t launch_ssd_tc(const SSDParams &p, cudaStream_t stream) {
    Maps m{};
    const int64_t B = p.batch, L = p.seqlen, H = p.nheads, G = p.ngroups;
    // bf16 boxes of 64 columns x 128 steps, 128-byte swizzle (the UMMA operand layout)
    bool ok = make_tma_map_3d(&m.C, p.Cm, true, B, L, G * kN, 64, kQ, 128) &&
              make_tma_map_3d(&m.B, p.Bm, true, B, L, G * kN, 64, kQ, 128) &&
              make_tma_map_3d(&m.X, p.x, true, B, L, H * kP, 64, kQ, 128) &&
              make_tma_map_3d(&m.Y, p.y, true, B, L, H * kP, 64, kQ, 128);
    if (ok && p.z) ok = make_tma_map_3d(&m.Z, p.z, true, B, L, H * kP, 64, kQ, 128);
    if (!ok) return cudaErrorInvalidValue;
    Split sk{};
    sk.nch = static_cast<int>((L + kQ - 1) / kQ);
    sk.units = B * H * sk.nch;
    sk.ticket = reinterpret_cast<uint32_t *>(p.work);
    sk.flags = sk.ticket + 1;
    sk.states = reinterpret_cast<float *>(static_cast<char *>(p.work) + ssd_tc_flag_bytes(p));
    const void *func = p.z ? reinterpret_cast<const void *>(ssd_tc_kernel<true>)
                           : reinterpret_cast<const void *>(ssd_tc_kernel<false>);
    const int smem = p.z ? Smem<true>::bytes : Smem<false>::bytes;
    cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // all of the SM's unified L1/shared storage as shared memory, so that two blocks fit
    e = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    // two blocks per SM (their TMEM, shared memory and registers fill it); the ticket
    // keeps the hand-over waits safe whatever the hardware keeps resident
    sk.nctas = ssd_tc_ctas(p);
    auto kern = p.z ? ssd_tc_kernel<true> : ssd_tc_kernel<false>;
    kern<<<sk.nctas, kThreads, smem, stream>>>(m, p, sk);
    return cudaGetLastError();
}

}  // namespace ssm
