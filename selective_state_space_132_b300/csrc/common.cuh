// Device helpers shared by the scan, SSD and decode kernels: I/O element
// conversion, the exponential used for the discretised decay, softplus for the
// step size and SiLU for the gate.  Two precision modes:
//   * kFast (bf16 I/O): the hardware approximations ex2.approx / lg2.approx /
//     tanh.approx.  Their relative error (~1e-7 for ex2, ~1e-4 for the softplus
//     of tiny steps) is far below the bf16 output rounding.
//   * accurate (fp32 I/O): CUDA's expf / log1pf, so the fp32 result tracks the
//     double-precision definition to ~1e-6.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------- I/O types
template <typename T> struct Io;
template <> struct Io<float> {
    static __device__ __forceinline__ float load(const float *p) { return __ldg(p); }
    static __device__ __forceinline__ float to_f(float v) { return v; }
    static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <> struct Io<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16 *p) {
        return __bfloat162float(__ldg(p));
    }
    static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float v) {
        return __float2bfloat16_rn(v);
    }
};

// ---------------------------------------------------------------- math
__device__ __forceinline__ float ex2_approx(float v) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float lg2_approx(float v) {
    float r;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float tanh_approx(float v) {
    float r;
    asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// softplus(v) = log(1 + e^v).  Above 20 the correction log1p(e^-v) < 2.1e-9 is
// below fp32 resolution of v, so v itself is returned.
template <bool kFast> __device__ __forceinline__ float softplus(float v) {
    if (kFast) {
        float e = ex2_approx(v * kLog2e);
        float r = lg2_approx(1.0f + e) * kLn2;
        return v > 20.0f ? v : r;
    } else {
        return v > 20.0f ? v : log1pf(expf(v));
    }
}

// SiLU(z) = z * sigmoid(z) = 0.5 z (1 + tanh(z / 2)).
template <bool kFast> __device__ __forceinline__ float silu(float z) {
    if (kFast) {
        float hz = 0.5f * z;
        return fmaf(hz, tanh_approx(hz), hz);
    } else {
        return z / (1.0f + expf(-z));
    }
}

// Discretised decay exp(dl * A).  The fast form receives A pre-multiplied by
// log2(e) and computes 2^(dl * A log2 e).
template <bool kFast> __device__ __forceinline__ float decay(float dl, float a_scaled) {
    if (kFast) return ex2_approx(dl * a_scaled);
    return expf(dl * a_scaled);
}
template <bool kFast> __device__ __forceinline__ float scale_A(float a) {
    return kFast ? a * kLog2e : a;
}

// Zero-order-hold input coefficient (exp(v) - 1) / A with v = dl * A (natural log),
// given a = exp(v) already computed and invA = 1 / A (0 when A = 0).  Near v = 0 the
// difference a - 1 loses its leading digits, so there the series
// dl (1 + v / 2 + v^2 / 6) is used (relative error below 1.5e-6 at |v| = 1/32; it
// is also the A -> 0 limit dl).  The accurate mode uses expm1f.
template <bool kFast> __device__ __forceinline__ float zoh_coef(float dl, float v, float a,
                                                               float invA) {
    const float series = dl * fmaf(v, fmaf(v, 1.f / 6.f, 0.5f), 1.f);
    const float direct = kFast ? (a - 1.f) * invA : expm1f(v) * invA;
    return fabsf(v) < (1.f / 32.f) ? series : direct;
}

// Step size from the raw value and the bias, with or without softplus.
template <bool kFast> __device__ __forceinline__ float step_size(float raw, float bias,
                                                                 int use_softplus) {
    float v = raw + bias;
    return use_softplus ? softplus<kFast>(v) : v;
}

// ---------------------------------------------------------------- device status word
// The first 256 bytes of every workspace hold a status header; word 0 is an
// ssm_status value the kernels set (never clear) when a bounded wait gives up.
struct DeviceStatus {
    int32_t code;
    int32_t where;
    int32_t pad[62];
};
constexpr size_t kStatusBytes = 256;
// Clock budget of a block waiting for the chunk summaries of its predecessors in the
// single-launch scan (about one second at 2 GHz).
constexpr long long kScanWaitCycles = 2000000000LL;

__device__ __forceinline__ void report_status(DeviceStatus *st, int code, int where) {
    if (st) {
        atomicCAS(&st->code, 0, code);
        st->where = where;
    }
}

// Index checks of the debug-bounds build (SSM_DEBUG_BOUNDS=1): the kernels guard their
// global writes and TMA coordinates with in_bounds(...); a failed check records
// SSM_ERR_BOUNDS with the site number in the status word and the caller skips the
// access.  Release builds compile the checks out (in_bounds is true).
#ifndef SSM_DEBUG_BOUNDS
#define SSM_DEBUG_BOUNDS 0
#endif
constexpr bool kDebugBounds = SSM_DEBUG_BOUNDS != 0;
__device__ __forceinline__ bool in_bounds(bool ok, DeviceStatus *st, int site) {
    if constexpr (kDebugBounds) {
        if (!ok) report_status(st, 7 /* SSM_ERR_BOUNDS */, site);
        return ok;
    } else {
        (void)ok; (void)st; (void)site;
        return true;
    }
}

}  // namespace ssm
