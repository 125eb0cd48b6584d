/*
 * ssm.h — C ABI of the B300 selective state-space library (libssm.so).
 *
 * Three operations, all forward, all on one GPU:
 *
 *   ssm_scan_fwd      the selective (S6) scan.  Per channel d of batch b:
 *                       dl_t  = softplus(delta_t + bias_d)      (or without softplus)
 *                       h_t   = exp(dl_t * A_d) (.) h_{t-1} + dl_t * B_t * x_t
 *                       y_t   = (C_t . h_t + D_d * x_t) * silu(z_t)   (gate optional)
 *                     Defined by "Mamba 논문 리뷰: 선형 시간복잡도로 Transformer에
 *                     도전하는 Selective State Space Model" (tildalice.io), sections
 *                     "Selection Mechanism" (Δ_t = softplus(s_Δ(x_t))), "Δ의 직관적
 *                     이해" (the recurrence with B̄ = ΔB) and "Mamba 블록 아키텍처"
 *                     (the SiLU gate); the D skip term from "[yongggg's] Mamba ...
 *                     (Review)", section "State Space Model".
 *
 *   ssm_ssd_chunk_fwd the same recurrence with a scalar decay per head and a P x N
 *                     matrix state per head (Mamba-2), computed in its chunked dual
 *                     form: inside a chunk Y = (L o C B^T)(dl x), between chunks the
 *                     state is passed on.  "Mamba-2: 상태 공간 기반 시퀀스 모델"
 *                     (obsidian-dorae222.pages.dev), sections "1-세미분리 행렬",
 *                     "SSM-Attention 동치성", "멀티-헤드 구조" and "SSD 타일링 알고리즘".
 *
 *   ssm_step_decode   one recurrent step for one new token per sequence, updating a
 *                     fixed-size state in place (tildalice review, section "추론 속도":
 *                     O(D x N) state, no cache that grows with the sequence).
 *
 * Conventions shared by every entry point
 *   - Every data pointer is a DEVICE pointer to a dense row-major array; the caller
 *     allocates and owns all of them, the workspace included.  The library never
 *     allocates or frees memory and keeps no per-call state.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).  They
 *     validate their arguments on the host first and, on any error, return a status
 *     without launching anything.
 *   - I/O dtype: x, delta, B, C, z and y are all `io_dtype` (fp32 or bf16).  A, D,
 *     delta_bias, the states and every intermediate are fp32.  bf16 outputs are
 *     rounded once, to nearest even.
 *   - y must not alias any input.  The decode state is updated in place by design.
 *   - Errors found on the device (a bounded wait that ran out, or in a build with
 *     SSM_DEBUG_BOUNDS=1 a failed index check) are written to a status word at the
 *     start of the workspace; read it with ssm_read_device_status.
 *   - No C++ exception crosses this interface.
 */
#ifndef SSM_B300_H
#define SSM_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SSM_API __attribute__((visibility("default")))
#else
#define SSM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as cudaStream_t. */
typedef struct CUstream_st *ssm_stream_t;

typedef enum {
    SSM_OK = 0,
    SSM_ERR_INVALID_ARG = 1, /* a null required pointer, a negative size, H % G != 0, ... */
    SSM_ERR_UNSUPPORTED = 2, /* a valid request the library does not implement (e.g. N > 64) */
    SSM_ERR_ALIGNMENT = 3,   /* a pointer is not aligned to its element size */
    SSM_ERR_WORKSPACE = 4,   /* workspace missing or smaller than *_workspace_size says */
    SSM_ERR_CUDA = 5,        /* the CUDA runtime reported an error at launch */
    SSM_ERR_TIMEOUT = 6,     /* (device status only) a bounded wait gave up */
    SSM_ERR_BOUNDS = 7       /* (device status only, builds with SSM_DEBUG_BOUNDS=1) a
                                kernel's index check failed; the access was skipped */
} ssm_status;

typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype;

/* ------------------------------------------------------------------ S6 scan
 * Shapes (B = batch, L = seqlen, D = dim, N = dstate):
 *   x, delta, z, y : (B, L, D) io_dtype        B, C : (B, L, N) io_dtype
 *   A              : (D, N) fp32 (expected < 0) D, delta_bias : (D) fp32
 *   h0, h_final    : (B, D, N) fp32
 * Nullable: D (no skip), delta_bias (zero), z (no gate), h0 (zero initial state),
 * h_final (final state not returned).  Sizes: B, L >= 0, D >= 1, 1 <= N <= 64.
 * B, L or D of zero is valid; then only h_final (= h0, or zeros) is written.
 * time_chunk: 0 lets the library choose how many time steps one thread block walks;
 * a positive value (a multiple of 32) forces it, which splits long sequences over
 * several blocks joined by a carry (exact up to rounding): each block of a later time
 * chunk folds the end states of the earlier chunks of its channels, computed from a
 * zero state (tildalice review, section "2. 병렬 스캔": the associative combine over
 * whole chunks).  The TMA kernel does this in one launch, each block publishing its
 * chunk's summary with a release store and acquiring its predecessors' with a bounded
 * wait (SSM_ERR_TIMEOUT in the status word if one ever gave up); the general kernel in
 * two (a summary pass, then the output pass).
 * Workspace: ssm_scan_workspace_size() bytes (it reads only the sizes and flags of
 * `args`, not the pointers), 256-byte aligned, always required: its first 256 bytes
 * hold the device status word, the rest the chunk summaries and the hand-over flags of
 * a time-split sequence; the call clears what must start at zero, so the contents need
 * no initialisation.
 * discretization: SSM_DISC_EULER (0, B̄ = dl B: the simplified form of the tildalice
 * review, section "Δ의 직관적 이해") or SSM_DISC_ZOH (1, zero-order hold:
 * B̄ = (exp(dl A) - 1) / A B, section "이산화"; the A -> 0 limit is dl B). */
typedef enum { SSM_DISC_EULER = 0, SSM_DISC_ZOH = 1 } ssm_discretization;
typedef struct {
    int64_t batch, seqlen, dim, dstate;
    int64_t time_chunk;
    int32_t io_dtype;       /* ssm_dtype */
    int32_t delta_softplus; /* 0 or 1 */
    const void *x, *delta, *B, *C, *z;
    const float *A, *D, *delta_bias, *h0;
    void *y;
    float *h_final;
    void *workspace;
    size_t workspace_bytes;
    int32_t discretization; /* ssm_discretization */
    int32_t reserved;       /* 0 */
} ssm_scan_args;

SSM_API ssm_status ssm_scan_workspace_size(const ssm_scan_args *args, size_t *bytes);
/* How ssm_scan_fwd will run these sizes (reads sizes and flags only): the time
 * steps per chunk, the number of chunks along time, and the kernel launches per
 * call (1, or 2 when a split sequence runs on the general kernel's summary pass). */
SSM_API ssm_status ssm_scan_plan(const ssm_scan_args *args, int64_t *chunk_len,
                                 int32_t *nchunks, int32_t *launches);
SSM_API ssm_status ssm_scan_fwd(const ssm_scan_args *args, ssm_stream_t stream);

/* ------------------------------------------------------------------ scan backward
 * Gradients of ssm_scan_fwd, rebuilding the hidden states from the inputs instead of
 * storing them in the forward pass (tildalice review, section "Hardware-Aware 병렬
 * 알고리즘", item "역전파 시 재계산"; yongggg review, section "하드웨어 인식 알고리즘").  The arithmetic is the adjoint of the recurrence of
 * ssm_scan_fwd, with lam = dLoss/dh_t walking back in time:
 *   g = dy silu(z);  dz = dy (C.h + D x) silu'(z);  dC_t += g h_t;  lam += g C_t;
 *   dB_t += lam c x;  dx = g D + sum_n lam c B;  ddl = sum_n lam (h_{t-1} a A + B x dc/ddl);
 *   dA += lam (h_{t-1} a dl + B x dc/dA);  lam *= a;  ddelta = ddl softplus'(delta + bias)
 * with a = exp(dl A) and c = dl (Euler) or (exp(dl A) - 1)/A (zero-order hold).
 *   - Forward inputs, sizes and flags: as in ssm_scan_args (x, delta, B, C, z in
 *     io_dtype; A (D,N), D, delta_bias (D), h0 (B,D,N) fp32; D, delta_bias, z, h0
 *     nullable).
 *   - dy (B,L,D) io_dtype: gradient of y.  dh_final (B,D,N) fp32: gradient of the
 *     final state, nullable (zero).
 *   - Outputs, all written (never accumulated into):
 *       dx, ddelta (B,L,D) io_dtype (ddelta is the gradient of the raw delta);
 *       dz (B,L,D) io_dtype, required iff z is given;
 *       dB, dC (B,L,N) fp32 (sums over channels); dA (D,N) fp32 (sum over batch rows);
 *       dD, ddelta_bias (D) fp32, nullable (gradients of D and of the bias, computed
 *       even when D or delta_bias is NULL, i.e. taken at zero); dh0 (B,D,N) fp32,
 *       nullable.
 *   - No output may overlap an input or another output.
 *   - workspace: ssm_scan_bwd_workspace_size bytes, 256-byte aligned: a status
 *     word and the state at the start of every time tile of every (b, d) chain, fp32.
 *   - N <= 64; the channels of one batch row run as one chain per channel, so a
 *     single very long sequence has B * ceil(D / 32) blocks of parallelism. */
typedef struct {
    int64_t batch, seqlen, dim, dstate;
    int32_t io_dtype;
    int32_t delta_softplus;
    int32_t discretization;
    int32_t reserved;
    const void *x, *delta, *B, *C, *z;
    const float *A, *D, *delta_bias, *h0;
    const void *dy;
    const float *dh_final;
    void *dx, *ddelta, *dz;
    float *dA, *dB, *dC, *dD, *ddelta_bias, *dh0;
    void *workspace;
    size_t workspace_bytes;
} ssm_scan_bwd_args;

SSM_API ssm_status ssm_scan_bwd_workspace_size(const ssm_scan_bwd_args *args, size_t *bytes);
SSM_API ssm_status ssm_scan_bwd(const ssm_scan_bwd_args *args, ssm_stream_t stream);

/* ------------------------------------------------------------------ state checkpoints
 * No counterpart in the pages: an optional trade of memory for backward time.
 * ssm_scan_bwd rebuilds the hidden states from checkpoints: the state before every
 * step t with t % T == 0, T = 32 (N <= 8), 16 (N <= 16), 8 (N <= 32) or 4 (N <= 64),
 * stored as a (B, ceil(L / T), D, N) fp32 tensor.  It computes them itself, in a
 * forward pass over the sequence at the start of the call.  A caller that can keep
 * them from its forward call to its backward call (L / T times the size of h_final)
 * saves that pass:
 *   - ssm_scan_ckpt_size: T and the bytes of the checkpoint tensor for the sizes of
 *     `args` (reads sizes only).
 *   - ssm_scan_fwd_ckpt: ssm_scan_fwd (same arguments, workspace and results), and
 *     it also writes the checkpoints to `ckpt` (device memory, caller-owned, 16-byte
 *     aligned, at least ssm_scan_ckpt_size bytes; SSM_ERR_INVALID_ARG when it is
 *     smaller or missing).  The states are the scan's own, to rounding: a sequence the
 *     scan splits over time holds the states folded through the chunk summaries.
 *   - ssm_scan_bwd_ckpt: ssm_scan_bwd (same arguments and results), reading the
 *     checkpoints from `ckpt` (as written by ssm_scan_fwd_ckpt for the same inputs)
 *     instead of computing them; its workspace needs only the 256-byte status word.
 *     Checkpoints of other inputs give wrong gradients, not an error. */
SSM_API ssm_status ssm_scan_ckpt_size(const ssm_scan_args *args, int64_t *steps,
                                      size_t *bytes);
SSM_API ssm_status ssm_scan_fwd_ckpt(const ssm_scan_args *args, float *ckpt,
                                     size_t ckpt_bytes, ssm_stream_t stream);
SSM_API ssm_status ssm_scan_bwd_ckpt(const ssm_scan_bwd_args *args, const float *ckpt,
                                     size_t ckpt_bytes, ssm_stream_t stream);

/* ------------------------------------------------------------------ scan without allocation
 * No counterpart in the pages: a library convenience.  Same computation, arguments
 * and results as ssm_scan_fwd, but the scratch that a time-split sequence needs
 * comes from a fixed buffer inside the library instead of args->workspace (which
 * is ignored), so the caller allocates nothing beyond its inputs and outputs.  It
 * is meant for callers that cannot allocate device memory on the call path: a
 * plugin inside another runtime that owns all device memory, a latency-critical
 * loop that cannot afford cudaMalloc's implicit synchronisation, or a process
 * limited to memory reserved at start-up.
 *   - The buffer holds SSM_NOALLOC_SCRATCH_BYTES (4 MiB) on every GPU that loads
 *     the library, until the process exits.  Problems whose scratch need, as
 *     reported by ssm_scan_workspace_size, is larger are rejected with
 *     SSM_ERR_UNSUPPORTED before anything is launched.
 *   - The first call on a device looks up the buffer's device address for that
 *     device (cudaGetSymbolAddress, with the device current); make that first
 *     call before any stream capture.  No call allocates memory.
 *   - Every call on a device shares the one buffer and leaves its contents behind;
 *     the call clears what must start at zero itself.  Calls whose work overlaps
 *     on the GPU (other streams, other host threads) race on the buffer: order
 *     them on one stream or synchronise between them.
 *   - The device status word that ssm_scan_fwd keeps at the start of the caller's
 *     workspace sits at the start of the library's buffer here, where the caller
 *     cannot read it (ssm_read_device_status needs a caller pointer) and the next
 *     call clears it: a bounded wait that runs out inside this call's kernels is not
 *     reported.  Callers that need that report use ssm_scan_fwd with a workspace. */
#define SSM_NOALLOC_SCRATCH_BYTES (4u << 20)
SSM_API ssm_status ssm_scan_fwd_noalloc(const ssm_scan_args *args, ssm_stream_t stream);

/* ------------------------------------------------------------------ SSD (Mamba-2)
 * Shapes (H = nheads, P = headdim, G = ngroups, N = dstate; head h reads group
 * h / (H / G)):
 *   x, z, y : (B, L, H, P) io_dtype     delta : (B, L, H) io_dtype
 *   B, C    : (B, L, G, N) io_dtype     A, D, delta_bias : (H) fp32
 *   h0, h_final : (B, H, P, N) fp32
 * Nullable: D, delta_bias, z, h0, h_final.  H % G == 0.  chunk_size (>= 0): the
 * chunk length Q asked for the dual form.  The tensor-core kernel (bf16 I/O, P = 64,
 * N = 128) always works in 128-step chunks: a longer chunk is the same sum with its
 * below-diagonal 128 x 128 blocks factored through the state at the block boundary,
 * so the result does not depend on chunk_size beyond rounding.  Other shapes run a
 * sequential recurrence kernel.  Workspace: ssm_ssd_workspace_size() bytes,
 * 256-byte aligned (its first 256 bytes hold the device status word). */
typedef struct {
    int64_t batch, seqlen, nheads, headdim, ngroups, dstate;
    int64_t chunk_size;
    int32_t io_dtype;
    int32_t delta_softplus;
    const void *x, *delta, *B, *C, *z;
    const float *A, *D, *delta_bias, *h0;
    void *y;
    float *h_final;
    void *workspace;
    size_t workspace_bytes;
} ssm_ssd_args;

SSM_API ssm_status ssm_ssd_workspace_size(const ssm_ssd_args *args, size_t *bytes);
SSM_API ssm_status ssm_ssd_chunk_fwd(const ssm_ssd_args *args, ssm_stream_t stream);
/* Which kernel ssm_ssd_chunk_fwd runs for these arguments (reads sizes, flags and
 * pointer alignment): 1 = the chunked dual form on tcgen05 tensor cores (chunk 128),
 * 0 = the sequential recurrence. */
SSM_API ssm_status ssm_ssd_plan(const ssm_ssd_args *args, int32_t *tensor_core);

/* ------------------------------------------------------------------ decode step
 * Shapes: state (B, D, N) fp32, read and written IN PLACE;
 *   x, delta, z, y : (B, D) io_dtype    B, C : (B, N) io_dtype
 *   A : (D, N) fp32                    D, delta_bias : (D) fp32
 * Nullable: D, delta_bias, z.  One call advances every sequence by one token;
 * calls on one stream are ordered, so L calls equal one ssm_scan_fwd over L steps
 * (up to rounding) with the same discretization.
 * workspace (optional): a 256-byte device status word, read with
 * ssm_read_device_status; the bulk-copy kernel (N a multiple of 8 up to 64, 16-byte
 * aligned rows) writes SSM_ERR_TIMEOUT there if one of its bounded waits gives up
 * (without a workspace such a timeout goes unreported).  The call clears it first. */
typedef struct {
    int64_t batch, dim, dstate;
    int32_t io_dtype;
    int32_t delta_softplus;
    float *state;
    const void *x, *delta, *B, *C, *z;
    const float *A, *D, *delta_bias;
    void *y;
    int32_t discretization; /* ssm_discretization */
    int32_t reserved;       /* 0 */
    void *workspace;        /* nullable; if given, >= 256 bytes, 256-byte aligned */
    size_t workspace_bytes;
} ssm_decode_args;

SSM_API ssm_status ssm_step_decode(const ssm_decode_args *args, ssm_stream_t stream);

/* ------------------------------------------------------------------ multi-head decode step
 * One token of the multi-head scalar-A recurrence that ssm_ssd_chunk_fwd computes in
 * its chunked form ("Mamba-2: 상태 공간 기반 시퀀스 모델", section "멀티-헤드 구조";
 * tildalice review, section "추론 속도" for the fixed-size state).  Per sequence b and
 * head h (group g = h / (H / G)), dl = softplus(delta + bias_h):
 *   S[p, :] <- exp(dl A_h) S[p, :] + dl x_p B_g ;   y_p = S[p, :] . C_g + D_h x_p  (x silu(z_p))
 * Shapes: state (B, H, P, N) fp32, read and written IN PLACE;
 *   x, z, y : (B, H, P) io_dtype     delta : (B, H) io_dtype
 *   B, C    : (B, G, N) io_dtype     A, D, delta_bias : (H) fp32
 * Nullable: D, delta_bias, z.  H % G == 0, 1 <= N <= 256.  L calls on one stream equal
 * one ssm_ssd_chunk_fwd over the same L tokens (up to rounding).  No workspace. */
typedef struct {
    int64_t batch, nheads, headdim, ngroups, dstate;
    int32_t io_dtype;
    int32_t delta_softplus;
    float *state;
    const void *x, *delta, *B, *C, *z;
    const float *A, *D, *delta_bias;
    void *y;
} ssm_ssd_decode_args;

SSM_API ssm_status ssm_ssd_step_decode(const ssm_ssd_decode_args *args, ssm_stream_t stream);

/* ------------------------------------------------------------------ causal conv1d + SiLU
 * The Conv1D (kernel K) + SiLU step in front of the selective scan in the Mamba block
 * (tildalice review, section "Mamba 블록 아키텍처" and its reference class: a depthwise
 * Conv1D with K - 1 steps of left padding, cropped to L, then SiLU):
 *   out[b, t, d] = silu( bias_d + sum_{k<K} weight[d, k] x[b, t - (K-1) + k, d] )
 * x at t < 0 comes from x_prev (the K - 1 inputs just before this call, oldest first),
 * or is zero when x_prev is NULL, so a sequence can be processed in pieces.
 * Shapes: x, out (B, L, D) io_dtype; x_prev (B, K - 1, D) io_dtype; weight (D, K) fp32;
 * bias (D) fp32.  Nullable: bias, x_prev.  1 <= K <= 8; silu 0 returns the
 * convolution alone.  out may not alias x or x_prev.
 * workspace (optional): a 256-byte device status word, read with
 * ssm_read_device_status; the TMA-tiled kernel records SSM_ERR_TIMEOUT there if one of
 * its bounded waits gives up (without a workspace such a timeout goes unreported). */
typedef struct {
    int64_t batch, seqlen, dim, width;
    int32_t io_dtype;
    int32_t silu;
    const void *x, *x_prev;
    const float *weight, *bias;
    void *out;
    void *workspace;           /* nullable; if given, >= 256 bytes, 256-byte aligned */
    size_t workspace_bytes;
} ssm_conv1d_args;

SSM_API ssm_status ssm_conv1d(const ssm_conv1d_args *args, ssm_stream_t stream);

/* ------------------------------------------------------------------ utilities */
SSM_API const char *ssm_status_string(ssm_status status);
SSM_API int ssm_version(void); /* major * 10000 + minor * 100 + patch */

/* Synchronises `stream`, then reads the device status word that the kernels of
 * the last call using `workspace` left there (SSM_OK when none failed). */
SSM_API ssm_status ssm_read_device_status(const void *workspace, ssm_stream_t stream,
                                  ssm_status *device_status);

/* Diagnostic, no counterpart in the pages.  Every spin-wait in the kernels is bounded;
 * this call shows what happens when one runs out.  It clears the 256-byte status header
 * at `workspace` (256-byte aligned), then runs one thread that waits, through the same
 * acquire-and-back-off routine the SSD kernel uses to take over the state of the block
 * before it, on a flag that nothing sets.  After `budget_cycles` SM clock cycles
 * (1 .. 2e9; about 1 ms per 2e6 on B300) the wait gives up and the kernel records
 * SSM_ERR_TIMEOUT, which ssm_read_device_status then returns; the CUDA context stays
 * usable.  Asynchronous on `stream`. */
SSM_API ssm_status ssm_check_bounded_wait(void *workspace, int64_t budget_cycles,
                                          ssm_stream_t stream);

/* Diagnostic, no counterpart in the pages.  Runs ssm_scan_fwd's single-launch form
 * (a sequence the TMA kernel splits over time chunks; otherwise SSM_ERR_UNSUPPORTED)
 * with the chunk summaries left unpublished and a wait budget of `budget_cycles` SM
 * clock cycles (1 .. 2e9).  The blocks of every chunk after the first wait for a
 * predecessor that never publishes, give up after the budget, record SSM_ERR_TIMEOUT in
 * the status word at the start of args->workspace and return without writing their
 * outputs; the CUDA context stays usable.  Arguments and workspace as ssm_scan_fwd.
 * Asynchronous on `stream`. */
SSM_API ssm_status ssm_check_scan_lookback(const ssm_scan_args *args, int64_t budget_cycles,
                                           ssm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SSM_B300_H */
