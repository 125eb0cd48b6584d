// Launch interfaces between the C ABI layer (ssm_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ssm {

struct ScanParams {
    int64_t batch, seqlen, dim, dstate;
    int io_bf16;        // 1: bf16 I/O, fast math; 0: fp32 I/O, accurate math
    int softplus;
    const void *x, *delta, *Bm, *Cm, *z;
    const float *A, *Dv, *bias, *h0;
    void *y;
    float *h_final;
    // carry across time chunks (workspace)
    int64_t chunk_len;  // steps per time chunk (multiple of the time tile)
    int nchunks;        // K
    float *hloc;        // (B, K, D, N) local end states of chunks 0..K-2
    float *dsum;        // (B, K, D) sum of steps of chunks 0..K-2
    void *status;       // DeviceStatus at the start of the workspace (may be null)
    int clear_status;   // the first block of this launch clears the status word
    int zoh;            // 1: zero-order-hold input coefficient instead of dl
    // single-launch carry (TMA kernel, nchunks > 1): a block ticket and one flag per
    // (batch row, chunk, 32-channel slab), zeroed by the caller; null: two launches
    uint32_t *ticket;
    uint32_t *flags;
    long long wait_budget;  // clock cycles a block may wait for its predecessors
    int publish;            // 0 only in the look-back self-test: summaries stay unpublished
    // optional state checkpoints for the backward pass: the state before every step t
    // with t % 2^ckpt_shift == 0, as (B, ceil(L / 2^ckpt_shift), D, N) fp32; null: none
    float *ckpt;
    int ckpt_shift;
};

// TMA-staged scan (scan_tma.cu): warps per 32-channel block for these sizes (0 = the
// sizes are not supported), whether a call can take it, and the launch.
int scan_tma_blocks_per_sm(int io_bf16, int64_t dstate);
bool scan_tma_sizes_ok(int io_bf16, int64_t seqlen, int64_t dim, int64_t dstate);
bool scan_tma_pointers_ok(const void *const *ptrs, int nptrs);
int device_sm_count();
cudaError_t launch_scan_tma(const ScanParams &p, cudaStream_t stream);

// Number of time chunks and chunk length the scan uses for these sizes; `tma_warps` > 0
// selects the plan of the TMA-staged path (blocks of 32 channels and that many warps).
void scan_plan(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int64_t time_chunk,
               int tma_blocks_per_sm, int64_t *chunk_len, int *nchunks);
size_t scan_workspace_bytes(int64_t batch, int64_t dim, int64_t dstate, int nchunks);
// Byte offset and size of the look-back ticket and flags inside a scan workspace (zero
// size when the call needs none).
void scan_lookback_region(int64_t batch, int64_t dim, int64_t dstate, int nchunks,
                          size_t *offset, size_t *bytes);
cudaError_t launch_scan(const ScanParams &p, cudaStream_t stream);

struct DecodeParams {
    int64_t batch, dim, dstate;
    int io_bf16;
    int softplus;
    int zoh;            // 1: zero-order-hold input coefficient instead of dl
    float *state;
    const void *x, *delta, *Bm, *Cm, *z;
    const float *A, *Dv, *bias;
    void *y;
    void *status;       // DeviceStatus (nullable)
};
cudaError_t launch_decode(const DecodeParams &p, cudaStream_t stream);

struct SSDParams {
    int64_t batch, seqlen, nheads, headdim, ngroups, dstate, chunk;
    int io_bf16;
    int softplus;
    const void *x, *delta, *Bm, *Cm, *z;
    const float *A, *Dv, *bias, *h0;
    void *y;
    float *h_final;
    void *status;  // DeviceStatus at the start of the workspace
    void *work;    // rest of the workspace
    size_t work_bytes;
};
size_t ssd_workspace_bytes(const SSDParams &p);
// Bytes at the start of the workspace the call must zero (status word, hand-over flags).
size_t ssd_clear_bytes(const SSDParams &p);
cudaError_t launch_ssd(const SSDParams &p, cudaStream_t stream);
cudaError_t launch_ssd_recurrent(const SSDParams &p, cudaStream_t stream);
// Chunked dual form on tcgen05 (ssd_tc.cu): bf16 I/O, headdim 64, dstate 128.
bool ssd_tc_eligible(const SSDParams &p);
cudaError_t launch_ssd_tc(const SSDParams &p, cudaStream_t stream);

struct SSDDecodeParams {
    int64_t batch, nheads, headdim, ngroups, dstate;
    int io_bf16;
    int softplus;
    float *state;
    const void *x, *delta, *Bm, *Cm, *z;
    const float *A, *Dv, *bias;
    void *y;
};
cudaError_t launch_ssd_decode(const SSDDecodeParams &p, cudaStream_t stream);

struct ScanBwdParams {
    int64_t batch, seqlen, dim, dstate;
    int io_bf16, softplus, zoh;
    const void *x, *delta, *B, *C, *z, *dy;
    const float *A, *D, *bias, *h0, *dh_final;
    void *dx, *ddelta, *dz;
    float *dA, *dB, *dC, *dD, *ddelta_bias, *dh0;
    float *ckpt;   // (B, ntiles, D, N) states at the tile starts
    int ckpt_given;  // 1: ckpt holds them already (written by the forward pass)
    void *status;    // DeviceStatus at the start of the workspace
};
size_t scan_bwd_ckpt_floats(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate);
// Steps between the backward pass's state checkpoints (its time tile): a power of two.
int scan_ckpt_steps(int64_t dstate);
cudaError_t launch_scan_bwd(const ScanBwdParams &p, cudaStream_t stream);

struct Conv1dParams {
    int64_t batch, seqlen, dim, width;
    int io_bf16;
    int silu;
    const void *x, *x_prev;
    const float *weight, *bias;
    void *out;
    void *status;   // device status word (nullable)
};
int conv1d_max_width();
bool conv1d_tma_ok(const Conv1dParams &p);
cudaError_t launch_conv1d(const Conv1dParams &p, cudaStream_t stream);

}  // namespace ssm
