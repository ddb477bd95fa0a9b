// Host-side launchers shared between the translation units of the ft_moe library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace ftm {

// Router logits in the fixed fp32 order (see route.cu): x [T][d], wr [E][d] -> logits [T][E].
void launch_router(const uint16_t *x, const uint16_t *wr, const float *bias, float *logits,
                   int T, int E, int d, cudaStream_t s);

// Top-k per token (warp per token): idx [T][k], w [T][k], tie [T].
void launch_topk(const float *logits, int32_t *idx, float *w, uint8_t *tie, int T, int E,
                 int k, cudaStream_t s);

// Stable grouping of the T*k pairs by expert for large P (three kernels).
void launch_perm_multi(const ControlArgs &a, int32_t *chunk_scratch, cudaStream_t s);
size_t perm_multi_scratch_ints(int P, int E);

// Single-CTA control: (optionally) permutation, then LRU update + fill list (decode) or
// buffer mapping (prefill), work list, counters.
void launch_control(const ControlArgs &a, bool perm_ready, cudaStream_t s);
constexpr int kPermSingleMax = 1024;  // largest P the single-CTA control permutes itself

// Copy the fill list's entries from the mapped host pool into their slots.
void launch_fill(const uint16_t *pool_dev, uint16_t *slots, const int32_t *fills,
                 const DevCounters *ctr, size_t entry_bytes, int E, int max_fill, cudaStream_t s);

// Decode expert FFN (T <= kGemvMaxTokens): gate/up GEMV + SwiGLU into h, then down GEMV with
// the weighted combine into out.
void launch_gateup_gemv(const WorkItem *work, const DevCounters *ctr, int max_work,
                        const uint16_t *x, const int32_t *tok, uint16_t *h, int T, int d,
                        int d_ff, cudaStream_t s);
void launch_down_gemv(const WorkItem *work, const DevCounters *ctr, int max_work,
                      const uint16_t *h, const int32_t *tok, const float *wq, uint16_t *out,
                      int T, int d, int d_ff, cudaStream_t s);

// Grouped-GEMM expert FFN for larger T.
void launch_gather_rows(const uint16_t *x, const int32_t *tok, uint16_t *xp, int rows, int d,
                        cudaStream_t s);
void launch_gemm_gateup(const WorkItem *work, const DevCounters *ctr, int max_work, int max_rows,
                        const uint16_t *xp, uint16_t *h, int d, int d_ff, cudaStream_t s);
void launch_gemm_down(const WorkItem *work, const DevCounters *ctr, int max_work, int max_rows,
                      const uint16_t *h, const int32_t *tok, const float *wq, float *acc, int d,
                      int d_ff, cudaStream_t s);
void launch_cast_out(const float *acc, uint16_t *out, size_t n, const DevCounters *ctr,
                     cudaStream_t s);

// Record `code` and a message (with the CUDA error string if e != cudaSuccess) as this
// thread's ft_last_error(); returns code.
int report_error(int code, const char *what, cudaError_t e);

}  // namespace ftm
