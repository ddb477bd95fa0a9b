// Host-side launchers shared between the translation units of the ft_moe library.
#pragma once

#include <cuda.h>
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

// Decode routing in one launch: router logits, then (last CTA) top-k + control.  T <= 16.
void launch_route_decode(const uint16_t *x, const uint16_t *wr, const float *bias, float *logits,
                         const ControlArgs &a, cudaStream_t s);

// Copy the fill list's entries from the mapped host pool into their slots.
void launch_fill(const uint16_t *pool_dev, const CacheDesc *cache, const int32_t *fills,
                 DevCounters *ctr, size_t entry_bytes, int E, int max_fill, cudaStream_t s);

// Decode expert FFN (T <= kGemvMaxTokens): gate/up GEMV + SwiGLU into h; down GEMV into the
// fp32 per-row buffer y [(T*k + T)][d]; then the deterministic weighted combine into out.
// fp4: the entries are MXFP4 (codes then block scales) instead of bf16
void launch_gateup_gemv(const WorkItem *work, DevCounters *ctr, int max_work, const uint16_t *x,
                        const int32_t *tok, uint16_t *h, int T, int d, int d_ff, bool fp4,
                        cudaStream_t s);
void launch_down_gemv(const WorkItem *work, DevCounters *ctr, int max_work, const uint16_t *h,
                      float *y, int T, int d, int d_ff, bool fp4, cudaStream_t s);
void launch_combine(const float *y, const float *w, const int32_t *inv, const DevCounters *ctr,
                    uint16_t *out, int T, int k, int d, int shared, cudaStream_t s);

// Grouped-GEMM expert FFN for larger T.
void launch_gather_rows(const uint16_t *x, const int32_t *tok, uint16_t *xp, int rows, int d,
                        const DevCounters *ctr,
                        cudaStream_t s);
void launch_cast_out(const float *acc, uint16_t *out, size_t n, const DevCounters *ctr,
                     cudaStream_t s);

// Tensor maps of the tcgen05 grouped GEMMs for one weight buffer (slots, a prefill buffer):
// A views of the gathered activations and of h, B views of the buffer's entries (rows of d
// for W_gate/W_up, rows of d_ff for W_down) and of the shared-expert array.
struct TcMaps {
  CUtensorMap a_x, a_h, b_gu, b_dn256, b_dn128, bs_gu, bs_dn256, bs_dn128;
};
// 2-D bf16 view [rows][inner] of base with a box of [box_rows][64] and 128-byte swizzle.
bool make_tmap(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, uint32_t box_rows);
// gate/up then down (+ weighted red-add combine into acc) on the tensor cores.
void launch_tc_ffn(const TcMaps &maps, const WorkItem *work, DevCounters *ctr, int *prefix,
                   uint16_t *h, const int32_t *tok, const float *wq, float *acc, int d, int d_ff,
                   int shared_entry, cudaStream_t s);

// Record `code` and a message (with the CUDA error string if e != cudaSuccess) as this
// thread's ft_last_error(); returns code.
int report_error(int code, const char *what, cudaError_t e);

}  // namespace ftm
