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

// Decode expert path (T <= kGemvMaxTokens) in one persistent launch: miss fills from the
// mapped pool, gate/up + SwiGLU into h, down into the fp32 per-row buffer y, and the
// deterministic gate-weighted combine into out (decode.cu).
struct DecodeArgs {
  const WorkItem *work;     // [n_work]: hits, then misses (item n_hit + m uses fill m), shared
  DevCounters *ctr;
  const int32_t *fills;     // [n_fill][3] (destination entry, layer, expert)
  const uint4 *pool;        // mapped host pool [L][E][entry]
  const CacheDesc *cache;   // slot storage
  const uint16_t *x;        // [T][d]
  const int32_t *tok;       // [P + T] token of FFN row q
  const float *w;           // [T][k] gates
  const int32_t *inv;       // [P] FFN row of pair p
  uint16_t *h;              // [P + T][d_ff]
  float *y;                 // [P + T][d]
  uint16_t *out;            // [T][d]
  int32_t *sync;            // phase counters and flags [kSyncPhaseInts] | fill_done [kMaxE] |
                            // fill_dn [kMaxE]
  int T, k, d, d_ff, E, shared;
  int max_items;            // largest possible n_work: min(E, T*k) + shared (set by the launcher)
  int n_rows;               // FFN rows: T*k, plus T for the shared expert (set by the launcher)
  int R_gu, R_dn;           // rows per gate/up and per down task (set by the launcher)
  uint32_t stage_bytes;
  int n_stages;
  size_t entry_bytes;
};
constexpr int kSyncPhaseInts = 192;  // three counters and three flags, one 128-byte line each
constexpr int kSyncInts(int d) { return (void)d, kSyncPhaseInts + 2 * kMaxE; }

struct DecodePlan {
  bool xs;          // x staged in shared memory
  uint32_t ring, stage;
  int n_stages;
  int R_gu, R_dn, n_ib;
  size_t smem;
};
DecodePlan plan_decode(int T, int d, int d_ff, int max_items, int n_rows, bool fp4);
int launch_decode_experts(DecodeArgs a, bool fp4, cudaStream_t s);

// Grouped-GEMM expert FFN for larger T.
void launch_gather_rows(const uint16_t *x, const int32_t *tok, uint16_t *xp, int rows, int d,
                        const DevCounters *ctr,
                        cudaStream_t s);
// out = bf16(acc) (n % 8 == 0); with next != null also next = bf16(x + out), the residual
// stream's input of the next prefill layer.
void launch_cast_out(const float *acc, uint16_t *out, size_t n, const uint16_t *x, uint16_t *next,
                     const DevCounters *ctr, cudaStream_t s);

// Tensor maps of the tcgen05 grouped GEMMs for one weight buffer (slots, a prefill buffer):
// A views of the gathered activations and of h, B views of the buffer's entries (rows of d
// for W_gate/W_up, rows of d_ff for W_down) and of the shared-expert array.
struct TcMaps {
  CUtensorMap a_x, a_h, b_gu, b_dn256, b_dn128, bs_gu, bs_dn256, bs_dn128;
};
// 2-D bf16 view [rows][inner] of base with a box of [box_rows][64] and 128-byte swizzle.
bool make_tmap(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, uint32_t box_rows);
// gate/up then down (+ weighted red-add combine into acc) on the tensor cores.  by_item: the
// weights of work item u are entry u of the maps' buffer (expanded MXFP4 scratch), otherwise
// entry work[u].slot.
void launch_tc_ffn(const TcMaps &maps, const WorkItem *work, DevCounters *ctr, int *prefix,
                   uint16_t *h, const int32_t *tok, const float *wq, float *acc, int d, int d_ff,
                   int shared_entry, bool by_item, cudaStream_t s);
// Expand the MXFP4 entries of the call's work items to bf16: item u -> scratch entry u.
void launch_dequant_work(const WorkItem *work, const DevCounters *ctr, uint16_t *scratch, int d,
                         int d_ff, int max_items, cudaStream_t s);

// Record `code` and a message (with the CUDA error string if e != cudaSuccess) as this
// thread's ft_last_error(); returns code.
int report_error(int code, const char *what, cudaError_t e);

}  // namespace ftm
