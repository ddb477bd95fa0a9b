// Routing and control kernels: router logits, top-k + gates, grouping of (token, rank) pairs
// by expert, and the device-side LRU update of the (layer, expert) -> slot cache.
//
// FreeToken RTX 4090, section "how the MoE memory hierarchy works": each token selects a
// few routed experts per layer (6 of 256 in its example); the GPU cache holds complete
// (layer, expert) entries under one logical mapping and is managed as an LRU shared across
// layers and tokens.  FreeToken benchmark, "graph compatibility": routing-dependent
// decisions stay in device memory so the step can be captured; nothing here returns
// control data to the host.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <type_traits>

#include "internal.h"

namespace ftm {

// ---------------------------------------------------------------------------------------
// Router logits.
//
// Summation order (fixed, so the chosen experts are a reproducible function of the inputs;
// the fp32 CPU oracle follows the same order):  d is cut into chunks of 8 features; lane
// lam of a warp owns chunks c = lam, lam+32, ... in increasing order and adds the 8 products
// of each chunk in feature order from +0.0; the 32 lane sums are combined by the xor
// butterfly 16, 8, 4, 2, 1; the bias is added last.  A warp computes TT tokens x EE experts
// at once: every lane keeps TT*EE partial sums, each following exactly that order.
// ---------------------------------------------------------------------------------------
template <int TT, int EE>
__global__ void __launch_bounds__(256) k_router(const uint16_t *__restrict__ x,
                                                const uint16_t *__restrict__ wr,
                                                const float *__restrict__ bias,
                                                float *__restrict__ logits, int T, int E,
                                                int d) {
  const int lane = threadIdx.x & 31;
  const long warp = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int n_eb = (E + EE - 1) / EE;
  const long tb = warp / n_eb;
  const int eb = (int)(warp - tb * n_eb);
  const int t0 = (int)tb * TT, e0 = eb * EE;
  if (t0 >= T) return;
  float acc[TT][EE];
#pragma unroll
  for (int i = 0; i < TT; ++i)
#pragma unroll
    for (int j = 0; j < EE; ++j) acc[i][j] = 0.f;
  const int nchunk = d >> 3;
#pragma unroll 2
  for (int c = lane; c < nchunk; c += 32) {
    uint4 xv[TT], wv[EE];
#pragma unroll
    for (int i = 0; i < TT; ++i)
      xv[i] = (t0 + i < T) ? __ldg(reinterpret_cast<const uint4 *>(x + (size_t)(t0 + i) * d) + c)
                           : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int j = 0; j < EE; ++j)
      wv[j] = (e0 + j < E) ? __ldg(reinterpret_cast<const uint4 *>(wr + (size_t)(e0 + j) * d) + c)
                           : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < TT; ++i)
#pragma unroll
      for (int j = 0; j < EE; ++j) acc[i][j] = dot8_seq(xv[i], wv[j], acc[i][j]);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
    for (int i = 0; i < TT; ++i)
#pragma unroll
      for (int j = 0; j < EE; ++j) acc[i][j] = acc[i][j] + __shfl_xor_sync(0xffffffffu, acc[i][j], off);
#pragma unroll
  for (int i = 0; i < TT; ++i)
#pragma unroll
    for (int j = 0; j < EE; ++j) {
      if (lane == ((i * EE + j) & 31) && t0 + i < T && e0 + j < E) {
        float v = acc[i][j];
        if (bias) v = v + bias[e0 + j];
        logits[(size_t)(t0 + i) * E + e0 + j] = v;
      }
    }
}

void launch_router(const uint16_t *x, const uint16_t *wr, const float *bias, float *logits, int T,
                   int E, int d, cudaStream_t s) {
  const int threads = 256, wpb = threads / 32;
  auto grid = [&](int tt, int ee) {
    long warps = (long)((T + tt - 1) / tt) * ((E + ee - 1) / ee);
    return (unsigned)((warps + wpb - 1) / wpb);
  };
  if (T == 1)
    k_router<1, 1><<<grid(1, 1), threads, 0, s>>>(x, wr, bias, logits, T, E, d);
  else if (T <= 2)
    k_router<2, 2><<<grid(2, 2), threads, 0, s>>>(x, wr, bias, logits, T, E, d);
  else
    k_router<4, 4><<<grid(4, 4), threads, 0, s>>>(x, wr, bias, logits, T, E, d);
}

// ---------------------------------------------------------------------------------------
// Top-k per token, one warp per token.  k+1 rounds of a warp argmax over the not yet
// selected experts, ordered by (logit descending, expert id ascending); the (k+1)-th value
// only feeds the near-tie report.  Gates: softmax over the k selected logits (which equals
// the full softmax renormalised over the top-k).
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// One warp: top-k of one token's E logits (NV = ceil(E/32) values per lane).
template <int NV>
__device__ __forceinline__ void topk_warp(const float *__restrict__ row, int E, int k,
                                          int32_t *idx_row, float *w_row, uint8_t *tie_t) {
  const int lane = threadIdx.x & 31;
  float v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? __ldcg(row + e) : -INFINITY;
  }
  uint32_t taken = 0;  // bit i: expert lane+32i already selected
  float sel_v = 0.f;   // lane j keeps the j-th selected logit
  int sel_i = 0;
  float next_v = -INFINITY;
  const int rounds = (k < E) ? k + 1 : k;
  for (int r = 0; r < rounds; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && better(v[i], e, bv, bi)) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (r < k) {
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (lane == r) {
        sel_v = bv;
        sel_i = bi;
      }
    } else {
      next_v = bv;
    }
  }
  // gates: w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0)
  const float l0 = __shfl_sync(0xffffffffu, sel_v, 0);
  const float ex = (lane < k) ? expf(sel_v - l0) : 0.f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  // near-tie: exact differences of fp32 logits (done in double)
  const float nxt_sel = __shfl_down_sync(0xffffffffu, sel_v, 1);
  bool near = false;
  if (lane + 1 < k) near = ((double)sel_v - (double)nxt_sel) <= kNearTie;
  if (lane == k - 1 && k < E) near = near || ((double)sel_v - (double)next_v) <= kNearTie;
  const bool any_near = __any_sync(0xffffffffu, near);
  if (lane < k) {
    idx_row[lane] = sel_i;
    w_row[lane] = ex / sum;
  }
  if (lane == 0) *tie_t = any_near ? 1 : 0;
}

template <int NV>
__global__ void __launch_bounds__(256) k_topk(const float *__restrict__ logits, int32_t *idx,
                                              float *w, uint8_t *tie, int T, int E, int k) {
  const int t = (int)(((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if (t >= T) return;
  topk_warp<NV>(logits + (size_t)t * E, E, k, idx + (size_t)t * k, w + (size_t)t * k, tie + t);
}

template <typename F>
void dispatch_nv(int E, F &&f) {
  if (E <= 32) f(std::integral_constant<int, 1>{});
  else if (E <= 64) f(std::integral_constant<int, 2>{});
  else if (E <= 128) f(std::integral_constant<int, 4>{});
  else if (E <= 256) f(std::integral_constant<int, 8>{});
  else if (E <= 512) f(std::integral_constant<int, 16>{});
  else f(std::integral_constant<int, 32>{});
}

void launch_topk(const float *logits, int32_t *idx, float *w, uint8_t *tie, int T, int E, int k,
                 cudaStream_t s) {
  const int threads = 256;
  const unsigned blocks = (unsigned)((T * 32 + threads - 1) / threads);
  dispatch_nv(E, [&](auto nv) {
    k_topk<decltype(nv)::value><<<blocks, threads, 0, s>>>(logits, idx, w, tie, T, E, k);
  });
}

// ---------------------------------------------------------------------------------------
// Block-wide scan helpers (blockDim.x == 1024).
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ int block_incl_scan(int v, int *s_warp, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  if (lane == 31) s_warp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int wv = s_warp[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, wv, off);
      if (lane >= off) wv += o;
    }
    s_warp[lane] = wv;
  }
  __syncthreads();
  if (warp > 0) v += s_warp[warp - 1];
  *total = s_warp[31];
  __syncthreads();
  return v;
}

// ---------------------------------------------------------------------------------------
// Multi-CTA grouping for large P: per-chunk histograms, a per-expert scan over chunks,
// and a stable scatter (rank inside a warp by __match_any_sync, across the chunk's warps
// by per-warp histograms).  Chunk = 256 pairs.
// ---------------------------------------------------------------------------------------
constexpr int kChunk = 256;

size_t perm_multi_scratch_ints(int P, int E) {
  return (size_t)((P + kChunk - 1) / kChunk) * E;
}

__global__ void __launch_bounds__(kChunk) k_perm_hist(const int32_t *__restrict__ idx,
                                                      int32_t *chunk_hist, int P, int E,
                                                      DevCounters *ctr) {
  __shared__ int h[kMaxE];
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  __syncthreads();
  const int p = blockIdx.x * kChunk + threadIdx.x;
  if (p < P) {
    const int e = idx[p];
    if (e >= 0 && e < E)
      atomicAdd(&h[e], 1);
    else
      set_status(ctr, FT_ERR_INVALID);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_hist[(size_t)blockIdx.x * E + e] = h[e];
}

__global__ void __launch_bounds__(1024) k_perm_scan(int32_t *chunk_hist, int n_chunks, int E,
                                                    int P, int32_t *counts, int32_t *offsets) {
  __shared__ int s_warp[32];
  const int e = threadIdx.x;
  int running = 0;
  if (e < E) {
    for (int c = 0; c < n_chunks; ++c) {
      int *p = &chunk_hist[(size_t)c * E + e];
      const int v = *p;
      *p = running;
      running += v;
    }
  }
  int total;
  const int v = (e < E) ? running : 0;
  const int incl = block_incl_scan(v, s_warp, &total);
  const int off = incl - v;
  if (e < E) {
    counts[e] = running;
    offsets[e] = off;
    for (int c = 0; c < n_chunks; ++c) chunk_hist[(size_t)c * E + e] += off;
  }
  if (e == 0) offsets[E] = P;
}

__global__ void __launch_bounds__(kChunk) k_perm_scatter(const int32_t *__restrict__ idx,
                                                         const float *__restrict__ w,
                                                         const int32_t *__restrict__ chunk_base,
                                                         int P, int E, int k, int32_t *perm,
                                                         int32_t *inv, int32_t *tok, float *wq) {
  extern __shared__ int whist[];  // [kChunk/32][E]
  const int nw = kChunk / 32;
  for (int i = threadIdx.x; i < nw * E; i += blockDim.x) whist[i] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int p = blockIdx.x * kChunk + threadIdx.x;
  const bool valid = p < P;
  int e = valid ? idx[p] : -1;
  if (e >= E) e = -1;
  const unsigned act = __ballot_sync(0xffffffffu, e >= 0);
  unsigned mask = 0;
  int rank = 0;
  if (e >= 0) {
    mask = __match_any_sync(act, e);
    rank = __popc(mask & ((1u << lane) - 1u));
    if (rank == 0) whist[warp * E + e] = __popc(mask);
  }
  __syncthreads();
  if (e >= 0) {
    int base = chunk_base[(size_t)blockIdx.x * E + e];
    for (int w2 = 0; w2 < warp; ++w2) base += whist[w2 * E + e];
    const int pos = base + rank;
    perm[pos] = p;
    inv[p] = pos;
    tok[pos] = p / k;
    wq[pos] = w[p];
  }
}

void launch_perm_multi(const ControlArgs &a, int32_t *chunk_scratch, cudaStream_t s) {
  const int n_chunks = (a.P + kChunk - 1) / kChunk;
  if (n_chunks == 0) return;
  k_perm_hist<<<n_chunks, kChunk, 0, s>>>(a.idx, chunk_scratch, a.P, a.E, a.ctr);
  k_perm_scan<<<1, 1024, 0, s>>>(chunk_scratch, n_chunks, a.E, a.P, a.counts, a.offsets);
  const size_t smem = (size_t)(kChunk / 32) * a.E * sizeof(int);
  k_perm_scatter<<<n_chunks, kChunk, smem, s>>>(a.idx, a.w, chunk_scratch, a.P, a.E, a.k, a.perm,
                                                a.inv, a.tok, a.wq);
}

// ---------------------------------------------------------------------------------------
// Control: one CTA of 1024 threads.
//   1. counts, offsets and the stable grouping of the P = T*k pairs by expert (from the
//      pairs the in-CTA top-k left in shared memory, from idx in global memory, or, when
//      perm_ready, as a multi-CTA pass left them);
//   2. decode: the LRU update.  Touched set S = experts with count > 0.  Hits (ascending e)
//      get stamps tick0+1.., misses (ascending e) take the lowest free slots, then the
//      eligible slots (stamp <= tick0) in increasing (stamp, slot) order, and get stamps
//      after the hits'; every miss is appended to the fill list.  |S| > n_slots sets
//      FT_ERR_CAPACITY and leaves the cache and the outputs untouched.
//      prefill: expert e reads entry e of the layer's double buffer.
//      With admission counts (a.freq), every touched key's count grows by one and all counts
//      are halved once 10 * n_slots accesses have accumulated; a miss that finds no free
//      slot takes the next victim only if its count is >= the victim's, else it is staged
//      for this call in entry n_slots + b and the cache does not change.
//   3. the work list (touched experts ascending, then the shared expert) and counters.
// Threads leave data-dependent loops at different times; every block barrier that may
// follow such a loop is preceded by __syncwarp() (cta_sync), so warps reach it converged.
// ---------------------------------------------------------------------------------------
constexpr int kStampSmem = 2048;                     // slots whose keys fit in shared memory
constexpr int kSlotBits = 21;                        // slot id bits of a packed victim key
constexpr int kFewVictims = 4;                       // victims found by repeated minima
constexpr int kPairSmem = kGemvMaxTokens * kMaxK;    // pairs of the in-CTA top-k
constexpr int kFieldBits = 21;                       // packed per-expert scan fields
constexpr unsigned long long kFieldMask = (1ull << kFieldBits) - 1;

enum {
  kMiscNear = 0, kMiscDigit, kMiscNeed, kMiscCand, kMiscErr,
  kMiscHalve, kMiscAdmit, kMiscEvict, kMiscBypass, kMiscBad, kMiscN
};

struct CtlSmem {
  int cnt[kMaxE];
  int off[kMaxE + 1];
  int slot[kMaxE];  // grouping: running base per expert; LRU: slot taken by miss rank m
  int cand[kMaxE];  // eviction candidates below the threshold key
  int hist[2][256];
  unsigned long long wsum[32];
  unsigned long long tick0;  // the LRU clock at the start of the call (read by thread 0)
  int occupied0;             // occupied slots at the start of the call (read by thread 0)
  int misc[kMiscN];
  int pe[kPairSmem];    // expert of pair p (in-CTA top-k)
  float pv[kPairSmem];  // its logit
  float pw[kPairSmem];  // its gate
  union alignas(16) {
    unsigned long long key[kStampSmem];
    struct {              // admission decisions, by miss rank m / victim rank j
      unsigned mf[kMaxE];   // count of miss m
      unsigned vf[kMaxE];   // count of victim j's key
      int dest[kMaxE];      // slot, or staging entry n_slots + b
      int rank[kMaxE];      // stamp rank among admitted misses, -1 = bypassed
    } adm;
  } u;
};

__device__ __forceinline__ void cta_sync() {
  __syncwarp();
  __syncthreads();
}

// Inclusive scan over the 1024 threads of the CTA; *total = sum over all threads.
__device__ __forceinline__ unsigned long long cta_scan_u64(unsigned long long v,
                                                           unsigned long long *wsum,
                                                           unsigned long long *total) {
  __syncwarp();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned long long o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  if (lane == 31) wsum[warp] = v;
  cta_sync();
  if (warp == 0) {
    unsigned long long wv = wsum[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const unsigned long long o = __shfl_up_sync(0xffffffffu, wv, off);
      if (lane >= off) wv += o;
    }
    wsum[lane] = wv;
  }
  cta_sync();
  if (warp > 0) v += wsum[warp - 1];
  *total = wsum[31];
  cta_sync();
  return v;
}

// Warp of token t, lane j < k holding the j-th selected expert sel_i and logit sel_v (lanes
// >= k: anything), next_v the (k+1)-th logit (-inf if none): gates w_j = exp(l_j - l_0) /
// sum_i exp(l_i - l_0), near-tie when two adjacent selected logits, or the k-th and
// (k+1)-th, differ by <= kNearTie (in double); pairs t*k + j into sm.pe / pv / pw and idx,
// w, tie.
__device__ __forceinline__ void gates_and_ties(const ControlArgs &a, CtlSmem &sm, int t, int lane,
                                               int sel_i, float sel_v, float next_v) {
  const int k = a.k, E = a.E;
  const float l0 = __shfl_sync(0xffffffffu, sel_v, 0);
  const float ex = (lane < k) ? expf(sel_v - l0) : 0.f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  const float nxt_sel = __shfl_down_sync(0xffffffffu, sel_v, 1);
  bool near = false;
  if (lane + 1 < k) near = ((double)sel_v - (double)nxt_sel) <= kNearTie;
  if (lane == k - 1 && k < E) near = near || ((double)sel_v - (double)next_v) <= kNearTie;
  const bool any_near = __any_sync(0xffffffffu, near);
  if (lane < k) {
    const float w = ex / sum;
    sm.pe[t * k + lane] = sel_i;
    sm.pv[t * k + lane] = sel_v;
    sm.pw[t * k + lane] = w;
    const_cast<int32_t *>(a.idx)[t * k + lane] = sel_i;
    const_cast<float *>(a.w)[t * k + lane] = w;
  }
  if (lane == 0) {
    const_cast<uint8_t *>(a.tie)[t] = any_near ? 1 : 0;
    if (any_near) atomicAdd(&sm.misc[kMiscNear], 1);
  }
}

// Top-k of T <= kGemvMaxTokens tokens inside the CTA, one warp per token: k+1 rounds of a
// warp argmax under (logit descending, expert id ascending) over the token's logits (NV per
// lane), the (k+1)-th only for the near-tie report.  Gates w_j = exp(l_j - l_0) / sum_i
// exp(l_i - l_0); near-tie when two adjacent selected logits, or the k-th and (k+1)-th,
// differ by <= kNearTie (in double).  Leaves pair p = t*k + j in sm.pe / sm.pv / sm.pw (an
// expert no round selects - all remaining logits NaN - stays -1: an invalid pair) and writes
// idx, w and tie.  O(T k E) work, against O(T E^2) for ranking every (t, e) by counting.
template <int NV>
__device__ __forceinline__ void topk_warps(const ControlArgs &a, const float *logits, CtlSmem &sm) {
  const int T = a.T, E = a.E, k = a.k, tid = threadIdx.x;
  const int lane = tid & 31, t = tid >> 5;
  for (int p = tid; p < T * k; p += 1024) {
    sm.pe[p] = -1;
    sm.pv[p] = 0.f;
    sm.pw[p] = 0.f;
  }
  cta_sync();
  if (t < T) {
    const float *row = logits + (size_t)t * E;
    float v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      v[i] = (e < E) ? __ldcg(row + e) : -INFINITY;
    }
    uint32_t taken = 0;  // bit i: expert lane+32i already selected
    float sel_v = 0.f;   // lane j keeps the j-th selected logit
    int sel_i = -1;
    float next_v = -INFINITY;
    const int rounds = (k < E) ? k + 1 : k;
    for (int r = 0; r < rounds; ++r) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && better(v[i], e, bv, bi)) {
          bv = v[i];
          bi = e;
        }
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (better(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if (r < k) {
        if (bi < E && (bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == r) {
          sel_v = bv;
          sel_i = bi < E ? bi : -1;
        }
      } else {
        next_v = bv;
      }
    }
    gates_and_ties(a, sm, t, lane, sel_i, sel_v, next_v);
  }
}


// The same top-k by ranking, for small T*E^2: each (t, e) counts the logits of token t that
// come before it under (logit descending, expert id ascending); rank j < k puts e at pair
// t*k + j and rank k is the (k+1)-th logit of the near-tie report.  A NaN logit is never
// ranked, and never counts as coming before another (in the argmax rounds a NaN never wins),
// so every selection matches the rounds'.  O(T E^2) work over the whole CTA: cheaper than
// k+1 dependent warp reductions when T*E^2 <= kRankWork.
constexpr int kRankWork = 1 << 16;
constexpr int kRankSmem = kStampSmem * 2;  // floats of the logits staged in sm.u.key
// Stage the logits and clear the pairs; the caller's next block barrier orders this before
// topk_rank (so the loads overlap the rest of the control prologue).
__device__ __forceinline__ void topk_rank_stage(const ControlArgs &a, const float *logits,
                                                CtlSmem &sm) {
  const int T = a.T, E = a.E, k = a.k, tid = threadIdx.x;
  float *lg = reinterpret_cast<float *>(sm.u.key);
  float *nxt = reinterpret_cast<float *>(&sm.hist[0][0]);
  for (int i = tid; i < T * E; i += 1024) lg[i] = __ldcg(logits + i);
  for (int p = tid; p < T * k; p += 1024) {
    sm.pe[p] = -1;
    sm.pv[p] = -INFINITY;
    sm.pw[p] = 0.f;
  }
  if (tid < T) nxt[tid] = -INFINITY;
}
__device__ __forceinline__ bool use_topk_rank(const ControlArgs &a) {
  return a.T * a.E * a.E <= kRankWork && a.T * a.E <= kRankSmem;
}
__device__ __forceinline__ void topk_rank(const ControlArgs &a, CtlSmem &sm) {
  const int T = a.T, E = a.E, k = a.k, tid = threadIdx.x, lane = tid & 31;
  const float *lg = reinterpret_cast<const float *>(sm.u.key);
  float *nxt = reinterpret_cast<float *>(&sm.hist[0][0]);
  auto place = [&](int t, int e, float v, int r) {
    if (r < k) {
      sm.pe[t * k + r] = e;
      sm.pv[t * k + r] = v;
    } else if (r == k) {
      nxt[t] = v;
    }
  };
  const int pairs = T * E;
  for (int i = tid; i < pairs; i += 1024) {
    const int t = i / E, e = i - t * E;
    const float v = lg[i];
    if (!(v == v)) continue;
    const float *row = lg + t * E;
    int r = 0;
    if ((E & 3) == 0) {
      // four independent counts over 16-byte rows (row t starts at a multiple of 16 bytes)
      int r1 = 0, r2 = 0, r3 = 0;
#pragma unroll 4
      for (int j = 0; j < E; j += 4) {
        const float4 u = *reinterpret_cast<const float4 *>(row + j);
        r += (u.x > v || (u.x == v && j < e)) ? 1 : 0;
        r1 += (u.y > v || (u.y == v && j + 1 < e)) ? 1 : 0;
        r2 += (u.z > v || (u.z == v && j + 2 < e)) ? 1 : 0;
        r3 += (u.w > v || (u.w == v && j + 3 < e)) ? 1 : 0;
      }
      r += r1 + r2 + r3;
    } else {
#pragma unroll 8
      for (int j = 0; j < E; ++j) {
        const float u = row[j];
        r += (u > v || (u == v && j < e)) ? 1 : 0;
      }
    }
    place(t, e, v, r);
  }
  cta_sync();
  const int t = tid >> 5;
  if (t < T) {
    const int sel_i = lane < k ? sm.pe[t * k + lane] : -1;
    const float sel_v = lane < k ? sm.pv[t * k + lane] : 0.f;
    gates_and_ties(a, sm, t, lane, sel_i, sel_v, nxt[t]);
  }
}

// The nv smallest eviction keys (stamp of an occupied slot with stamp <= tick0; others are
// not eligible) in increasing (stamp, slot) order -> out[0 .. nv).  Up to kFewVictims of
// them (keys in shared memory, stamps below 2^43): nv rounds of a CTA minimum of the packed
// (stamp, slot) key, each taking its slot out.  Otherwise a radix select (8-bit digits from
// the top bit of tick0) finds the nv-th smallest stamp v*; the slots with a smaller stamp
// are ranked among themselves, the ones at v* follow in slot order.  Returns false if fewer
// than nv slots are eligible (out is then left in an unspecified state).
__device__ bool select_victims(const CacheDesc &cd, unsigned long long tick0, int nv, int *out,
                               CtlSmem &sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = cd.n_slots;
  const bool in_smem = n <= kStampSmem;
  auto key_g = [&](int s) -> unsigned long long {
    const unsigned long long st = cd.stamps[s];
    return (cd.owner[s] >= 0 && st <= tick0) ? st : ~0ull;
  };
  auto key = [&](int s) -> unsigned long long { return in_smem ? sm.u.key[s] : key_g(s); };
  if (in_smem)
    for (int s = tid; s < n; s += 1024) sm.u.key[s] = key_g(s);
  for (int i = tid; i < 512; i += 1024) (&sm.hist[0][0])[i] = 0;
  if (tid == 0) {
    sm.misc[kMiscErr] = 0;
    sm.misc[kMiscCand] = 0;
  }
  cta_sync();
  if (in_smem && nv <= kFewVictims && tick0 < (1ull << (64 - kSlotBits))) {
    for (int j = 0; j < nv; ++j) {
      unsigned long long best = ~0ull;
      for (int s = tid; s < n; s += 1024) {
        const unsigned long long kk = sm.u.key[s];
        if (kk != ~0ull) best = min(best, (kk << kSlotBits) | (unsigned long long)s);
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) best = min(best, __shfl_xor_sync(0xffffffffu, best, off));
      if (lane == 0) sm.wsum[warp] = best;
      cta_sync();
      if (warp == 0) {
        best = sm.wsum[lane];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
          best = min(best, __shfl_xor_sync(0xffffffffu, best, off));
        if (lane == 0) {
          if (best == ~0ull) {
            sm.misc[kMiscErr] = 1;
          } else {
            const int s = (int)(best & ((1ull << kSlotBits) - 1));
            out[j] = s;
            sm.u.key[s] = ~0ull;
          }
        }
      }
      cta_sync();
      if (sm.misc[kMiscErr]) return false;
    }
    return true;
  }
  const int nbits = 64 - __clzll(tick0 | 1ull);
  unsigned long long prefix = 0;  // digits of v* fixed so far
  int need = nv;                  // rank of v* among the keys that match the prefix
  int buf = 0;
  for (int shift = ((nbits + 7) / 8 - 1) * 8; shift >= 0; shift -= 8, buf ^= 1) {
    int *hist = sm.hist[buf];
    for (int s = tid; s < n; s += 1024) {
      const unsigned long long kk = key(s);
      if (kk != ~0ull && ((kk >> shift) >> 8) == prefix) atomicAdd(&hist[(kk >> shift) & 255], 1);
    }
    cta_sync();
    if (warp == 0) {
      int c[8], local = 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        c[b] = hist[8 * lane + b];
        local += c[b];
      }
      int incl = local;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      const int excl = incl - local;
      if (excl < need && need <= incl) {
        int cum = excl;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          if (cum < need && need <= cum + c[b]) {
            sm.misc[kMiscDigit] = 8 * lane + b;
            sm.misc[kMiscNeed] = need - cum;
          }
          cum += c[b];
        }
      }
      if (lane == 31 && incl < need) sm.misc[kMiscErr] = 1;
      for (int b = lane; b < 256; b += 32) sm.hist[buf ^ 1][b] = 0;
    }
    cta_sync();
    if (sm.misc[kMiscErr]) return false;
    prefix = (prefix << 8) | (unsigned long long)sm.misc[kMiscDigit];
    need = sm.misc[kMiscNeed];
  }
  const unsigned long long vstar = prefix;
  // keys below v*: exactly nv - need of them
  for (int s = tid; s < n; s += 1024)
    if (key(s) < vstar) sm.cand[atomicAdd(&sm.misc[kMiscCand], 1)] = s;
  cta_sync();
  const int na = sm.misc[kMiscCand];
  for (int i = tid; i < na; i += 1024) {
    const int s = sm.cand[i];
    const unsigned long long kk = key(s);
    int r = 0;
    for (int i2 = 0; i2 < na; ++i2) {
      const int s2 = sm.cand[i2];
      const unsigned long long k2 = key(s2);
      r += (k2 < kk || (k2 == kk && s2 < s)) ? 1 : 0;
    }
    out[r] = s;
  }
  // keys equal to v*: the `need` lowest slot ids
  int base = 0;
  for (int c0 = 0; c0 < n && base < need; c0 += 1024) {
    const int s = c0 + tid;
    const bool f = s < n && key(s) == vstar;
    unsigned long long tot;
    const int r = (int)cta_scan_u64(f ? 1ull : 0ull, sm.wsum, &tot) - (f ? 1 : 0);
    if (f && base + r < need) out[na + base + r] = s;
    base += (int)tot;
  }
  cta_sync();
  return true;
}

// mode: 0 = pairs from idx in global memory (P <= kPermSingleMax), 1 = perm_ready (counts
// and offsets from a multi-CTA pass), 2 = in-CTA top-k from `logits` (fused decode).
template <int NV>
__device__ __forceinline__ void control_body(const ControlArgs &a, int mode,
                                             const float *logits) {
  __shared__ CtlSmem sm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E, P = a.P;
  const bool lru = a.slot_table != nullptr;
  int *table = lru ? a.slot_table + (size_t)a.layer * E : nullptr;
  const int cur = (lru && tid < E) ? table[tid] : -1;  // issued early, used after grouping
  if (tid == 0) {
    a.ctr->call_status = 0;
    // One read of the clock for the whole CTA, ordered before thread 0's update of it at the
    // end of the call by the barriers below.  (Every thread reading ctr->tick itself raced with
    // that update in calls without misses, which have no barrier in between.)
    if (lru) {
      sm.tick0 = a.ctr->tick;
      sm.occupied0 = a.ctr->occupied;
    }
  }
  if (tid < kMiscN) sm.misc[tid] = 0;
  // the decode expert kernel of the previous call has finished (this kernel waited for it):
  // its completion counters start again from zero
  for (int i = tid; i < a.n_sync; i += 1024) a.sync[i] = 0;
  for (int e = tid; e < E; e += 1024) sm.cnt[e] = 0;
  const bool rank_topk = mode == 2 && use_topk_rank(a);
  if (rank_topk) topk_rank_stage(a, logits, sm);
  cta_sync();

  // 1. counts (and, below, offsets and grouping)
  float my_w = 0.f;
  if (mode == 2) {
    if (rank_topk)
      topk_rank(a, sm);
    else
      topk_warps<NV>(a, logits, sm);
    cta_sync();
    my_w = tid < P ? sm.pw[tid] : 0.f;
    if (tid < P) {
      const int e = sm.pe[tid];
      if (e >= 0 && e < E)
        atomicAdd(&sm.cnt[e], 1);
      else
        atomicAdd(&sm.misc[kMiscBad], 1);
    }
  } else if (mode == 0) {
    for (int p = tid; p < P; p += 1024) {
      const int e = a.idx[p];
      if (e >= 0 && e < E)
        atomicAdd(&sm.cnt[e], 1);
      else
        atomicAdd(&sm.misc[kMiscBad], 1);
    }
  } else {
    for (int e = tid; e < E; e += 1024) sm.cnt[e] = a.counts[e];
    // the multi-CTA grouping skips invalid pairs: then its counts do not add up to P
    if (tid == 0 && a.offsets[E - 1] + a.counts[E - 1] != P) atomicAdd(&sm.misc[kMiscBad], 1);
  }
  cta_sync();
  // an invalid pair (non-finite logits leave experts unranked) refuses the call like a
  // capacity overflow: nothing downstream runs on a partial grouping
  if (sm.misc[kMiscBad]) {
    if (tid == 0) {
      set_status(a.ctr, FT_ERR_INVALID);
      a.ctr->call_status = FT_ERR_INVALID;
      a.ctr->n_work = 0;
      a.ctr->n_fill = 0;
    }
    return;
  }

  // one scan over experts: offsets (modes 0, 2), hit / touched rank, miss rank
  const int cnt = tid < E ? sm.cnt[tid] : 0;
  const bool touched = cnt > 0;
  const bool hit = lru ? (touched && cur >= 0) : touched;
  const bool miss = lru && touched && cur < 0;
  const unsigned long long pk = (mode == 1 ? 0ull : (unsigned long long)cnt) |
                                ((unsigned long long)hit << kFieldBits) |
                                ((unsigned long long)miss << (2 * kFieldBits));
  unsigned long long tot;
  const unsigned long long ex = cta_scan_u64(pk, sm.wsum, &tot) - pk;
  const int hrank = (int)((ex >> kFieldBits) & kFieldMask);
  const int mrank = (int)(ex >> (2 * kFieldBits));
  const int n_hit = (int)((tot >> kFieldBits) & kFieldMask);
  const int n_miss = (int)(tot >> (2 * kFieldBits));
  const int n_touched = n_hit + n_miss;
  // work list order: hits (ascending expert), then misses (ascending expert), then the
  // shared expert; miss m is item n_hit + m and fill m
  const int wrank = hit ? hrank : n_hit + mrank;
  if (mode == 1) {
    for (int e = tid; e <= E; e += 1024) sm.off[e] = a.offsets[e];
  } else {
    if (tid < E) {
      sm.off[tid] = (int)(ex & kFieldMask);
      sm.slot[tid] = (int)(ex & kFieldMask);
      a.counts[tid] = cnt;
      a.offsets[tid] = (int)(ex & kFieldMask);
    }
    if (tid == 0) {
      sm.off[E] = P;
      a.offsets[E] = P;
    }
  }
  cta_sync();

  // grouping: pair p goes to off[e] + #{p' < p with the same expert}
  if (mode == 2) {
    if (tid < P) {
      const int e = sm.pe[tid];
      int r = 0;
      for (int p2 = 0; p2 < tid; ++p2) r += (sm.pe[p2] == e) ? 1 : 0;
      const int pos = sm.off[e] + r;
      a.perm[pos] = tid;
      a.inv[tid] = pos;
      a.tok[pos] = tid / a.k;
      a.wq[pos] = my_w;
    }
  } else if (mode == 0) {
    // chunks of 1024 pairs; inside a chunk the warps go in order
    for (int pc = 0; pc < P; pc += 1024) {
      const int p = pc + tid;
      int e = (p < P) ? a.idx[p] : -1;
      if (e >= E) e = -1;
      const unsigned act = __ballot_sync(0xffffffffu, e >= 0);
      unsigned mask = 0;
      int rank = 0;
      if (e >= 0) {
        mask = __match_any_sync(act, e);
        rank = __popc(mask & ((1u << lane) - 1u));
      }
      const int nwarps = min(32, (P - pc + 31) / 32);
      for (int w2 = 0; w2 < nwarps; ++w2) {
        if (warp == w2 && e >= 0) {
          const int pos = sm.slot[e] + rank;
          a.perm[pos] = p;
          a.inv[p] = pos;
          a.tok[pos] = p / a.k;
          a.wq[pos] = a.w[p];
        }
        __syncwarp();
        if (warp == w2 && e >= 0 && rank == 0) sm.slot[e] += __popc(mask);
        cta_sync();
      }
    }
  }
  if (a.shared) {
    for (int t = tid; t < a.T; t += 1024) {
      a.tok[P + t] = t;
      a.wq[P + t] = 1.0f;
    }
  }
  // near-tie count of this call
  if (mode != 2 && warp == 0) {
    int nt = 0;
    for (int t = lane; t < a.T; t += 32) nt += a.tie[t] ? 1 : 0;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) nt += __shfl_xor_sync(0xffffffffu, nt, off);
    if (lane == 0) sm.misc[kMiscNear] = nt;
  }

  // 2. the LRU update
  int slot_of = -1;
  CacheDesc cd{};
  int nv = 0;
  if (lru) {
    cd = *a.cache;
    if (n_touched > cd.n_slots) {
      if (tid == 0) {
        set_status(a.ctr, FT_ERR_CAPACITY);
        a.ctr->call_status = FT_ERR_CAPACITY;
        a.ctr->n_work = 0;
        a.ctr->n_fill = 0;
      }
      return;
    }
    const unsigned long long tick0 = sm.tick0;
    if (a.freq) {
      if (touched) a.freq[(size_t)a.layer * E + tid] += 1u;
      if (tid == 0) {
        unsigned long long acc = a.ctr->acc + (unsigned long long)n_touched;
        const unsigned long long H = 10ull * (unsigned long long)cd.n_slots;
        sm.misc[kMiscHalve] = acc >= H ? 1 : 0;
        a.ctr->acc = acc >= H ? acc - H : acc;
      }
      cta_sync();
      if (sm.misc[kMiscHalve]) {
        for (int i = tid; i < a.L * E; i += 1024) a.freq[i] >>= 1;
        cta_sync();
      }
    }
    if (hit) {
      if (cur < cd.n_slots)
        cd.stamps[cur] = tick0 + 1 + (unsigned long long)hrank;
      else
        set_status(a.ctr, FT_ERR_INVALID);
    }
    int n_free = 0;
    int n_admit = n_miss, n_evict = 0, n_bypass = 0;
    bool decided = false;  // admission decisions in sm.u.adm
    if (n_miss > 0) {
      cta_sync();  // hit stamps written before eviction keys are read
      // the n_miss lowest free slots (none to look for once every slot is occupied)
      if (sm.occupied0 < cd.n_slots) {
        for (int b0 = 0; b0 < cd.n_slots && n_free < n_miss; b0 += 1024) {
          const int s = b0 + tid;
          const bool f = s < cd.n_slots && cd.owner[s] < 0;
          unsigned long long tf;
          const int r = (int)cta_scan_u64(f ? 1ull : 0ull, sm.wsum, &tf) - (f ? 1 : 0);
          if (f && n_free + r < n_miss) sm.slot[n_free + r] = s;
          n_free += (int)tf;
        }
        n_free = min(n_free, n_miss);
      }
      nv = n_miss - n_free;
      if (nv > 0 && !select_victims(cd, tick0, nv, sm.slot + n_free, sm)) {
        if (tid == 0) {
          set_status(a.ctr, FT_ERR_INVALID);
          a.ctr->call_status = FT_ERR_INVALID;
          a.ctr->n_work = 0;
          a.ctr->n_fill = 0;
        }
        return;
      }
      cta_sync();
      n_evict = nv;
      if (a.freq && nv > 0) {
        // misses in ascending expert id: a free slot while any is left, else the next victim
        // if the miss's count is at least the victim key's, else a staging entry
        if (miss) sm.u.adm.mf[mrank] = a.freq[(size_t)a.layer * E + tid];
        if (tid < nv) sm.u.adm.vf[tid] = a.freq[cd.owner[sm.slot[n_free + tid]]];
        cta_sync();
        if (tid == 0) {
          int j = 0, b = 0, r = 0;
          for (int m = 0; m < n_miss; ++m) {
            if (m < n_free) {
              sm.u.adm.dest[m] = sm.slot[m];
              sm.u.adm.rank[m] = r++;
            } else if (j < nv && sm.u.adm.mf[m] >= sm.u.adm.vf[j]) {
              sm.u.adm.dest[m] = sm.slot[n_free + j++];
              sm.u.adm.rank[m] = r++;
            } else {
              sm.u.adm.dest[m] = cd.n_slots + b++;
              sm.u.adm.rank[m] = -1;
            }
          }
          sm.misc[kMiscAdmit] = r;
          sm.misc[kMiscEvict] = j;
          sm.misc[kMiscBypass] = b;
        }
        cta_sync();
        n_admit = sm.misc[kMiscAdmit];
        n_evict = sm.misc[kMiscEvict];
        n_bypass = sm.misc[kMiscBypass];
        decided = true;
      }
    }
    if (miss) {
      const int m = mrank;
      const int slot = decided ? sm.u.adm.dest[m] : sm.slot[m];
      const int arank = decided ? sm.u.adm.rank[m] : m;
      if (arank >= 0) {
        if (m >= n_free) {
          const int ev = cd.owner[slot];
          if (ev >= 0 && ev < a.L * E) a.slot_table[ev] = -1;
        }
        cd.owner[slot] = a.layer * E + tid;
        table[tid] = slot;
        cd.stamps[slot] = tick0 + (unsigned long long)n_hit + 1ull + (unsigned long long)arank;
      }
      a.fills[3 * m + 0] = slot;
      a.fills[3 * m + 1] = a.layer;
      a.fills[3 * m + 2] = tid;
      slot_of = slot;
    } else if (hit) {
      slot_of = cur;
    }
    if (tid == 0) {
      a.ctr->tick = tick0 + (unsigned long long)(n_hit + n_admit);
      a.ctr->calls += 1;
      a.ctr->hits += (unsigned long long)n_hit;
      a.ctr->misses += (unsigned long long)n_miss;
      a.ctr->fill_bytes += (unsigned long long)n_miss * a.entry_elems * 2ull;
      a.ctr->evictions += (unsigned long long)n_evict;
      a.ctr->bypasses += (unsigned long long)n_bypass;
      a.ctr->n_fill = n_miss;
      a.ctr->occupied += n_admit - n_evict;
    }
  } else {
    slot_of = touched ? tid : -1;
    if (tid == 0) a.ctr->n_fill = 0;
  }

  // 3. work list and counters
  if (touched) {
    WorkItem wi;
    wi.W = (lru ? cd.slots : a.buffer) + (size_t)slot_of * a.entry_elems;
    wi.q0 = sm.off[tid];
    wi.count = cnt;
    wi.expert = tid;
    wi.slot = slot_of;
    a.work[wrank] = wi;
  }
  cta_sync();
  if (tid == 0) {
    int nw = n_touched;
    if (a.shared) {
      WorkItem wi;
      wi.W = a.shared;
      wi.q0 = P;
      wi.count = a.T;
      wi.expert = -1;
      wi.slot = -1;
      a.work[nw++] = wi;
    }
    a.ctr->n_work = nw;
    a.ctr->n_hit = n_hit;
    if (sm.misc[kMiscNear]) atomicAdd(&a.ctr->near_ties, (unsigned long long)sm.misc[kMiscNear]);
  }
}

__global__ void __launch_bounds__(1024) k_control(ControlArgs a, int perm_ready) {
  control_body<1>(a, perm_ready ? 1 : 0, nullptr);
}

// ---------------------------------------------------------------------------------------
// Decode routing in one launch (T <= kGemvMaxTokens).  The T*E router logits are one warp
// task each, spread over up to one CTA per SM (task = CTA + warp * grid, so a call with few
// logits uses one warp on each of many SMs: their loads run in parallel); the CTA that
// finishes last (atomic arrival counter, no waiting) runs the top-k of every token, one warp
// per token, and then the control body above.
// ---------------------------------------------------------------------------------------
template <int NV>
__global__ void __launch_bounds__(1024) k_route_decode(const uint16_t *__restrict__ x,
                                                       const uint16_t *__restrict__ wr,
                                                       const float *__restrict__ bias,
                                                       float *__restrict__ logits,
                                                       ControlArgs a) {
  pdl_trigger();
  const int T = a.T, E = a.E, d = a.d, nchunk = d >> 3;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n_tasks = T * E, G = gridDim.x;
  // The router weights change only through ft_moe_load_router (a copy, fully ordered):
  // stage this warp's rows in L2 while the previous kernel finishes.  x may be that
  // kernel's output and the bias a copy queued after it, so both are read after the wait.
  for (int task = blockIdx.x + warp * G; task < n_tasks; task += 32 * G) {
    const int e = task % E;
    for (int c = lane; c < nchunk; c += 32) prefetch_l2(wr + (size_t)e * d + (size_t)c * 8);
  }
  pdl_wait();
  for (int task = blockIdx.x + warp * G; task < n_tasks; task += 32 * G) {
    const int t = task / E, e = task - t * E;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)t * d);
    const uint4 *wrr = reinterpret_cast<const uint4 *>(wr + (size_t)e * d);
    float acc = 0.f;  // lane lam: chunks lam, lam+32, ... in order, features in order
#pragma unroll 8
    for (int c = lane; c < nchunk; c += 32) acc = dot8_seq(__ldg(xr + c), __ldg(wrr + c), acc);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc = acc + __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) logits[task] = bias ? acc + __ldg(bias + e) : acc;
  }
  // the last CTA to arrive continues
  __shared__ int s_last;
  __threadfence();
  cta_sync();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(&a.ctr->route_arrive, 1u);
    s_last = (prev == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (threadIdx.x == 0) a.ctr->route_arrive = 0;
  control_body<NV>(a, 2, logits);
}

static int route_sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

void launch_route_decode(const uint16_t *x, const uint16_t *wr, const float *bias, float *logits,
                         const ControlArgs &a, cudaStream_t s) {
  const int grid = std::max(1, std::min(a.T * a.E, route_sm_count()));
  dispatch_nv(a.E, [&](auto nv) {
    constexpr int NV = decltype(nv)::value;
    launch_pdl(k_route_decode<NV>, dim3(grid), dim3(1024), 0, s, x, wr, bias, logits, a);
  });
}

void launch_control(const ControlArgs &a, bool perm_ready, cudaStream_t s) {
  k_control<<<1, 1024, 0, s>>>(a, perm_ready ? 1 : 0);
}

}  // namespace ftm
