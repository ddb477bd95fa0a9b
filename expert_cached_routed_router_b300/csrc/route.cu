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
//   1. (unless perm_ready) counts, offsets and the stable grouping of the P pairs;
//   2. decode: the LRU update.  Touched set S = experts with count > 0.  Hits (ascending e)
//      get stamps tick0+1.., misses (ascending e) take the lowest free slots, then the
//      eligible slots (stamp <= tick0) in increasing (stamp, slot) order, and get stamps
//      after the hits'; every miss is appended to the fill list.  |S| > n_slots sets
//      FT_ERR_CAPACITY and leaves the cache and the outputs untouched.
//      prefill: expert e reads entry e of the layer's double buffer.
//   3. the work list (touched experts ascending, then the shared expert) and counters.
// ---------------------------------------------------------------------------------------
constexpr int kStampSmem = 2048;  // slots whose eviction keys are staged in shared memory

__device__ __forceinline__ void control_body(const ControlArgs &a, int perm_ready) {
  __shared__ int s_cnt[kMaxE];
  __shared__ int s_off[kMaxE + 1];
  __shared__ int s_base[kMaxE];
  __shared__ int s_list[kMaxE];    // free slots, in increasing slot order
  __shared__ int s_victim[kMaxE];  // victims, in increasing (stamp, slot) order
  __shared__ int s_warp[32];
  __shared__ unsigned long long s_key[kStampSmem];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E, P = a.P;
  int total;
  if (tid == 0) a.ctr->call_status = 0;

  if (!perm_ready) {
    for (int e = tid; e < E; e += 1024) s_cnt[e] = 0;
    __syncthreads();
    for (int p = tid; p < P; p += 1024) {
      const int e = a.idx[p];
      if (e >= 0 && e < E)
        atomicAdd(&s_cnt[e], 1);
      else
        set_status(a.ctr, FT_ERR_INVALID);
    }
    __syncthreads();
    {
      const int v = (tid < E) ? s_cnt[tid] : 0;
      const int incl = block_incl_scan(v, s_warp, &total);
      if (tid < E) {
        s_off[tid] = incl - v;
        s_base[tid] = incl - v;
      }
      if (tid == 0) s_off[E] = P;
    }
    __syncthreads();
    // stable scatter: chunks of 1024 pairs, the warps of a chunk in order
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
          const int pos = s_base[e] + rank;
          a.perm[pos] = p;
          a.inv[p] = pos;
          a.tok[pos] = p / a.k;
          a.wq[pos] = a.w[p];
        }
        __syncwarp();
        if (warp == w2 && e >= 0 && rank == 0) s_base[e] += __popc(mask);
        __syncthreads();
      }
    }
    for (int e = tid; e < E; e += 1024) a.counts[e] = s_cnt[e];
    for (int e = tid; e <= E; e += 1024) a.offsets[e] = s_off[e];
  } else {
    for (int e = tid; e < E; e += 1024) s_cnt[e] = a.counts[e];
    for (int e = tid; e <= E; e += 1024) s_off[e] = a.offsets[e];
  }
  __syncthreads();
  if (a.shared) {
    for (int t = tid; t < a.T; t += 1024) {
      a.tok[P + t] = t;
      a.wq[P + t] = 1.0f;
    }
  }

  // touched experts, ranked in ascending id
  const bool touched = tid < E && s_cnt[tid] > 0;
  const int trank = block_incl_scan(touched ? 1 : 0, s_warp, &total) - (touched ? 1 : 0);
  const int n_touched = total;

  // near-tie count of this call
  if (warp == 0) {
    int nt = 0;
    for (int t = lane; t < a.T; t += 32) nt += a.tie[t] ? 1 : 0;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) nt += __shfl_xor_sync(0xffffffffu, nt, off);
    if (lane == 0 && nt) atomicAdd(&a.ctr->near_ties, (unsigned long long)nt);
  }

  int slot_of = -1;
  CacheDesc cd{};
  if (a.slot_table) cd = *a.cache;
  if (a.slot_table) {
    if (n_touched > cd.n_slots) {
      if (tid == 0) {
        set_status(a.ctr, FT_ERR_CAPACITY);
        a.ctr->call_status = FT_ERR_CAPACITY;
        a.ctr->n_work = 0;
        a.ctr->n_fill = 0;
      }
      return;
    }
    const unsigned long long tick0 = a.ctr->tick;
    int *table = a.slot_table + (size_t)a.layer * E;
    const int cur = touched ? table[tid] : -1;
    const bool hit = touched && cur >= 0;
    const bool miss = touched && cur < 0;
    const int hrank = block_incl_scan(hit ? 1 : 0, s_warp, &total) - (hit ? 1 : 0);
    const int n_hit = total;
    const int mrank = block_incl_scan(miss ? 1 : 0, s_warp, &total) - (miss ? 1 : 0);
    const int n_miss = total;
    if (hit) {
      if (cur < cd.n_slots)
        cd.stamps[cur] = tick0 + 1 + (unsigned long long)hrank;
      else
        set_status(a.ctr, FT_ERR_INVALID);
    }
    // the n_miss lowest free slots
    int n_free = 0;
    for (int base = 0; base < cd.n_slots; base += 1024) {
      const int s = base + tid;
      const bool f = s < cd.n_slots && cd.owner[s] < 0;
      const int r = block_incl_scan(f ? 1 : 0, s_warp, &total) - (f ? 1 : 0);
      if (f && n_free + r < n_miss) s_list[n_free + r] = s;
      n_free += total;
      if (n_free >= n_miss) break;
    }
    const int nv = n_miss > n_free ? n_miss - n_free : 0;
    if (nv > 0) {
      // eviction keys: (stamp, slot) of occupied slots not touched in this call
      const bool in_smem = cd.n_slots <= kStampSmem;
      if (in_smem) {
        for (int s = tid; s < cd.n_slots; s += 1024) {
          const unsigned long long st = cd.stamps[s];
          s_key[s] = (cd.owner[s] >= 0 && st <= tick0) ? st : ~0ull;
        }
      }
      __syncthreads();
      for (int s = tid; s < cd.n_slots; s += 1024) {
        const unsigned long long ks =
            in_smem ? s_key[s] : ((cd.owner[s] >= 0 && cd.stamps[s] <= tick0) ? cd.stamps[s] : ~0ull);
        if (ks == ~0ull) continue;
        int rank = 0;
        for (int s2 = 0; s2 < cd.n_slots && rank < nv; ++s2) {
          const unsigned long long k2 =
              in_smem ? s_key[s2]
                      : ((cd.owner[s2] >= 0 && cd.stamps[s2] <= tick0) ? cd.stamps[s2] : ~0ull);
          rank += (k2 < ks || (k2 == ks && s2 < s)) ? 1 : 0;
        }
        if (rank < nv) s_victim[rank] = s;
      }
    }
    __syncthreads();
    if (miss) {
      const int m = mrank;
      const int slot = (m < n_free) ? s_list[m] : s_victim[m - n_free];
      if (m >= n_free) {
        const int ev = cd.owner[slot];
        if (ev >= 0 && ev < a.L * E) a.slot_table[ev] = -1;
      }
      cd.owner[slot] = a.layer * E + tid;
      table[tid] = slot;
      cd.stamps[slot] = tick0 + (unsigned long long)n_hit + 1ull + (unsigned long long)m;
      a.fills[3 * m + 0] = slot;
      a.fills[3 * m + 1] = a.layer;
      a.fills[3 * m + 2] = tid;
      slot_of = slot;
    } else if (hit) {
      slot_of = cur;
    }
    if (tid == 0) {
      a.ctr->tick = tick0 + (unsigned long long)(n_hit + n_miss);
      a.ctr->calls += 1;
      a.ctr->hits += (unsigned long long)n_hit;
      a.ctr->misses += (unsigned long long)n_miss;
      a.ctr->fill_bytes += (unsigned long long)n_miss * a.entry_elems * 2ull;
      a.ctr->evictions += (unsigned long long)nv;
      a.ctr->n_fill = n_miss;
      a.ctr->occupied += n_miss - nv;
    }
  } else {
    slot_of = touched ? tid : -1;
    if (tid == 0) a.ctr->n_fill = 0;
  }
  if (touched) {
    WorkItem wi;
    wi.W = (a.slot_table ? cd.slots : a.buffer) + (size_t)slot_of * a.entry_elems;
    wi.q0 = s_off[tid];
    wi.count = s_cnt[tid];
    wi.expert = tid;
    wi.slot = slot_of;
    a.work[trank] = wi;
  }
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
  }
}

__global__ void __launch_bounds__(1024) k_control(ControlArgs a, int perm_ready) {
  control_body(a, perm_ready);
}

// ---------------------------------------------------------------------------------------
// Decode routing in one launch (T <= kGemvMaxTokens): every CTA computes a block of router
// logits; the CTA that finishes last (atomic arrival counter, no waiting) runs the top-k of
// all T tokens, one warp per token, and then the control body above.
// ---------------------------------------------------------------------------------------
template <int TT, int EE, int NV>
__global__ void __launch_bounds__(1024) k_route_decode(const uint16_t *__restrict__ x,
                                                       const uint16_t *__restrict__ wr,
                                                       const float *__restrict__ bias,
                                                       float *__restrict__ logits,
                                                       ControlArgs a) {
  pdl_trigger();
  const int T = a.T, E = a.E;
  const int lane = threadIdx.x & 31;
  const int n_eb = (E + EE - 1) / EE;
  const int n_tasks = ((T + TT - 1) / TT) * n_eb;
  const int task = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if (task < n_tasks) {
    const int tb = task / n_eb, eb = task - tb * n_eb;
    const int t0 = tb * TT, e0 = eb * EE;
    float acc[TT][EE];
#pragma unroll
    for (int i = 0; i < TT; ++i)
#pragma unroll
      for (int j = 0; j < EE; ++j) acc[i][j] = 0.f;
    const int d = a.d, nchunk = d >> 3;
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
        for (int j = 0; j < EE; ++j)
          acc[i][j] = acc[i][j] + __shfl_xor_sync(0xffffffffu, acc[i][j], off);
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
  // the previous kernel (which reads the routing state this launch rewrites) must be done
  pdl_wait();
  // the last CTA to arrive continues
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(&a.ctr->route_arrive, 1u);
    s_last = (prev == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int warp = threadIdx.x >> 5;
  for (int t = warp; t < T; t += 32)
    topk_warp<NV>(logits + (size_t)t * E, E, a.k, const_cast<int32_t *>(a.idx) + (size_t)t * a.k,
                  const_cast<float *>(a.w) + (size_t)t * a.k, const_cast<uint8_t *>(a.tie) + t);
  __syncthreads();
  if (threadIdx.x == 0) a.ctr->route_arrive = 0;
  control_body(a, 0);
}

void launch_route_decode(const uint16_t *x, const uint16_t *wr, const float *bias, float *logits,
                         const ControlArgs &a, cudaStream_t s) {
  dispatch_nv(a.E, [&](auto nv) {
    constexpr int NV = decltype(nv)::value;
    auto go = [&](auto kern, int tt, int ee) {
      const int tasks = ((a.T + tt - 1) / tt) * ((a.E + ee - 1) / ee);
      launch_pdl(kern, dim3((tasks + 31) / 32), dim3(1024), 0, s, x, wr, bias, logits, a);
    };
    if (a.T == 1)
      go(k_route_decode<1, 1, NV>, 1, 1);
    else if (a.T <= 2)
      go(k_route_decode<2, 2, NV>, 2, 2);
    else
      go(k_route_decode<4, 2, NV>, 4, 2);
  });
}

void launch_control(const ControlArgs &a, bool perm_ready, cudaStream_t s) {
  k_control<<<1, 1024, 0, s>>>(a, perm_ready ? 1 : 0);
}

}  // namespace ftm
