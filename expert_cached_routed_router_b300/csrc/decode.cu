// Decode expert path in one persistent launch per layer call (T <= kGemvMaxTokens): the miss
// fills from the host pool, gate/up + SwiGLU, down, and the gate-weighted combine.
//
// FreeToken benchmark, "how FreeToken serves large MoE models" (runtime-layer table): the host
// link moves missed experts into the GPU cache while the GPU executes the layer; FreeToken RTX
// 4090, "how the MoE memory hierarchy works": every expert runs from its complete (layer,
// expert) entry wherever the mapping says it lives.  On one B300 the decode layer is a batched
// GEMV over the touched entries, bound by HBM for cached entries and by the host link for
// missed ones, so the kernel overlaps the two: the hit experts stream from HBM while the misses
// cross the link, and each miss is computed as soon as its own fill has landed.
//
// One CTA per SM (all co-resident), three warp roles:
//   warps 0..7  consumers: dot weight rows held in a shared-memory ring with x (gate/up) or h
//               (down);
//   warp 8      producer: streams each task's weight rows into the ring with 1-D bulk (TMA)
//               copies, one stage per task, stage ownership as in Ring below;
//   warps 9..10 fill: copy the missed entries from the mapped pinned pool into their slots
//               (SM loads over the host link, 4 KB per warp per chunk).
// The tasks of a call form one list, in the order: gate/up of the resident items (hits and the
// shared expert), down of the resident items, gate/up of the missed items, down of the missed
// items.  Task g goes to CTA g mod gridDim.x, and a CTA takes its tasks in increasing g.  Every
// wait is for an earlier task of the list or for a fill, and fills wait for nothing, so with all
// CTAs resident the waits always end; they are still bounded (globaltimer, abort flag):
//   - a missed item's tasks wait (producer) until its whole entry is filled: fill_done[m];
//   - a down task waits (consumer) until its item's h is complete: gu_done[u] == gate/up tasks;
//   - the down task that completes a block of output rows (dn_done[block] == n_work) combines
//     that block for every token: out[t][i] = sum_j w[t][j] * y[row(t, j)][i], j ascending,
//     then + y[shared row of t][i]; a fixed order, so the output is deterministic.
// The counters are zeroed by the control CTA of the same call before this kernel starts.
// On a timeout the kernel records FT_ERR_TIMEOUT, stops issuing, waits (bounded) for its own
// copies in flight and returns.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <map>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace ftm {

constexpr int kConsumers = 8;
constexpr int kProducerWarp = kConsumers;
constexpr int kFillWarps = 2;
constexpr int kDecThreads = (kConsumers + 1 + kFillWarps) * 32;
constexpr int kMaxStagesPerWarp = 4;
constexpr uint32_t kDecRing = 192u << 10;  // all stages together (at most)
constexpr uint32_t kDecSmemMax = 224u << 10;
constexpr int kDownRows = 8;               // W_down rows per down task (at most)
constexpr int kFillLoads = 8;              // 16-byte loads in flight per lane
constexpr int kFillChunk = 32 * kFillLoads;  // uint4 per fill chunk (4 KB)

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// ---------------------------------------------------------------------------------------
// Bounded waits.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ int ld_acquire(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Order this thread's earlier generic-proxy accesses of global memory with its later
// async-proxy (bulk copy) accesses, and the other way round.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Spin (one thread) until *p >= target; false on abort or after limit_ns.
__device__ __noinline__ bool wait_count(const int *p, int target, uint64_t limit_ns,
                                        volatile int *abort) {
  if (ld_acquire(p) >= target) return true;
  const uint64_t t0 = globaltimer();
  for (long i = 0; i < (1L << 30); ++i) {
    __nanosleep(32);
    if (ld_acquire(p) >= target) return true;
    if ((i & 15) == 15 && (*abort || globaltimer() - t0 > limit_ns)) return false;
  }
  return false;
}

// mbarrier phase wait that also gives up on abort or after limit_ns.
__device__ __forceinline__ bool mbar_wait_abortable(uint64_t *bar, uint32_t parity,
                                                    uint64_t limit_ns, volatile int *abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (long i = 0; i < (1L << 30); ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 63 && (*abort || globaltimer() - t0 > limit_ns)) return false;
  }
  return false;
}

// ---------------------------------------------------------------------------------------
// The ring: consumer warp w owns stages w*spw .. w*spw+spw-1 and takes this CTA's tasks
// w, w+8, w+16, ...; its j-th task uses stage w*spw + (j % spw) for the (j / spw)-th time.
// A stage therefore has one consumer that waits on its phases strictly in order, so a parity
// wait can never match an older phase.
// ---------------------------------------------------------------------------------------
struct Ring {
  uint8_t *base;
  uint32_t stage_bytes;
  int spw;
  uint64_t *full;
  uint64_t *empty;
  __device__ __forceinline__ uint8_t *stage(int s) const { return base + (size_t)s * stage_bytes; }
  __device__ __forceinline__ int n() const { return spw * kConsumers; }
  __device__ __forceinline__ void slot_of(long it, int &s, long &use) const {
    const int w = (int)(it % kConsumers);
    const long j = it / kConsumers;
    s = w * spw + (int)(j % spw);
    use = j / spw;
  }
};

__host__ __device__ __forceinline__ int dec_spw(uint32_t ring_bytes, uint32_t stage_bytes) {
  int s = (int)(ring_bytes / (stage_bytes * kConsumers));
  return s < 1 ? 1 : (s > kMaxStagesPerWarp ? kMaxStagesPerWarp : s);
}

static size_t dec_smem_bytes(size_t x_bytes, uint32_t stage_bytes, uint32_t ring_bytes) {
  const int n = dec_spw(ring_bytes, stage_bytes) * kConsumers;
  return ((x_bytes + 127) & ~(size_t)127) + (size_t)n * stage_bytes + 2 * (size_t)n * 8 + 16;
}

// One task of the list.
struct Task {
  int down;  // 0 = gate/up rows, 1 = down rows
  int u;     // work item
  int blk;   // row block
  int miss;  // fill index of the item, or -1 for a resident item
};

struct TaskList {
  int n_hit, n_miss, n_res, n_jb, n_ib;
  long nA, nB, nC, n;
  __device__ __forceinline__ int res_item(int r) const { return r < n_hit ? r : n_hit + n_miss; }
  __device__ __forceinline__ Task at(long g) const {
    Task t;
    if (g < nA) {
      const int r = (int)(g / n_jb);
      t = {0, res_item(r), (int)(g - (long)r * n_jb), -1};
    } else if (g < nA + nB) {
      g -= nA;
      const int r = (int)(g / n_ib);
      t = {1, res_item(r), (int)(g - (long)r * n_ib), -1};
    } else if (g < nA + nB + nC) {
      g -= nA + nB;
      const int m = (int)(g / n_jb);
      t = {0, n_hit + m, (int)(g - (long)m * n_jb), m};
    } else {
      g -= nA + nB + nC;
      const int m = (int)(g / n_ib);
      t = {1, n_hit + m, (int)(g - (long)m * n_ib), m};
    }
    return t;
  }
};

// ---------------------------------------------------------------------------------------
// Consumer bodies, bf16 entries.
// ---------------------------------------------------------------------------------------

// G token rows against one gate row and one up row held in shared memory.
template <int G, bool XS>
__device__ __forceinline__ void gateup_dots(const uint4 *__restrict__ g, const uint4 *__restrict__ uu,
                                            const uint4 *__restrict__ xs, const int32_t *tk,
                                            int n, int nchunk, int lane, float (&ag)[G],
                                            float (&au)[G]) {
  int row[G];
#pragma unroll
  for (int t = 0; t < G; ++t) {
    ag[t] = au[t] = 0.f;
    row[t] = (t < n) ? tk[t] * nchunk : 0;
  }
  for (int ch = lane; ch < nchunk; ch += 32) {
    const uint4 gv = g[ch], uv = uu[ch];
#pragma unroll
    for (int t = 0; t < G; ++t) {
      if (t < n) {
        const uint4 xv = XS ? xs[row[t] + ch] : __ldg(xs + row[t] + ch);
        ag[t] = dot8_seq(gv, xv, ag[t]);
        au[t] = dot8_seq(uv, xv, au[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < G; ++t) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      ag[t] += __shfl_xor_sync(0xffffffffu, ag[t], off);
      au[t] += __shfl_xor_sync(0xffffffffu, au[t], off);
    }
  }
}

// h is written by other CTAs of this launch: read it through L2 (.cg), never the
// non-coherent path.
__device__ __forceinline__ uint4 ld_cg16(const void *p) {
  return __ldcg(reinterpret_cast<const uint4 *>(p));
}

// Up to kDownRows W_down rows (shared memory) against G rows of h.
template <int G>
__device__ __forceinline__ void down_dots(const uint8_t *__restrict__ st, int rows,
                                          const uint16_t *__restrict__ hq, int n, int d_ff,
                                          int nchunk, int lane, float (&part)[kDownRows][G]) {
#pragma unroll
  for (int r = 0; r < kDownRows; ++r)
#pragma unroll
    for (int t = 0; t < G; ++t) part[r][t] = 0.f;
  for (int ch = lane; ch < nchunk; ch += 32) {
    uint4 hv[G];
#pragma unroll
    for (int t = 0; t < G; ++t)
      hv[t] = (t < n) ? ld_cg16(hq + (size_t)t * d_ff + 8 * ch) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int r = 0; r < kDownRows; ++r) {
      if (r < rows) {
        const uint4 wv = reinterpret_cast<const uint4 *>(st + (size_t)r * d_ff * 2)[ch];
#pragma unroll
        for (int t = 0; t < G; ++t) part[r][t] = dot8_seq(wv, hv[t], part[r][t]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kDownRows; ++r)
#pragma unroll
    for (int t = 0; t < G; ++t)
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1)
        part[r][t] += __shfl_xor_sync(0xffffffffu, part[r][t], off);
}

// ---------------------------------------------------------------------------------------
// MXFP4 entries.  Codes Wg | Wu | Wd, then scales Wg | Wu | Wd; a row of K inputs has K/2 code
// bytes (input 2i in the low nibble of byte i) and K/32 scale bytes.  A 16-byte chunk of a
// row's codes is one 32-input scale block: the block's E2M1 values are dotted with the inputs,
// then the sum is multiplied by the block's power-of-two scale (exact).
// ---------------------------------------------------------------------------------------

__device__ __forceinline__ void decode8(uint32_t w, float (&v)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) v[e] = e2m1_f32(w >> (4 * e));
}

// acc + sum_e v[e] * x[e] over 8 bf16 inputs x (one uint4), in input order.
__device__ __forceinline__ float dot8_vals(const float (&v)[8], uint4 xv, float acc) {
  const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc = fmaf(v[2 * i], __uint_as_float(xw[i] << 16), acc);
    acc = fmaf(v[2 * i + 1], __uint_as_float(xw[i] & 0xFFFF0000u), acc);
  }
  return acc;
}

template <int G, bool XS>
__device__ __forceinline__ void gateup_dots_fp4(const uint4 *__restrict__ g,
                                                const uint4 *__restrict__ uu,
                                                const uint8_t *__restrict__ sg,
                                                const uint8_t *__restrict__ su,
                                                const uint4 *__restrict__ xs, const int32_t *tk,
                                                int n, int nchunk, int nblk, int lane,
                                                float (&ag)[G], float (&au)[G]) {
  int row[G];
#pragma unroll
  for (int t = 0; t < G; ++t) {
    ag[t] = au[t] = 0.f;
    row[t] = (t < n) ? tk[t] * nchunk : 0;
  }
  for (int ch = lane; ch < nblk; ch += 32) {
    const uint4 qg = g[ch], qu = uu[ch];
    const uint32_t wg[4] = {qg.x, qg.y, qg.z, qg.w}, wu[4] = {qu.x, qu.y, qu.z, qu.w};
    float bg[G], bu[G];
#pragma unroll
    for (int t = 0; t < G; ++t) bg[t] = bu[t] = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float vg[8], vu[8];
      decode8(wg[q], vg);
      decode8(wu[q], vu);
#pragma unroll
      for (int t = 0; t < G; ++t) {
        if (t < n) {
          const int xi = row[t] + 4 * ch + q;
          const uint4 xv = XS ? xs[xi] : __ldg(xs + xi);
          bg[t] = dot8_vals(vg, xv, bg[t]);
          bu[t] = dot8_vals(vu, xv, bu[t]);
        }
      }
    }
    const float scg = e8m0_f32(sg[ch]), scu = e8m0_f32(su[ch]);
#pragma unroll
    for (int t = 0; t < G; ++t) {
      ag[t] = fmaf(bg[t], scg, ag[t]);
      au[t] = fmaf(bu[t], scu, au[t]);
    }
  }
#pragma unroll
  for (int t = 0; t < G; ++t) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      ag[t] += __shfl_xor_sync(0xffffffffu, ag[t], off);
      au[t] += __shfl_xor_sync(0xffffffffu, au[t], off);
    }
  }
}

template <int G>
__device__ __forceinline__ void down_dots_fp4(const uint8_t *__restrict__ st, int R,
                                              const uint16_t *__restrict__ hq, int n, int d_ff,
                                              int lane, float (&part)[kDownRows][G]) {
  const int nblk = d_ff >> 5;
  const size_t cb = (size_t)d_ff / 2, sbr = (size_t)d_ff / 32;
#pragma unroll
  for (int r = 0; r < kDownRows; ++r)
#pragma unroll
    for (int t = 0; t < G; ++t) part[r][t] = 0.f;
  for (int ch = lane; ch < nblk; ch += 32) {
    uint4 hv[G][4];
#pragma unroll
    for (int t = 0; t < G; ++t)
#pragma unroll
      for (int q = 0; q < 4; ++q)
        hv[t][q] = (t < n) ? ld_cg16(hq + (size_t)t * d_ff + 32 * ch + 8 * q)
                           : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int r = 0; r < kDownRows; ++r) {
      if (r < R) {
        const uint4 qr = reinterpret_cast<const uint4 *>(st + r * cb)[ch];
        const uint32_t w[4] = {qr.x, qr.y, qr.z, qr.w};
        float b[G];
#pragma unroll
        for (int t = 0; t < G; ++t) b[t] = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float v[8];
          decode8(w[q], v);
#pragma unroll
          for (int t = 0; t < G; ++t) b[t] = dot8_vals(v, hv[t][q], b[t]);
        }
        const float sc = e8m0_f32(st[R * cb + r * sbr + ch]);
#pragma unroll
        for (int t = 0; t < G; ++t) part[r][t] = fmaf(b[t], sc, part[r][t]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kDownRows; ++r)
#pragma unroll
    for (int t = 0; t < G; ++t)
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1)
        part[r][t] += __shfl_xor_sync(0xffffffffu, part[r][t], off);
}

// ---------------------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------------------
template <bool FP4, bool XS>
__global__ void __launch_bounds__(kDecThreads, 1) k_decode_experts(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, d_ff = a.d_ff, T = a.T;
  const int nchunk = d >> 3;
  const size_t x_bytes = XS ? (size_t)T * d * 2 : 0;
  Ring r;
  r.base = smem + ((x_bytes + 127) & ~(size_t)127);
  r.stage_bytes = a.stage_bytes;
  r.spw = dec_spw(a.ring_bytes, a.stage_bytes);
  r.full = reinterpret_cast<uint64_t *>(r.base + (size_t)r.n() * a.stage_bytes);
  r.empty = r.full + r.n();
  volatile int *abort = reinterpret_cast<volatile int *>(r.empty + r.n());
  if (threadIdx.x == 0) {
    for (int s = 0; s < r.n(); ++s) {
      mbar_init(&r.full[s], 1);
      mbar_init(&r.empty[s], 1);
    }
    *abort = 0;
    fence_barrier_init();
  }
  // everything below reads what the control kernel of this call wrote (work list, fills,
  // zeroed counters), and x may be the previous call's output
  pdl_wait();
  if (XS)
    for (int i = threadIdx.x; i < T * nchunk; i += blockDim.x)
      reinterpret_cast<uint4 *>(smem)[i] = __ldg(reinterpret_cast<const uint4 *>(a.x) + i);
  __syncthreads();
  DevCounters *ctr = a.ctr;
  if (ctr->call_status != 0) return;
  const uint64_t limit = ctr->wait_ns;
  const int n_work = ctr->n_work, n_hit = ctr->n_hit, n_fill = ctr->n_fill;
  int *gu_done = a.sync;
  int *fill_done = a.sync + kMaxE + 1;
  int *dn_done = a.sync + 2 * kMaxE + 1;
  TaskList tl;
  tl.n_hit = n_hit;
  tl.n_miss = n_fill;
  tl.n_res = n_work - n_fill;
  tl.n_jb = (d_ff + a.R_gu - 1) / a.R_gu;
  tl.n_ib = (d + a.R_dn - 1) / a.R_dn;
  tl.nA = (long)tl.n_res * tl.n_jb;
  tl.nB = (long)tl.n_res * tl.n_ib;
  tl.nC = (long)tl.n_miss * tl.n_jb;
  tl.n = tl.nA + tl.nB + tl.nC + (long)tl.n_miss * tl.n_ib;
  const long fill_chunks = (long)((a.entry_bytes / 16 + kFillChunk - 1) / kFillChunk);

  if (warp > kProducerWarp) {
    // ------------------------------------------------------------ fill warps
    const int fw = blockIdx.x * kFillWarps + (warp - kProducerWarp - 1);
    const int n_fw = gridDim.x * kFillWarps;
    const int hold = ctr->hold_fills;
    const size_t ev = a.entry_bytes / 16;
    const CacheDesc *cd = a.cache;
    uint4 *slots = reinterpret_cast<uint4 *>(cd->slots);
    for (long c = fw; c < (long)n_fill * fill_chunks; c += n_fw) {
      const int m = (int)(c / fill_chunks);
      const long cc = c - (long)m * fill_chunks;
      const int dst_e = a.fills[3 * m], l = a.fills[3 * m + 1], e = a.fills[3 * m + 2];
      const uint4 *src = a.pool + ((size_t)l * a.E + e) * ev;
      uint4 *dst = slots + (size_t)dst_e * ev;
      const size_t i0 = (size_t)cc * kFillChunk + lane;
      uint4 v[kFillLoads];
#pragma unroll
      for (int u = 0; u < kFillLoads; ++u)
        if (i0 + 32 * u < ev) v[u] = src[i0 + 32 * u];
#pragma unroll
      for (int u = 0; u < kFillLoads; ++u)
        if (i0 + 32 * u < ev) dst[i0 + 32 * u] = v[u];
      // every lane orders its stores before the count, also for the bulk copies that read
      // the entry next
      fence_proxy_async_global();
      __threadfence();
      __syncwarp();
      if (lane == 0 && !hold) atomicAdd(&fill_done[m], 1);
    }
    return;
  }

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      long it = 0;
      int cu = -1, ready_m = -1;
      const uint8_t *W = nullptr;
      for (long g = blockIdx.x; g < tl.n; g += gridDim.x, ++it) {
        const Task t = tl.at(g);
        int s;
        long use;
        r.slot_of(it, s, use);
        if (use > 0 && !mbar_wait_abortable(&r.empty[s], (uint32_t)((use - 1) & 1), limit, abort)) {
          ok = false;
          break;
        }
        if (t.miss >= 0 && t.miss != ready_m) {
          if (!wait_count(&fill_done[t.miss], (int)fill_chunks, limit, abort)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
          ready_m = t.miss;
        }
        if (t.u != cu) {
          cu = t.u;
          W = reinterpret_cast<const uint8_t *>(a.work[t.u].W);
        }
        uint8_t *st = r.stage(s);
        uint64_t *bar = &r.full[s];
        if (!FP4) {
          if (!t.down) {
            const int j0 = t.blk * a.R_gu, rows = min(a.R_gu, d_ff - j0);
            const uint32_t bytes = (uint32_t)rows * d * 2;
            mbar_arrive_expect_tx(bar, 2 * bytes);
            bulk_g2s(st, W + (size_t)j0 * d * 2, bytes, bar);
            bulk_g2s(st + (size_t)a.R_gu * d * 2, W + (size_t)(d_ff + j0) * d * 2, bytes, bar);
          } else {
            const int i0 = t.blk * a.R_dn, rows = min(a.R_dn, d - i0);
            const uint32_t bytes = (uint32_t)rows * d_ff * 2;
            mbar_arrive_expect_tx(bar, bytes);
            bulk_g2s(st, W + ((size_t)2 * d_ff * d + (size_t)i0 * d_ff) * 2, bytes, bar);
          }
        } else {
          const size_t scale0 = (size_t)3 * d * d_ff / 2;  // start of the scale region
          if (!t.down) {
            const int j0 = t.blk * a.R_gu;
            const size_t cb = (size_t)d / 2, sbr = (size_t)d / 32;
            const uint32_t c_bytes = (uint32_t)(a.R_gu * cb), s_bytes = (uint32_t)(a.R_gu * sbr);
            mbar_arrive_expect_tx(bar, 2 * c_bytes + 2 * s_bytes);
            bulk_g2s(st, W + (size_t)j0 * cb, c_bytes, bar);
            bulk_g2s(st + c_bytes, W + (size_t)d_ff * cb + (size_t)j0 * cb, c_bytes, bar);
            bulk_g2s(st + 2 * c_bytes, W + scale0 + (size_t)j0 * sbr, s_bytes, bar);
            bulk_g2s(st + 2 * c_bytes + s_bytes, W + scale0 + (size_t)d_ff * sbr + (size_t)j0 * sbr,
                     s_bytes, bar);
          } else {
            const int i0 = t.blk * a.R_dn;
            const size_t cb = (size_t)d_ff / 2, sbr = (size_t)d_ff / 32;
            const size_t codes_d = (size_t)d * d_ff;
            const size_t scales_d = scale0 + (size_t)2 * d_ff * (d / 32);
            const uint32_t c_bytes = (uint32_t)(a.R_dn * cb), s_bytes = (uint32_t)(a.R_dn * sbr);
            mbar_arrive_expect_tx(bar, c_bytes + s_bytes);
            bulk_g2s(st, W + codes_d + (size_t)i0 * cb, c_bytes, bar);
            bulk_g2s(st + c_bytes, W + scales_d + (size_t)i0 * sbr, s_bytes, bar);
          }
        }
      }
      if (!ok) {
        *abort = 1;
        set_status(ctr, FT_ERR_TIMEOUT);
      }
      // drain: the copies of the last issued tasks (at most one in flight per stage)
      const long n = r.n();
      for (long i = (it > n ? it - n : 0); i < it; ++i) {
        int s;
        long use;
        r.slot_of(i, s, use);
        mbar_wait(&r.full[s], (uint32_t)(use & 1));
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const uint4 *xs = XS ? reinterpret_cast<const uint4 *>(smem) : reinterpret_cast<const uint4 *>(a.x);
  const int P = T * a.k;
  long it = 0;
  int cu = -1;
  WorkItem wi{};
  for (long g = blockIdx.x; g < tl.n; g += gridDim.x, ++it) {
    if ((int)(it % kConsumers) != warp) continue;
    const Task t = tl.at(g);
    int s;
    long use;
    r.slot_of(it, s, use);
    bool ok = true;
    if (lane == 0) ok = mbar_wait_abortable(&r.full[s], (uint32_t)(use & 1), limit, abort);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      if (lane == 0) {
        *abort = 1;
        set_status(ctr, FT_ERR_TIMEOUT);
      }
      return;
    }
    const uint8_t *st = r.stage(s);
    if (t.u != cu) {
      cu = t.u;
      wi = a.work[t.u];
    }
    const int c = wi.count;
    if (!t.down) {
      // gate/up + SwiGLU: h[q][j] = silu(g) * u for the item's rows q
      const int j0 = t.blk * a.R_gu;
      const int rows = FP4 ? a.R_gu : min(a.R_gu, d_ff - j0);
      for (int rr = 0; rr < rows; ++rr) {
        const uint4 *gr, *ur;
        const uint8_t *sg = nullptr, *su = nullptr;
        if (!FP4) {
          gr = reinterpret_cast<const uint4 *>(st + (size_t)rr * d * 2);
          ur = reinterpret_cast<const uint4 *>(st + (size_t)(a.R_gu + rr) * d * 2);
        } else {
          const size_t cb = (size_t)d / 2, sbr = (size_t)d / 32;
          gr = reinterpret_cast<const uint4 *>(st + rr * cb);
          ur = reinterpret_cast<const uint4 *>(st + (a.R_gu + rr) * cb);
          sg = st + 2 * a.R_gu * cb + rr * sbr;
          su = st + 2 * a.R_gu * cb + (a.R_gu + rr) * sbr;
        }
        for (int t0 = 0; t0 < c; t0 += 4) {
          const int n = min(4, c - t0);
          const int32_t *tk = a.tok + wi.q0 + t0;
          uint16_t *hq = a.h + (size_t)(wi.q0 + t0) * d_ff + j0 + rr;
          if (n == 1) {
            float ag[1], au[1];
            if (FP4)
              gateup_dots_fp4<1, XS>(gr, ur, sg, su, xs, tk, 1, nchunk, d >> 5, lane, ag, au);
            else
              gateup_dots<1, XS>(gr, ur, xs, tk, 1, nchunk, lane, ag, au);
            if (lane == 0) hq[0] = f32_to_bf16(silu_mul(ag[0], au[0]));
          } else {
            float ag[4], au[4];
            if (FP4)
              gateup_dots_fp4<4, XS>(gr, ur, sg, su, xs, tk, n, nchunk, d >> 5, lane, ag, au);
            else
              gateup_dots<4, XS>(gr, ur, xs, tk, n, nchunk, lane, ag, au);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              if (lane == q && q < n) hq[(size_t)q * d_ff] = f32_to_bf16(silu_mul(ag[q], au[q]));
          }
        }
      }
      __threadfence();  // every lane: its h stores before the count
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&r.empty[s]);
        atomicAdd(&gu_done[t.u], 1);
      }
    } else {
      // down: y[q][i] for the item's rows q, after the item's h is complete
      const int i0 = t.blk * a.R_dn;
      const int rows = FP4 ? a.R_dn : min(a.R_dn, d - i0);
      if (lane == 0) ok = wait_count(&gu_done[t.u], tl.n_jb, limit, abort);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) {
          *abort = 1;
          set_status(ctr, FT_ERR_TIMEOUT);
        }
        return;
      }
      (void)ld_acquire(&gu_done[t.u]);  // every lane orders its h reads after the count
      for (int t0 = 0; t0 < c; t0 += 4) {
        const int n = min(4, c - t0);
        const uint16_t *hq = a.h + (size_t)(wi.q0 + t0) * d_ff;
        float *yq = a.y + (size_t)(wi.q0 + t0) * d + i0;
        if (n == 1) {
          float part[kDownRows][1];
          if (FP4)
            down_dots_fp4<1>(st, a.R_dn, hq, 1, d_ff, lane, part);
          else
            down_dots<1>(st, rows, hq, 1, d_ff, d_ff >> 3, lane, part);
#pragma unroll
          for (int q = 0; q < kDownRows; ++q)
            if (lane == q && q < rows) yq[q] = part[q][0];
        } else {
          float part[kDownRows][4];
          if (FP4)
            down_dots_fp4<4>(st, a.R_dn, hq, n, d_ff, lane, part);
          else
            down_dots<4>(st, rows, hq, n, d_ff, d_ff >> 3, lane, part);
#pragma unroll
          for (int q = 0; q < kDownRows; ++q)
#pragma unroll
            for (int tt = 0; tt < 4; ++tt)
              if (lane == q * 4 + tt && q < rows && tt < n) yq[(size_t)tt * d + q] = part[q][tt];
        }
      }
      __threadfence();  // every lane: its y stores before the count
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        mbar_arrive(&r.empty[s]);
        last = atomicAdd(&dn_done[t.blk], 1) == n_work - 1;
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        // every item's rows of this block are in y: combine them for every token, in rank
        // order, then the shared expert
        (void)ld_acquire(&dn_done[t.blk]);
        const int k = a.k;
        for (int e = lane; e < T * rows; e += 32) {
          const int tt = e / rows, i = i0 + (e - tt * rows);
          float acc = 0.f;
          for (int j = 0; j < k; ++j)
            acc = fmaf(a.w[tt * k + j], __ldcg(a.y + (size_t)a.inv[tt * k + j] * d + i), acc);
          if (a.shared) acc += __ldcg(a.y + (size_t)(P + tt) * d + i);
          a.out[(size_t)tt * d + i] = f32_to_bf16(acc);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------------------
static int dec_sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

// Dynamic shared memory attribute, and a check that one CTA fits on an SM (the kernel's waits
// need every CTA of the grid resident at once: one per SM).
template <typename K>
static bool prepare_kernel(K kern, size_t smem) {
  static std::mutex mu;
  static std::map<const void *, size_t> done;
  std::lock_guard<std::mutex> lock(mu);
  size_t &v = done[reinterpret_cast<const void *>(kern)];
  if (smem > v) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return false;
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kern, kDecThreads, smem) !=
            cudaSuccess ||
        blocks < 1)
      return false;
    v = smem;
  }
  return true;
}

DecodePlan plan_decode(int T, int d, int d_ff, bool fp4) {
  DecodePlan p{};
  const size_t xb = (size_t)T * d * 2, xr = (xb + 127) & ~(size_t)127;
  if (!fp4) {
    const uint32_t unit_gu = 4u * d, unit_dn = 2u * d_ff;
    const uint32_t unit = std::max(unit_gu, unit_dn);
    p.xs = xr + (size_t)kConsumers * unit + 1024 <= kDecSmemMax;
    p.ring = p.xs ? (uint32_t)std::min<size_t>(kDecRing, kDecSmemMax - 1024 - xr) : kDecRing;
    p.R_gu = std::max(1, std::min({d_ff, 4, (int)(p.ring / kConsumers / unit_gu)}));
    const uint32_t sgu = (uint32_t)p.R_gu * unit_gu;
    p.R_dn = std::max(1, std::min({d, kDownRows, (int)(std::max(sgu, unit_dn) / unit_dn)}));
    p.stage = std::max(sgu, (uint32_t)p.R_dn * unit_dn);
  } else {
    const uint32_t unit_gu = (uint32_t)d * 17 / 16, unit_dn = (uint32_t)d_ff * 17 / 32;
    p.xs = xr + (size_t)kConsumers * 4 * unit_gu + 1024 <= kDecSmemMax;
    p.ring = p.xs ? (uint32_t)std::min<size_t>(kDecRing, kDecSmemMax - 1024 - xr) : kDecRing;
    p.R_gu = 4;
    for (int c : {16, 8})
      if (d_ff % c == 0 && (c * d) % 512 == 0 && (size_t)kConsumers * c * unit_gu <= p.ring) {
        p.R_gu = c;
        break;
      }
    p.R_dn = ((size_t)kConsumers * kDownRows * unit_dn <= p.ring) ? kDownRows : 4;
    p.stage = std::max((uint32_t)p.R_gu * unit_gu, (uint32_t)p.R_dn * unit_dn);
  }
  p.smem = dec_smem_bytes(p.xs ? xb : 0, p.stage, p.ring);
  p.n_ib = (d + p.R_dn - 1) / p.R_dn;
  return p;
}

int launch_decode_experts(DecodeArgs a, bool fp4, cudaStream_t s) {
  const DecodePlan p = plan_decode(a.T, a.d, a.d_ff, fp4);
  a.R_gu = p.R_gu;
  a.R_dn = p.R_dn;
  a.stage_bytes = p.stage;
  a.ring_bytes = p.ring;
  cudaError_t e = cudaSuccess;
  auto go = [&](auto kern) {
    if (!prepare_kernel(kern, p.smem)) {
      e = cudaErrorInvalidConfiguration;
      return;
    }
    e = launch_pdl(kern, dim3(dec_sm_count()), dim3(kDecThreads), p.smem, s, a);
  };
  if (fp4) {
    if (p.xs) go(k_decode_experts<true, true>); else go(k_decode_experts<true, false>);
  } else {
    if (p.xs) go(k_decode_experts<false, true>); else go(k_decode_experts<false, false>);
  }
  return e == cudaSuccess ? FT_OK : report_error(FT_ERR_CUDA, "decode expert kernel launch", e);
}

}  // namespace ftm
