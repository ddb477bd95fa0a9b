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
//               (SM loads over the host link, 16 KB per warp per chunk).
// The tasks of a call form one list, in the order: gate/up of the resident items (hits and the
// shared expert), down of the resident items, gate/up of the missed items, down of the missed
// items.  Task g goes to CTA g mod gridDim.x, and a CTA takes its tasks in increasing g.  The
// waits, all bounded (globaltimer, abort flag):
//   - a missed item's gate/up tasks wait (producer) until the gate/up rows of its entry are
//     filled (fill_done[m]), its down tasks until the rest is too (fill_dn[m]); the fill warps
//     copy the gate/up rows of every missed entry before any down rows, so the missed experts'
//     gate/up runs while their down rows still cross the host link (bf16 entries; an MXFP4
//     entry, whose scales follow all its codes, is one region);
//   - the down tasks of resident items wait (consumer) until every consumer warp of the grid
//     has finished its gate/up tasks of resident items (phase counter A), those of missed
//     items until every warp has finished its gate/up tasks of missed items (counter C);
//   - after its last task a warp counts itself in Y, and once every warp is counted each one
//     combines a slice of the output: out[t][i] = sum_j w[t][j] * y[row(t, j)][i], j
//     ascending, then + y[shared row of t][i]; a fixed order, so the output is deterministic.
// Every wait is for tasks earlier in the list or for a fill, fills wait for nothing, and a
// CTA's producer issues its tasks in list order, so with all CTAs resident the waits end.
// Each consumer warp fences its stores once per phase, not once per task.  The counters are
// zeroed by the control CTA of the same call before this kernel starts.
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
constexpr uint32_t kDecRing = 192u << 10;  // all stages together (at most)
constexpr uint32_t kDecSmemMax = 224u << 10;
constexpr int kDownRows = 8;               // W_down rows per down task (at most)
constexpr int kFillLoads = 32;             // 16-byte loads in flight per lane
constexpr int kFillChunk = 32 * kFillLoads;  // uint4 per fill chunk (16 KB)

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

// Spin (one thread) until *p >= target, backing off from 128 ns to 1 us between polls; false
// on abort or after limit_ns.
__device__ __noinline__ bool wait_count(const int *p, int target, uint64_t limit_ns,
                                        volatile int *abort) {
  if (ld_acquire(p) >= target) return true;
  const uint64_t t0 = globaltimer();
  unsigned ns = 128;
  for (long i = 0; i < (1L << 30); ++i) {
    __nanosleep(ns);
    if (ld_acquire(p) >= target) return true;
    ns = ns < 1024 ? 2 * ns : 1024;
    if ((i & 3) == 3 && (*abort || globaltimer() - t0 > limit_ns)) return false;
  }
  return false;
}

// Spin (one thread) until the shared-memory flag is set; false on abort or after limit_ns.
__device__ __noinline__ bool wait_smem_flag(volatile int *f, uint64_t limit_ns,
                                            volatile int *abort) {
  if (*f) return true;
  const uint64_t t0 = globaltimer();
  for (long i = 0; i < (1L << 30); ++i) {
    __nanosleep(64);
    if (*f) return true;
    if ((i & 15) == 15 && (*abort || globaltimer() - t0 > limit_ns)) return false;
  }
  return false;
}

// mbarrier phase wait that also gives up on abort or after limit_ns; polls sleep up to 1 us.
__device__ __forceinline__ bool mbar_wait_abortable(uint64_t *bar, uint32_t parity,
                                                    uint64_t limit_ns, volatile int *abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (long i = 0; i < (1L << 30); ++i) {
    if (mbar_try_wait_sleep(bar, parity, 1000)) return true;
    if ((i & 7) == 7 && (*abort || globaltimer() - t0 > limit_ns)) return false;
  }
  return false;
}

// ---------------------------------------------------------------------------------------
// The ring: n stages; the CTA's j-th task uses stage j % n for the (j / n)-th time.  Every
// consumer warp takes every task of its CTA, in order, and works on its own rows of the
// stage, so each stage's phases are waited for in order by all of them ("full", one arrival
// with the transaction bytes) and released by all of them ("empty", one arrival per consumer
// warp): a parity wait can never match an older phase.  Stages are large (about a third of
// the ring) because the bulk-copy throughput of an SM grows with the bytes per copy: 4 KB
// copies stream at a quarter of HBM bandwidth, 32 KB and larger ones at full bandwidth.
// ---------------------------------------------------------------------------------------
struct Ring {
  uint8_t *base;
  uint32_t stage_bytes;
  int n;
  uint64_t *full;
  uint64_t *empty;
  __device__ __forceinline__ uint8_t *stage(int s) const { return base + (size_t)s * stage_bytes; }
  __device__ __forceinline__ void slot_of(int it, int &s, int &use) const {
    s = it % n;
    use = it / n;
  }
};

// Shared memory: [x (XS) | work items | token of each FFN row | phase flags | stages |
// full / empty barriers | abort flag].
struct DecLayout {
  size_t items, tok, flags, ring;
};
__host__ __device__ __forceinline__ DecLayout dec_layout(size_t x_bytes, int max_items, int n_rows) {
  DecLayout l;
  l.items = (x_bytes + 127) & ~(size_t)127;
  l.tok = (l.items + (size_t)max_items * sizeof(WorkItem) + 15) & ~(size_t)15;
  l.flags = (l.tok + (size_t)n_rows * sizeof(int32_t) + 15) & ~(size_t)15;
  l.ring = (l.flags + 16 * sizeof(int) + 127) & ~(size_t)127;
  return l;
}
static size_t dec_smem_bytes(size_t x_bytes, int max_items, int n_rows, uint32_t stage_bytes,
                             int n_stages) {
  return dec_layout(x_bytes, max_items, n_rows).ring + (size_t)n_stages * stage_bytes +
         2 * (size_t)n_stages * 8 + 16;
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
  int nA, nB, nC, n;
  __device__ __forceinline__ int res_item(int r) const { return r < n_hit ? r : n_hit + n_miss; }
  __device__ __forceinline__ Task at(int g) const {
    Task t;
    if (g < nA) {
      const int r = g / n_jb;
      t = {0, res_item(r), g - r * n_jb, -1};
    } else if (g < nA + nB) {
      g -= nA;
      const int r = g / n_ib;
      t = {1, res_item(r), g - r * n_ib, -1};
    } else if (g < nA + nB + nC) {
      g -= nA + nB;
      const int m = g / n_jb;
      t = {0, n_hit + m, g - m * n_jb, m};
    } else {
      g -= nA + nB + nC;
      const int m = g / n_ib;
      t = {1, n_hit + m, g - m * n_ib, m};
    }
    return t;
  }
};

// ---------------------------------------------------------------------------------------
// Consumer bodies, bf16 entries.
// ---------------------------------------------------------------------------------------

// The 8 bf16 values of a 16-byte chunk as fp32, in feature order.
__device__ __forceinline__ void unpack8(uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// acc + sum_i a[i] * b[i], sequentially in feature order (the order dot8_seq uses).
__device__ __forceinline__ float fma8(const float (&a)[8], const float (&b)[8], float acc) {
#pragma unroll
  for (int i = 0; i < 8; ++i) acc = fmaf(a[i], b[i], acc);
  return acc;
}

// G token rows against one gate row and one up row held in shared memory.  Each chunk of the
// two weight rows is unpacked once, each token's chunk of x once, and shared by the gate and
// up sums (per-sum order: chunks lane, lane+32, ..., features in order, as dot8_seq).
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
    float gf[8], uf[8];
    unpack8(g[ch], gf);
    unpack8(uu[ch], uf);
#pragma unroll
    for (int t = 0; t < G; ++t) {
      if (t < n) {
        float xf[8];
        unpack8(XS ? xs[row[t] + ch] : __ldg(xs + row[t] + ch), xf);
        ag[t] = fma8(xf, gf, ag[t]);
        au[t] = fma8(xf, uf, au[t]);
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
    float hf[G][8];  // each token's chunk of h, unpacked once for all rows
#pragma unroll
    for (int t = 0; t < G; ++t)
      unpack8((t < n) ? ld_cg16(hq + (size_t)t * d_ff + 8 * ch) : make_uint4(0, 0, 0, 0), hf[t]);
#pragma unroll
    for (int r = 0; r < kDownRows; ++r) {
      if (r < rows) {
        float wf[8];
        unpack8(reinterpret_cast<const uint4 *>(st + (size_t)r * d_ff * 2)[ch], wf);
#pragma unroll
        for (int t = 0; t < G; ++t) part[r][t] = fma8(wf, hf[t], part[r][t]);
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

// One token: h chunks ch = lane + 32 i for i < kHPre preloaded in hp (issued before the
// task's stage had arrived), the rest loaded here.
constexpr int kHPre = 8;

__device__ __forceinline__ void load_h1(const uint16_t *__restrict__ hq, int nchunk, int lane,
                                        uint4 (&hp)[kHPre]) {
#pragma unroll
  for (int i = 0; i < kHPre; ++i) {
    const int ch = lane + 32 * i;
    hp[i] = ch < nchunk ? ld_cg16(hq + 8 * ch) : make_uint4(0, 0, 0, 0);
  }
}

__device__ __forceinline__ void down_dots1(const uint8_t *__restrict__ st, int rows,
                                           const uint16_t *__restrict__ hq, const uint4 (&hp)[kHPre],
                                           int d_ff, int nchunk, int lane,
                                           float (&part)[kDownRows][1]) {
#pragma unroll
  for (int r = 0; r < kDownRows; ++r) part[r][0] = 0.f;
#pragma unroll
  for (int i = 0; i < kHPre; ++i) {
    const int ch = lane + 32 * i;
    if (ch < nchunk) {
      float hf[8];
      unpack8(hp[i], hf);
#pragma unroll
      for (int r = 0; r < kDownRows; ++r) {
        if (r < rows) {
          float wf[8];
          unpack8(reinterpret_cast<const uint4 *>(st + (size_t)r * d_ff * 2)[ch], wf);
          part[r][0] = fma8(wf, hf, part[r][0]);
        }
      }
    }
  }
  for (int ch = lane + 32 * kHPre; ch < nchunk; ch += 32) {
    const uint4 hv = ld_cg16(hq + 8 * ch);
#pragma unroll
    for (int r = 0; r < kDownRows; ++r)
      if (r < rows)
        part[r][0] = dot8_seq(reinterpret_cast<const uint4 *>(st + (size_t)r * d_ff * 2)[ch], hv,
                              part[r][0]);
  }
#pragma unroll
  for (int r = 0; r < kDownRows; ++r)
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
      part[r][0] += __shfl_xor_sync(0xffffffffu, part[r][0], off);
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
          float xf[8];  // unpacked once for the gate and the up sum
          unpack8(XS ? xs[xi] : __ldg(xs + xi), xf);
          bg[t] = fma8(vg, xf, bg[t]);
          bu[t] = fma8(vu, xf, bu[t]);
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

// rows W_down rows: their codes at `codes` (d_ff/2 bytes per row), their scales at `scales`
// (d_ff/32 bytes per row).  Per 32-input block: each token's h words are unpacked once for
// all rows; each row's block sum runs over its 32 inputs in order, then takes the block scale.
template <int G>
__device__ __forceinline__ void down_dots_fp4(const uint8_t *__restrict__ codes,
                                              const uint8_t *__restrict__ scales, int rows,
                                              const uint16_t *__restrict__ hq, int n, int d_ff,
                                              int lane, float (&part)[kDownRows][G]) {
  const int nblk = d_ff >> 5;
  const size_t cb = (size_t)d_ff / 2, sbr = (size_t)d_ff / 32;
#pragma unroll
  for (int r = 0; r < kDownRows; ++r)
#pragma unroll
    for (int t = 0; t < G; ++t) part[r][t] = 0.f;
  for (int ch = lane; ch < nblk; ch += 32) {
    uint4 qr[kDownRows];
#pragma unroll
    for (int r = 0; r < kDownRows; ++r)
      qr[r] = r < rows ? reinterpret_cast<const uint4 *>(codes + r * cb)[ch] : make_uint4(0, 0, 0, 0);
    float b[kDownRows][G];
#pragma unroll
    for (int r = 0; r < kDownRows; ++r)
#pragma unroll
      for (int t = 0; t < G; ++t) b[r][t] = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float hf[G][8];
#pragma unroll
      for (int t = 0; t < G; ++t)
        unpack8((t < n) ? ld_cg16(hq + (size_t)t * d_ff + 32 * ch + 8 * q) : make_uint4(0, 0, 0, 0),
                hf[t]);
#pragma unroll
      for (int r = 0; r < kDownRows; ++r) {
        if (r < rows) {
          const uint32_t w = q == 0 ? qr[r].x : (q == 1 ? qr[r].y : (q == 2 ? qr[r].z : qr[r].w));
          float v[8];
          decode8(w, v);
#pragma unroll
          for (int t = 0; t < G; ++t) b[r][t] = fma8(v, hf[t], b[r][t]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kDownRows; ++r) {
      if (r < rows) {
        const float sc = e8m0_f32(scales[r * sbr + ch]);
#pragma unroll
        for (int t = 0; t < G; ++t) part[r][t] = fmaf(b[r][t], sc, part[r][t]);
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
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, d_ff = a.d_ff, T = a.T;
  const int nchunk = d >> 3;
  const size_t x_bytes = XS ? (size_t)T * d * 2 : 0;
  const DecLayout lay = dec_layout(x_bytes, a.max_items, a.n_rows);
  WorkItem *items = reinterpret_cast<WorkItem *>(smem + lay.items);
  int32_t *tok_s = reinterpret_cast<int32_t *>(smem + lay.tok);
  int *flags = reinterpret_cast<int *>(smem + lay.flags);  // [4] arrivals, [4] ok, [4] poller
  Ring r;
  r.base = smem + lay.ring;
  r.stage_bytes = a.stage_bytes;
  r.n = a.n_stages;
  r.full = reinterpret_cast<uint64_t *>(r.base + (size_t)r.n * a.stage_bytes);
  r.empty = r.full + r.n;
  volatile int *abort = reinterpret_cast<volatile int *>(r.empty + r.n);
  if (threadIdx.x == 0) {
    for (int s = 0; s < r.n; ++s) {
      mbar_init(&r.full[s], 1);
      mbar_init(&r.empty[s], kConsumers);
    }
    *abort = 0;
    fence_barrier_init();
  }
  if (threadIdx.x < 16) flags[threadIdx.x] = 0;
  // everything below reads what the control kernel of this call wrote (work list, fills,
  // zeroed counters), and x may be the previous call's output
  pdl_wait();
  // the next kernel (the next call's routing) may start now: it reads nothing this kernel
  // writes before its own wait, and everything it prefetches earlier was last written by
  // this call's control kernel, which has completed
  pdl_trigger();
  // one round of independent loads: x, the work list, the rows' tokens and the counters
  DevCounters *ctr = a.ctr;
  const int call_status = ctr->call_status, n_work = ctr->n_work, n_hit = ctr->n_hit;
  const int n_fill = ctr->n_fill;
  const uint64_t limit = ctr->wait_ns;
  if (XS)
    for (int i = threadIdx.x; i < T * nchunk; i += blockDim.x)
      reinterpret_cast<uint4 *>(smem)[i] = __ldg(reinterpret_cast<const uint4 *>(a.x) + i);
  for (int i = threadIdx.x; i < a.max_items * (int)(sizeof(WorkItem) / 8); i += blockDim.x)
    reinterpret_cast<uint2 *>(items)[i] = reinterpret_cast<const uint2 *>(a.work)[i];
  for (int i = threadIdx.x; i < a.n_rows; i += blockDim.x) tok_s[i] = a.tok[i];
  __syncthreads();
  if (call_status != 0 || n_work > a.max_items) return;
  // phase counters and flags, one 128-byte line each: CTAs whose consumer warps have all
  // finished their gate/up tasks of resident items (A), of missed items (C), and all their
  // tasks (Y); a flag per phase set by the last CTA to count itself
  int *g_cnt = a.sync, *g_flag = a.sync + 3 * 32;
  int *fill_done = a.sync + kSyncPhaseInts, *fill_dn = fill_done + kMaxE;
  TaskList tl;
  tl.n_hit = n_hit;
  tl.n_miss = n_fill;
  tl.n_res = n_work - n_fill;
  tl.n_jb = (d_ff + a.R_gu - 1) / a.R_gu;
  tl.n_ib = (d + a.R_dn - 1) / a.R_dn;
  tl.nA = tl.n_res * tl.n_jb;
  tl.nB = tl.n_res * tl.n_ib;
  tl.nC = tl.n_miss * tl.n_jb;
  tl.n = tl.nA + tl.nB + tl.nC + tl.n_miss * tl.n_ib;
  const int fill_chunks = (int)((a.entry_bytes / 16 + kFillChunk - 1) / kFillChunk);
  // chunks holding W_gate and W_up (the first 4*d*d_ff bytes of a bf16 entry), then the rest
  const int gu_chunks =
      FP4 ? fill_chunks
          : min(fill_chunks, (int)(((size_t)4 * d * d_ff / 16 + kFillChunk - 1) / kFillChunk));
  const int dn_chunks = fill_chunks - gu_chunks;

  if (warp > kProducerWarp) {
    // ------------------------------------------------------------ fill warps
    const int fw = blockIdx.x * kFillWarps + (warp - kProducerWarp - 1);
    const int n_fw = gridDim.x * kFillWarps;
    const int hold = ctr->hold_fills;
    const size_t ev = a.entry_bytes / 16;
    const CacheDesc *cd = a.cache;
    uint4 *slots = reinterpret_cast<uint4 *>(cd->slots);
    const int gu_total = n_fill * gu_chunks;
    for (int c = fw; c < n_fill * fill_chunks; c += n_fw) {
      int m, cc;
      if (c < gu_total) {
        m = c / gu_chunks;
        cc = c - m * gu_chunks;
      } else {
        const int c2 = c - gu_total;
        m = c2 / dn_chunks;
        cc = gu_chunks + (c2 - m * dn_chunks);
      }
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
      if (lane == 0 && !hold) atomicAdd(cc < gu_chunks ? &fill_done[m] : &fill_dn[m], 1);
    }
    return;
  }

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      int it = 0;
      int ready_gu = -1, ready_dn = -1;
      for (int g = blockIdx.x; g < tl.n; g += gridDim.x, ++it) {
        const Task t = tl.at(g);
        int s, use;
        r.slot_of(it, s, use);
        if (use > 0 && !mbar_wait_abortable(&r.empty[s], (uint32_t)((use - 1) & 1), limit, abort)) {
          ok = false;
          break;
        }
        if (t.miss >= 0 && t.miss != ready_gu) {
          if (!wait_count(&fill_done[t.miss], gu_chunks, limit, abort)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
          ready_gu = t.miss;
        }
        if (t.miss >= 0 && t.down && dn_chunks > 0 && t.miss != ready_dn) {
          if (!wait_count(&fill_dn[t.miss], dn_chunks, limit, abort)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
          ready_dn = t.miss;
        }
        const uint8_t *W = reinterpret_cast<const uint8_t *>(items[t.u].W);
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
      for (int i = (it > r.n ? it - r.n : 0); i < it; ++i) {
        int s, use;
        r.slot_of(i, s, use);
        // suspended between polls: a spinning thread takes shared-memory cycles from the
        // consumers still at work
        for (long j = 0; j < (1L << 22); ++j)
          if (mbar_try_wait_sleep(&r.full[s], (uint32_t)(use & 1), 1000)) break;
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // Every consumer warp takes every task of its CTA, in list order, and works on its rows of
  // the task's stage: gate/up row pairs w, w+8, ..., down rows [w*rpw, (w+1)*rpw).  It counts
  // itself in phase A when it leaves A (first task past A, or no task left), waits for every
  // consumer warp of the grid there before the first down task of a resident item, does the
  // same with phase C before the first down task of a missed item, and counts itself in
  // phase Y after its last task; once all warps are counted there, each combines its slice of
  // the output.  One fence per warp and phase.
  const uint4 *xs = XS ? reinterpret_cast<const uint4 *>(smem) : reinterpret_cast<const uint4 *>(a.x);
  const int P = T * a.k;
  const int nchunk_h = d_ff >> 3;
  const int n_warps = kConsumers * gridDim.x;
  const int rpw = (a.R_dn + kConsumers - 1) / kConsumers;  // down rows per consumer warp
  auto fail = [&]() {
    if (lane == 0) {
      *abort = 1;
      set_status(ctr, FT_ERR_TIMEOUT);
    }
  };
  // Count this warp in phase ph (its stores ordered before the count).  The CTA's last warp
  // counts the CTA in g_cnt[ph]; the grid's last CTA raises g_flag[ph].
  auto arrive = [&](int ph) {
    __threadfence();
    __syncwarp();
    if (lane == 0 && atomicAdd_block(&flags[ph], 1) == kConsumers - 1) {
      __threadfence();
      if (atomicAdd(&g_cnt[32 * ph], 1) == (int)gridDim.x - 1) {
        __threadfence();
        atomicExch(&g_flag[32 * ph], 1);
      }
    }
  };
  // Wait until every consumer warp of the grid has counted itself in phase ph: one warp of
  // the CTA polls g_flag[ph] (acquire, gpu scope) and raises the CTA's flag, the others wait
  // on that flag; every lane then orders its reads after it.
  auto wait_all = [&](int ph) -> bool {
    bool ok = true;
    volatile int *cta_ok = flags + 4 + ph;
    if (lane == 0 && !*cta_ok) {
      if (atomicCAS_block(&flags[8 + ph], 0, 1) == 0) {
        ok = wait_count(&g_flag[32 * ph], 1, limit, abort);
        if (ok) {
          __threadfence_block();
          *cta_ok = 1;
        }
      } else {
        ok = wait_smem_flag(cta_ok, limit, abort);
      }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
      (void)*cta_ok;
      __threadfence_block();
    }
    return ok;
  };
  const int endA = tl.nA, endB = tl.nA + tl.nB, endC = endB + tl.nC;
  const bool need_A = tl.nB > 0, need_C = tl.n_miss > 0;  // phases some warp waits for
  bool passed_A = false, passed_C = false, waited_A = false, waited_C = false;
  int it = 0;
  for (int g = blockIdx.x; g < tl.n; g += gridDim.x, ++it) {
    if (!passed_A && g >= endA) {
      if (need_A) arrive(0);
      passed_A = true;
    }
    if (!passed_C && g >= endC) {
      if (need_C) arrive(1);
      passed_C = true;
    }
    const Task t = tl.at(g);
    int s, use;
    r.slot_of(it, s, use);
    const WorkItem wi = items[t.u];
    const int c = wi.count;
    bool ok = true;
    if (!t.down) {
      // gate/up + SwiGLU: h[q][j] = silu(g) * u for the item's rows q, row pairs w, w+8, ...
      if (lane == 0) ok = mbar_wait_abortable(&r.full[s], (uint32_t)(use & 1), limit, abort);
      if (!__shfl_sync(0xffffffffu, ok, 0)) return fail();
      const uint8_t *st = r.stage(s);
      const int j0 = t.blk * a.R_gu;
      const int rows = FP4 ? a.R_gu : min(a.R_gu, d_ff - j0);
      for (int rr = warp; rr < rows; rr += kConsumers) {
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
          const int32_t *tk = tok_s + wi.q0 + t0;
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
      __syncwarp();
      if (lane == 0) mbar_arrive(&r.empty[s]);
    } else {
      // down: y[q][i] for the item's rows q, rows [i0 + w*rpw, ...) of the block; the item's h
      // is complete once every warp has passed its gate/up phase.  h of a single token is
      // loaded before the stage is waited for.
      if (g < endB && !waited_A) {
        if (!wait_all(0)) return fail();
        waited_A = true;
      } else if (g >= endC && !waited_C) {
        if (!wait_all(1)) return fail();
        waited_C = true;
      }
      const int i0 = t.blk * a.R_dn;
      const int blk_rows = FP4 ? a.R_dn : min(a.R_dn, d - i0);
      const int r0 = warp * rpw;
      const int rows = max(0, min(rpw, blk_rows - r0));
      uint4 hp[kHPre];
      const bool pre = !FP4 && c == 1 && rows > 0;
      if (pre) load_h1(a.h + (size_t)wi.q0 * d_ff, nchunk_h, lane, hp);
      if (lane == 0) ok = mbar_wait_abortable(&r.full[s], (uint32_t)(use & 1), limit, abort);
      if (!__shfl_sync(0xffffffffu, ok, 0)) return fail();
      if (rows > 0) {
        const size_t row_bytes = FP4 ? (size_t)d_ff / 2 : (size_t)d_ff * 2;
        const uint8_t *st = r.stage(s) + (size_t)r0 * row_bytes;
        // MXFP4: this warp's scale rows follow all R_dn code rows of the stage
        const uint8_t *sc = r.stage(s) + (size_t)a.R_dn * (d_ff / 2) + (size_t)r0 * (d_ff / 32);
        if (pre) {
          float part[kDownRows][1];
          down_dots1(st, rows, a.h + (size_t)wi.q0 * d_ff, hp, d_ff, nchunk_h, lane, part);
          float *yq = a.y + (size_t)wi.q0 * d + i0 + r0;
#pragma unroll
          for (int q = 0; q < kDownRows; ++q)
            if (lane == q && q < rows) yq[q] = part[q][0];
        } else {
          for (int t0 = 0; t0 < c; t0 += 4) {
            const int n = min(4, c - t0);
            const uint16_t *hq = a.h + (size_t)(wi.q0 + t0) * d_ff;
            float *yq = a.y + (size_t)(wi.q0 + t0) * d + i0 + r0;
            if (n == 1) {
              float part[kDownRows][1];
              if (FP4)
                down_dots_fp4<1>(st, sc, rows, hq, 1, d_ff, lane, part);
              else
                down_dots<1>(st, rows, hq, 1, d_ff, nchunk_h, lane, part);
#pragma unroll
              for (int q = 0; q < kDownRows; ++q)
                if (lane == q && q < rows) yq[q] = part[q][0];
            } else {
              float part[kDownRows][4];
              if (FP4)
                down_dots_fp4<4>(st, sc, rows, hq, n, d_ff, lane, part);
              else
                down_dots<4>(st, rows, hq, n, d_ff, nchunk_h, lane, part);
#pragma unroll
              for (int q = 0; q < kDownRows; ++q)
#pragma unroll
                for (int tt = 0; tt < 4; ++tt)
                  if (lane == q * 4 + tt && q < rows && tt < n)
                    yq[(size_t)tt * d + q] = part[q][tt];
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&r.empty[s]);
    }
  }
  if (!passed_A && need_A) arrive(0);
  if (!passed_C && need_C) arrive(1);
  arrive(2);
  if (!wait_all(2)) return fail();
  // every y row is written: out[t][i] = sum_j w[t][j] * y[row of (t, j)][i] in rank order, then
  // the shared expert's row, for this warp's slice of (t, i)
  const int k = a.k;
  const int gw = blockIdx.x * kConsumers + warp;
  for (int e = gw * 32 + lane; e < T * d; e += n_warps * 32) {
    const int tt = e / d, i = e - tt * d;
    float acc = 0.f;
    for (int j = 0; j < k; ++j)
      acc = fmaf(a.w[tt * k + j], __ldcg(a.y + (size_t)a.inv[tt * k + j] * d + i), acc);
    if (a.shared) acc += __ldcg(a.y + (size_t)(P + tt) * d + i);
    a.out[e] = f32_to_bf16(acc);
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

// Stages of about a third of the ring (at least three in flight), each one task: R_gu
// gate/up row pairs, or R_dn down rows (at most kDownRows per consumer warp).  x stays in
// shared memory when it leaves room for three stages of at least 48 KB.
DecodePlan plan_decode(int T, int d, int d_ff, int max_items, int n_rows, bool fp4) {
  DecodePlan p{};
  const size_t xb = (size_t)T * d * 2;
  const size_t fixed = 1024 + (size_t)max_items * sizeof(WorkItem) + (size_t)n_rows * 4 + 512;
  p.xs = xb + fixed + 3 * (48u << 10) <= kDecSmemMax;
  p.ring = (uint32_t)std::min<size_t>(kDecRing, kDecSmemMax - fixed - (p.xs ? xb : 0));
  const uint32_t target = p.ring / 3;
  const int max_dn = kConsumers * kDownRows;
  if (!fp4) {
    const uint32_t unit_gu = 4u * d, unit_dn = 2u * d_ff;
    p.R_gu = std::max(1, std::min(d_ff, (int)(target / unit_gu)));
    p.R_dn = std::max(1, std::min({d, max_dn, (int)(target / unit_dn)}));
    p.stage = std::max((uint32_t)p.R_gu * unit_gu, (uint32_t)p.R_dn * unit_dn);
  } else {
    // whole tasks only (d_ff % R_gu == 0, d % R_dn == 0) and every scale copy a multiple of
    // 16 bytes (R_gu * d and R_dn * d_ff multiples of 512)
    const uint32_t unit_gu = (uint32_t)d * 17 / 16, unit_dn = (uint32_t)d_ff * 17 / 32;
    p.R_gu = 0;
    for (int c = std::min(d_ff, (int)(target / unit_gu)); c >= 1 && !p.R_gu; --c)
      if (d_ff % c == 0 && ((size_t)c * d) % 512 == 0) p.R_gu = c;
    p.R_dn = 0;
    for (int c = std::min({d, max_dn, (int)(target / unit_dn)}); c >= 1 && !p.R_dn; --c)
      if (d % c == 0 && ((size_t)c * d_ff) % 512 == 0) p.R_dn = c;
    if (!p.R_gu) p.R_gu = 4;  // d a multiple of 128 always allows 4
    if (!p.R_dn) p.R_dn = 4;
    p.stage = std::max((uint32_t)p.R_gu * unit_gu, (uint32_t)p.R_dn * unit_dn);
  }
  p.stage = (p.stage + 127) & ~127u;
  p.n_stages = std::max(1, std::min(8, (int)(p.ring / p.stage)));
  p.smem = dec_smem_bytes(p.xs ? xb : 0, max_items, n_rows, p.stage, p.n_stages);
  p.n_ib = (d + p.R_dn - 1) / p.R_dn;
  return p;
}

int launch_decode_experts(DecodeArgs a, bool fp4, cudaStream_t s) {
  a.max_items = std::min(a.E, a.T * a.k) + a.shared;
  a.n_rows = a.T * a.k + (a.shared ? a.T : 0);
  const DecodePlan p = plan_decode(a.T, a.d, a.d_ff, a.max_items, a.n_rows, fp4);
  a.R_gu = p.R_gu;
  a.R_dn = p.R_dn;
  a.stage_bytes = p.stage;
  a.n_stages = p.n_stages;
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
