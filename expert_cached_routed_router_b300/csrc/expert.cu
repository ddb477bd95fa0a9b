// Expert-side kernels: miss fills from the host pool, the decode GEMVs (gate/up + SwiGLU,
// down + weighted combine) and the CUDA-core grouped GEMM used for larger token counts
// when the tensor-core path is not selected.
//
// FreeToken benchmark, "how FreeToken serves large MoE models" (runtime-layer table): the
// host link moves selected experts into the GPU cache; decode misses are filled there and
// executed on the GPU (the pages' CPU execution of misses is not part of this library).
// FreeToken RTX 4090, "how the MoE memory hierarchy works": an expert is executed from its
// complete (layer, expert) entry wherever the mapping says it lives.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <map>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace ftm {

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// ---------------------------------------------------------------------------------------
// Miss fill: every fill-list entry (slot, layer, expert) is copied from the mapped pinned
// host pool to its slot by SM loads over the host link (16 bytes per thread per load, kFillU
// loads in flight per thread).  The grid is fixed; the count is read on the device, so the
// launch needs no host round trip and can be captured.
// ---------------------------------------------------------------------------------------
constexpr int kFillU = 8;

__global__ void __launch_bounds__(512) k_fill(const uint4 *__restrict__ pool,
                                              const CacheDesc *__restrict__ cache,
                                              const int32_t *__restrict__ fills,
                                              const DevCounters *__restrict__ ctr,
                                              size_t entry_vec, int E) {
  pdl_trigger();
  pdl_wait();
  const int n = ctr->n_fill;
  uint4 *slots = reinterpret_cast<uint4 *>(cache->slots);
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t t0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int f = 0; f < n; ++f) {
    const int slot = fills[3 * f], l = fills[3 * f + 1], e = fills[3 * f + 2];
    const uint4 *src = pool + ((size_t)l * E + e) * entry_vec;
    uint4 *dst = slots + (size_t)slot * entry_vec;
    size_t i = t0;
    for (; i + (kFillU - 1) * stride < entry_vec; i += kFillU * stride) {
      uint4 v[kFillU];
#pragma unroll
      for (int u = 0; u < kFillU; ++u) v[u] = src[i + u * stride];
#pragma unroll
      for (int u = 0; u < kFillU; ++u) dst[i + u * stride] = v[u];
    }
    for (; i < entry_vec; i += stride) dst[i] = src[i];
  }
}

void launch_fill(const uint16_t *pool_dev, const CacheDesc *cache, const int32_t *fills,
                 DevCounters *ctr, size_t entry_bytes, int E, int max_fill, cudaStream_t s) {
  (void)max_fill;
  launch_pdl(k_fill, dim3(148), dim3(512), 0, s, reinterpret_cast<const uint4 *>(pool_dev), cache,
             fills, (const DevCounters *)ctr, entry_bytes / 16, E);
}

// ---------------------------------------------------------------------------------------
// Decode GEMVs fed by bulk TMA copies.
//
// One persistent CTA per SM: warp 8 is the producer, warps 0..7 consume.  Work is a list of
// tasks (work item u, block of R consecutive weight rows); the rows of a block are contiguous
// in the entry, so the producer moves each block with one cp.async.bulk per matrix into a
// shared-memory stage (mbarrier "full" with transaction bytes, "empty" with the arrival of the
// stage's one consumer warp; the stage-to-warp assignment is RingSmem::slot_of below).  Bytes
// in flight per SM are the whole ring, independent of registers.  Consumers dot the rows with
// the item's token vectors (from shared memory when they fit).
// All waits are bounded; on a timeout the CTA records FT_ERR_TIMEOUT, waits (bounded) for its
// own copies in flight and returns.
// ---------------------------------------------------------------------------------------
constexpr int kGemvWarps = 8;            // consumer warps
constexpr int kGemvThreads = (kGemvWarps + 1) * 32;
constexpr int kMaxStagesPerWarp = 4;
constexpr uint32_t kRingBytes = 192u << 10;  // all stages together

// Stages per consumer warp for a ring of `ring_bytes` (at least one).
__host__ __device__ __forceinline__ int stages_per_warp(uint32_t ring_bytes, uint32_t stage_bytes) {
  int s = (int)(ring_bytes / (stage_bytes * kGemvWarps));
  return s < 1 ? 1 : (s > kMaxStagesPerWarp ? kMaxStagesPerWarp : s);
}

// The ring: consumer warp w owns stages w*spw .. w*spw+spw-1 and takes this CTA's tasks
// w, w+8, w+16, ...; its j-th task uses stage w*spw + (j % spw) for the (j / spw)-th time.  A
// stage therefore has one consumer that waits on its phases strictly in order, so a parity
// wait can never match an older phase.
struct RingSmem {
  uint8_t *base;
  uint32_t stage_bytes;
  int spw;  // stages per consumer warp
  uint64_t *full;
  uint64_t *empty;
  __device__ __forceinline__ uint8_t *stage(int s) const { return base + (size_t)s * stage_bytes; }
  __device__ __forceinline__ int n() const { return spw * kGemvWarps; }
  // stage and use count of this CTA's it-th task
  __device__ __forceinline__ void slot_of(long it, int &s, long &use) const {
    const int w = (int)(it % kGemvWarps);
    const long j = it / kGemvWarps;
    s = w * spw + (int)(j % spw);
    use = j / spw;
  }
};

// Carve the dynamic shared memory: [x staging | stages | barriers].
__device__ __forceinline__ RingSmem ring_layout(uint8_t *smem, size_t x_bytes, uint32_t stage_bytes,
                                                uint32_t ring_bytes) {
  RingSmem r;
  r.base = smem + ((x_bytes + 127) & ~(size_t)127);
  r.stage_bytes = stage_bytes;
  r.spw = stages_per_warp(ring_bytes, stage_bytes);
  r.full = reinterpret_cast<uint64_t *>(r.base + (size_t)r.n() * stage_bytes);
  r.empty = r.full + r.n();
  return r;
}

static size_t ring_smem_bytes(size_t x_bytes, uint32_t stage_bytes, uint32_t ring_bytes) {
  const int n = stages_per_warp(ring_bytes, stage_bytes) * kGemvWarps;
  return ((x_bytes + 127) & ~(size_t)127) + (size_t)n * stage_bytes + 2 * n * 8;
}

__device__ __forceinline__ void ring_init(RingSmem &r) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < r.n(); ++s) {
      mbar_init(&r.full[s], 1);
      mbar_init(&r.empty[s], 1);
    }
    fence_barrier_init();
  }
}

// Producer side of the ring (one thread): for each of this CTA's tasks, wait until the
// task's stage has been released by its previous use and issue the bulk copies that
// `issue(task, stage_ptr, bar)` describes.  Returns false on a timeout.  At the end it waits
// for its copies in flight.
template <typename Issue>
__device__ __forceinline__ bool ring_produce(RingSmem &r, long n_tasks, Issue issue) {
  long it = 0;
  bool ok = true;
  for (long task = blockIdx.x; task < n_tasks; task += gridDim.x, ++it) {
    int s;
    long use;
    r.slot_of(it, s, use);
    if (use > 0 && !mbar_wait(&r.empty[s], (uint32_t)((use - 1) & 1))) {
      ok = false;
      break;
    }
    issue(task, r.stage(s), &r.full[s]);
  }
  // drain: the copies of the last tasks (at most one in flight per stage)
  const long n = r.n();
  for (long i = (it > n ? it - n : 0); i < it; ++i) {
    int s;
    long use;
    r.slot_of(i, s, use);
    mbar_wait(&r.full[s], (uint32_t)(use & 1));
  }
  return ok;
}

// Consumer side: consumer warp w takes this CTA's tasks w, w+8, ... whole; for each it waits
// for the task's stage, runs `use`, and releases the stage.
template <typename Use>
__device__ __forceinline__ bool ring_consume(RingSmem &r, long n_tasks, Use fn) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long it = 0;
  for (long task = blockIdx.x; task < n_tasks; task += gridDim.x, ++it) {
    if ((int)(it % kGemvWarps) != warp) continue;
    int s;
    long use;
    r.slot_of(it, s, use);
    if (!mbar_wait(&r.full[s], (uint32_t)(use & 1))) return false;
    fn(task, r.stage(s));
    __syncwarp();
    if (lane == 0) mbar_arrive(&r.empty[s]);
  }
  return true;
}

// Token groups: an item's c tokens are processed G at a time (G = 1 or 4); the weight rows
// sit in shared memory, so going over them once per group costs shared-memory bandwidth only.
template <int G, bool XS>
__device__ __forceinline__ void gateup_rows(const uint4 *__restrict__ g, const uint4 *__restrict__ uu,
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

// gate/up + SwiGLU.  Task = (item u, rows j0 .. j0+R-1 of W_gate and of W_up); stage =
// [R gate rows | R up rows].  h[q][j] = silu(g) * u (bf16).  x is staged in shared memory
// when it fits next to the ring (XS).
template <bool XS>
__global__ void __launch_bounds__(kGemvThreads, 1) k_gateup_tma(
    const WorkItem *__restrict__ work, DevCounters *__restrict__ ctr,
    const uint16_t *__restrict__ x, const int32_t *__restrict__ tok, uint16_t *__restrict__ h,
    int T, int d, int d_ff, int R, uint32_t stage_bytes, uint32_t ring_bytes) {
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_trigger();
  const int nchunk = d >> 3;
  const size_t x_bytes = XS ? (size_t)T * d * 2 : 0;
  RingSmem r = ring_layout(smem, x_bytes, stage_bytes, ring_bytes);
  const uint4 *xs = XS ? reinterpret_cast<const uint4 *>(smem) : reinterpret_cast<const uint4 *>(x);
  ring_init(r);
  // the work list, the fills and the slot table come from the kernels before; so may x (the
  // previous call's output), which is staged only after the wait
  pdl_wait();
  if (XS)
    for (int i = threadIdx.x; i < T * nchunk; i += blockDim.x)
      reinterpret_cast<uint4 *>(smem)[i] = __ldg(reinterpret_cast<const uint4 *>(x) + i);
  __syncthreads();
  if (ctr->call_status != 0) return;
  const int n_work = ctr->n_work;
  const int n_jb = (d_ff + R - 1) / R;
  const long n_tasks = (long)n_work * n_jb;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  bool ok = true;
  if (warp == kGemvWarps) {
    if (lane == 0) {
      int cu = -1;
      const uint16_t *W = nullptr;
      ok = ring_produce(r, n_tasks, [&](long task, uint8_t *st, uint64_t *bar) {
        const int u = (int)(task / n_jb), j0 = (int)(task - (long)u * n_jb) * R;
        const int rows = min(R, d_ff - j0);
        const uint32_t bytes = (uint32_t)rows * d * 2;
        if (u != cu) {  // consecutive tasks mostly stay on one item
          cu = u;
          W = work[u].W;
        }
        mbar_arrive_expect_tx(bar, 2 * bytes);
        bulk_g2s(st, W + (size_t)j0 * d, bytes, bar);
        bulk_g2s(st + (size_t)R * d * 2, W + (size_t)(d_ff + j0) * d, bytes, bar);
      });
    }
  } else {
    int cu = -1;
    WorkItem wi{};
    ok = ring_consume(r, n_tasks, [&](long task, const uint8_t *st) {
      const int u = (int)(task / n_jb), j0 = (int)(task - (long)u * n_jb) * R;
      const int rows = min(R, d_ff - j0);
      if (u != cu) {
        cu = u;
        wi = work[u];
      }
      const int c = wi.count;
      for (int rr = 0; rr < rows; ++rr) {
        const uint4 *g = reinterpret_cast<const uint4 *>(st + (size_t)rr * d * 2);
        const uint4 *uu = reinterpret_cast<const uint4 *>(st + (size_t)(R + rr) * d * 2);
        for (int t0 = 0; t0 < c; t0 += 4) {
          const int n = min(4, c - t0);
          const int32_t *tk = tok + wi.q0 + t0;
          uint16_t *hq = h + (size_t)(wi.q0 + t0) * d_ff + j0 + rr;
          if (n == 1) {
            float ag[1], au[1];
            gateup_rows<1, XS>(g, uu, xs, tk, 1, nchunk, lane, ag, au);
            if (lane == 0) hq[0] = f32_to_bf16(silu_mul(ag[0], au[0]));
          } else {
            float ag[4], au[4];
            gateup_rows<4, XS>(g, uu, xs, tk, n, nchunk, lane, ag, au);
#pragma unroll
            for (int t = 0; t < 4; ++t)
              if (lane == t && t < n) hq[(size_t)t * d_ff] = f32_to_bf16(silu_mul(ag[t], au[t]));
          }
        }
      }
    });
  }
  if (!ok) set_status(ctr, FT_ERR_TIMEOUT);
}

// Up to kDownRows W_down rows of a task against G token rows of h: every h chunk is loaded once
// and used for all the task's rows (held in shared memory).
constexpr int kDownRows = 8;

template <int G>
__device__ __forceinline__ void down_rows(const uint8_t *__restrict__ st, int rows,
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
      hv[t] = (t < n) ? __ldg(reinterpret_cast<const uint4 *>(hq + (size_t)t * d_ff) + ch)
                      : make_uint4(0, 0, 0, 0);
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

// down: task = (item u, rows i0 .. i0+R-1 of W_down); y[q][i] fp32 for the item's rows q.
__global__ void __launch_bounds__(kGemvThreads, 1) k_down_tma(
    const WorkItem *__restrict__ work, DevCounters *__restrict__ ctr,
    const uint16_t *__restrict__ h, float *__restrict__ y, int d, int d_ff, int R,
    uint32_t stage_bytes, uint32_t ring_bytes) {
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_trigger();
  const int nchunk = d_ff >> 3;
  RingSmem r = ring_layout(smem, 0, stage_bytes, ring_bytes);
  ring_init(r);
  __syncthreads();
  pdl_wait();  // h comes from the gate/up kernel
  if (ctr->call_status != 0) return;
  const int n_work = ctr->n_work;
  const int n_ib = (d + R - 1) / R;
  const long n_tasks = (long)n_work * n_ib;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  bool ok = true;
  if (warp == kGemvWarps) {
    if (lane == 0) {
      int cu = -1;
      const uint16_t *W = nullptr;
      ok = ring_produce(r, n_tasks, [&](long task, uint8_t *st, uint64_t *bar) {
        const int u = (int)(task / n_ib), i0 = (int)(task - (long)u * n_ib) * R;
        const int rows = min(R, d - i0);
        const uint32_t bytes = (uint32_t)rows * d_ff * 2;
        if (u != cu) {
          cu = u;
          W = work[u].W;
        }
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(st, W + (size_t)2 * d_ff * d + (size_t)i0 * d_ff, bytes, bar);
      });
    }
  } else {
    int cu = -1;
    WorkItem wi{};
    ok = ring_consume(r, n_tasks, [&](long task, const uint8_t *st) {
      const int u = (int)(task / n_ib), i0 = (int)(task - (long)u * n_ib) * R;
      const int rows = min(R, d - i0);
      if (u != cu) {
        cu = u;
        wi = work[u];
      }
      const int c = wi.count;
      for (int t0 = 0; t0 < c; t0 += 4) {
        const int n = min(4, c - t0);
        const uint16_t *hq = h + (size_t)(wi.q0 + t0) * d_ff;
        float *yq = y + (size_t)(wi.q0 + t0) * d + i0;
        if (n == 1) {
          float part[kDownRows][1];
          down_rows<1>(st, rows, hq, 1, d_ff, nchunk, lane, part);
#pragma unroll
          for (int r = 0; r < kDownRows; ++r)
            if (lane == r && r < rows) yq[r] = part[r][0];
        } else {
          float part[kDownRows][4];
          down_rows<4>(st, rows, hq, n, d_ff, nchunk, lane, part);
#pragma unroll
          for (int r = 0; r < kDownRows; ++r)
#pragma unroll
            for (int t = 0; t < 4; ++t)
              if (lane == r * 4 + t && r < rows && t < n) yq[(size_t)t * d + r] = part[r][t];
        }
      }
    });
  }
  if (!ok) set_status(ctr, FT_ERR_TIMEOUT);
}

// ---------------------------------------------------------------------------------------
// MXFP4 entries (decode).  Codes Wg | Wu | Wd, then scales Wg | Wu | Wd; a row of K inputs
// has K/2 code bytes (input 2i in the low nibble of byte i) and K/32 scale bytes.  A 16-byte
// chunk of a row's codes is exactly one 32-input scale block, so lane work is per block:
// the block's E2M1 values are dotted with the inputs, then the sum is multiplied by the
// block's power-of-two scale (exact).
// ---------------------------------------------------------------------------------------

// E2M1 code (low 4 bits of c) -> fp32: the sign goes to bit 31 and the three magnitude bits
// (2 exponent, 1 mantissa) to bits 22..24, which is the value times 2^-126 (a subnormal when
// the exponent field is 0); one exact multiply by 2^126 restores it.  Relies on fp32
// subnormals being kept (no flush-to-zero build flags).
__device__ __forceinline__ float e2m1_f32(uint32_t c) {
  return __uint_as_float(((c & 8u) << 28) | ((c & 7u) << 22)) * 0x1p126f;
}

// E8M0 scale byte -> 2^(s - 127); s = 255 is NaN.
__device__ __forceinline__ float e8m0_f32(uint32_t s) {
  return s == 0 ? __uint_as_float(0x00400000u)
                : (s == 255 ? __uint_as_float(0x7FC00000u) : __uint_as_float(s << 23));
}

// The 8 inputs held by one 32-bit code word, in input order.
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
__device__ __forceinline__ void gateup_rows_fp4(const uint4 *__restrict__ g,
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

// gate/up + SwiGLU on MXFP4 entries.  Task = (item u, rows j0 .. j0+R-1; d_ff % R == 0);
// stage = [R gate code rows | R up code rows | R gate scale rows | R up scale rows].
template <bool XS>
__global__ void __launch_bounds__(kGemvThreads, 1) k_gateup_fp4(
    const WorkItem *__restrict__ work, DevCounters *__restrict__ ctr,
    const uint16_t *__restrict__ x, const int32_t *__restrict__ tok, uint16_t *__restrict__ h,
    int T, int d, int d_ff, int R, uint32_t stage_bytes, uint32_t ring_bytes) {
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_trigger();
  const int nchunk = d >> 3, nblk = d >> 5;
  const size_t cb = (size_t)d / 2, sbr = (size_t)d / 32;  // code / scale bytes of a row
  const size_t x_bytes = XS ? (size_t)T * d * 2 : 0;
  RingSmem r = ring_layout(smem, x_bytes, stage_bytes, ring_bytes);
  const uint4 *xs = XS ? reinterpret_cast<const uint4 *>(smem) : reinterpret_cast<const uint4 *>(x);
  ring_init(r);
  pdl_wait();  // work list, fills and slot table from the kernels before; x may be too
  if (XS)
    for (int i = threadIdx.x; i < T * nchunk; i += blockDim.x)
      reinterpret_cast<uint4 *>(smem)[i] = __ldg(reinterpret_cast<const uint4 *>(x) + i);
  __syncthreads();
  if (ctr->call_status != 0) return;
  const int n_work = ctr->n_work;
  const int n_jb = d_ff / R;
  const long n_tasks = (long)n_work * n_jb;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t scale0 = (size_t)3 * d * d_ff / 2;  // start of the scale region
  bool ok = true;
  if (warp == kGemvWarps) {
    if (lane == 0) {
      int cu = -1;
      const uint8_t *W = nullptr;
      ok = ring_produce(r, n_tasks, [&](long task, uint8_t *st, uint64_t *bar) {
        const int u = (int)(task / n_jb), j0 = (int)(task - (long)u * n_jb) * R;
        if (u != cu) {
          cu = u;
          W = reinterpret_cast<const uint8_t *>(work[u].W);
        }
        const uint32_t c_bytes = (uint32_t)(R * cb), s_bytes = (uint32_t)(R * sbr);
        mbar_arrive_expect_tx(bar, 2 * c_bytes + 2 * s_bytes);
        bulk_g2s(st, W + (size_t)j0 * cb, c_bytes, bar);
        bulk_g2s(st + c_bytes, W + (size_t)d_ff * cb + (size_t)j0 * cb, c_bytes, bar);
        bulk_g2s(st + 2 * c_bytes, W + scale0 + (size_t)j0 * sbr, s_bytes, bar);
        bulk_g2s(st + 2 * c_bytes + s_bytes, W + scale0 + (size_t)d_ff * sbr + (size_t)j0 * sbr,
                 s_bytes, bar);
      });
    }
  } else {
    int cu = -1;
    WorkItem wi{};
    ok = ring_consume(r, n_tasks, [&](long task, const uint8_t *st) {
      const int u = (int)(task / n_jb), j0 = (int)(task - (long)u * n_jb) * R;
      if (u != cu) {
        cu = u;
        wi = work[u];
      }
      const int c = wi.count;
      for (int rr = 0; rr < R; ++rr) {
        const uint4 *g = reinterpret_cast<const uint4 *>(st + rr * cb);
        const uint4 *uu = reinterpret_cast<const uint4 *>(st + (R + rr) * cb);
        const uint8_t *sg = st + 2 * R * cb + rr * sbr;
        const uint8_t *su = st + 2 * R * cb + (R + rr) * sbr;
        for (int t0 = 0; t0 < c; t0 += 4) {
          const int n = min(4, c - t0);
          const int32_t *tk = tok + wi.q0 + t0;
          uint16_t *hq = h + (size_t)(wi.q0 + t0) * d_ff + j0 + rr;
          if (n == 1) {
            float ag[1], au[1];
            gateup_rows_fp4<1, XS>(g, uu, sg, su, xs, tk, 1, nchunk, nblk, lane, ag, au);
            if (lane == 0) hq[0] = f32_to_bf16(silu_mul(ag[0], au[0]));
          } else {
            float ag[4], au[4];
            gateup_rows_fp4<4, XS>(g, uu, sg, su, xs, tk, n, nchunk, nblk, lane, ag, au);
#pragma unroll
            for (int t = 0; t < 4; ++t)
              if (lane == t && t < n) hq[(size_t)t * d_ff] = f32_to_bf16(silu_mul(ag[t], au[t]));
          }
        }
      }
    });
  }
  if (!ok) set_status(ctr, FT_ERR_TIMEOUT);
}

template <int G>
__device__ __forceinline__ void down_rows_fp4(const uint8_t *__restrict__ st, int R,
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
        hv[t][q] = (t < n) ? __ldg(reinterpret_cast<const uint4 *>(hq + (size_t)t * d_ff) + 4 * ch + q)
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

// down on MXFP4 entries: task = (item u, rows i0 .. i0+R-1 of W_down; d % R == 0, R <= 8);
// stage = [R code rows | R scale rows].
__global__ void __launch_bounds__(kGemvThreads, 1) k_down_fp4(
    const WorkItem *__restrict__ work, DevCounters *__restrict__ ctr,
    const uint16_t *__restrict__ h, float *__restrict__ y, int d, int d_ff, int R,
    uint32_t stage_bytes, uint32_t ring_bytes) {
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_trigger();
  const size_t cb = (size_t)d_ff / 2, sbr = (size_t)d_ff / 32;
  RingSmem r = ring_layout(smem, 0, stage_bytes, ring_bytes);
  ring_init(r);
  __syncthreads();
  pdl_wait();  // h comes from the gate/up kernel
  if (ctr->call_status != 0) return;
  const int n_work = ctr->n_work;
  const int n_ib = d / R;
  const long n_tasks = (long)n_work * n_ib;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t codes_d = (size_t)d * d_ff;                       // 2 * d_ff * d/2
  const size_t scales_d = (size_t)3 * d * d_ff / 2 + (size_t)2 * d_ff * (d / 32);
  bool ok = true;
  if (warp == kGemvWarps) {
    if (lane == 0) {
      int cu = -1;
      const uint8_t *W = nullptr;
      ok = ring_produce(r, n_tasks, [&](long task, uint8_t *st, uint64_t *bar) {
        const int u = (int)(task / n_ib), i0 = (int)(task - (long)u * n_ib) * R;
        if (u != cu) {
          cu = u;
          W = reinterpret_cast<const uint8_t *>(work[u].W);
        }
        const uint32_t c_bytes = (uint32_t)(R * cb), s_bytes = (uint32_t)(R * sbr);
        mbar_arrive_expect_tx(bar, c_bytes + s_bytes);
        bulk_g2s(st, W + codes_d + (size_t)i0 * cb, c_bytes, bar);
        bulk_g2s(st + c_bytes, W + scales_d + (size_t)i0 * sbr, s_bytes, bar);
      });
    }
  } else {
    int cu = -1;
    WorkItem wi{};
    ok = ring_consume(r, n_tasks, [&](long task, const uint8_t *st) {
      const int u = (int)(task / n_ib), i0 = (int)(task - (long)u * n_ib) * R;
      if (u != cu) {
        cu = u;
        wi = work[u];
      }
      const int c = wi.count;
      for (int t0 = 0; t0 < c; t0 += 4) {
        const int n = min(4, c - t0);
        const uint16_t *hq = h + (size_t)(wi.q0 + t0) * d_ff;
        float *yq = y + (size_t)(wi.q0 + t0) * d + i0;
        if (n == 1) {
          float part[kDownRows][1];
          down_rows_fp4<1>(st, R, hq, 1, d_ff, lane, part);
#pragma unroll
          for (int rr = 0; rr < kDownRows; ++rr)
            if (lane == rr && rr < R) yq[rr] = part[rr][0];
        } else {
          float part[kDownRows][4];
          down_rows_fp4<4>(st, R, hq, n, d_ff, lane, part);
#pragma unroll
          for (int rr = 0; rr < kDownRows; ++rr)
#pragma unroll
            for (int t = 0; t < 4; ++t)
              if (lane == rr * 4 + t && rr < R && t < n) yq[(size_t)t * d + rr] = part[rr][t];
        }
      }
    });
  }
  if (!ok) set_status(ctr, FT_ERR_TIMEOUT);
}

static int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

template <typename K>
static void allow_smem(K kern, size_t smem) {
  static std::mutex mu;
  static std::map<const void *, size_t> done;
  std::lock_guard<std::mutex> lock(mu);
  size_t &v = done[reinterpret_cast<const void *>(kern)];
  if (smem > v) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    v = smem;
  }
}

// MXFP4: R rows per task from {16, 8, 4} with R*d a multiple of 512 (every scale copy then
// starts and ends on a 16-byte boundary) and d_ff % R == 0 (no ragged task); 8 stages fit.
static void launch_gateup_fp4(const WorkItem *work, DevCounters *ctr, const uint16_t *x,
                              const int32_t *tok, uint16_t *h, int T, int d, int d_ff,
                              cudaStream_t s) {
  const uint32_t unit = (uint32_t)d * 17 / 16;  // code + scale bytes of one gate/up row pair
  const size_t xb = (size_t)T * d * 2, xr = (xb + 127) & ~(size_t)127;
  const bool xs = xr + (size_t)kGemvWarps * 4 * unit <= (224u << 10);
  const uint32_t ring = xs ? (uint32_t)std::min<size_t>(kRingBytes, (224u << 10) - xr) : kRingBytes;
  int R = 4;
  for (int c : {16, 8})
    if (d_ff % c == 0 && (c * d) % 512 == 0 && (size_t)kGemvWarps * c * unit <= ring) {
      R = c;
      break;
    }
  const uint32_t sb = (uint32_t)R * unit;
  const size_t smem = ring_smem_bytes(xs ? xb : 0, sb, ring);
  auto go = [&](auto kern) {
    allow_smem(kern, smem);
    launch_pdl(kern, dim3(sm_count()), dim3(kGemvThreads), smem, s, work, ctr, x, tok, h, T, d,
               d_ff, R, sb, ring);
  };
  if (xs)
    go(k_gateup_fp4<true>);
  else
    go(k_gateup_fp4<false>);
}

static void launch_down_fp4(const WorkItem *work, DevCounters *ctr, const uint16_t *h, float *y,
                            int d, int d_ff, cudaStream_t s) {
  const uint32_t unit = (uint32_t)d_ff * 17 / 32;  // code + scale bytes of one W_down row
  const int R = ((size_t)kGemvWarps * kDownRows * unit <= kRingBytes) ? kDownRows : 4;
  const uint32_t sb = (uint32_t)R * unit;
  const size_t smem = ring_smem_bytes(0, sb, kRingBytes);
  allow_smem(k_down_fp4, smem);
  launch_pdl(k_down_fp4, dim3(sm_count()), dim3(kGemvThreads), smem, s, work, ctr, h, y, d, d_ff,
             R, sb, kRingBytes);
}

void launch_gateup_gemv(const WorkItem *work, DevCounters *ctr, int max_work, const uint16_t *x,
                        const int32_t *tok, uint16_t *h, int T, int d, int d_ff, bool fp4,
                        cudaStream_t s) {
  (void)max_work;
  if (fp4) {
    launch_gateup_fp4(work, ctr, x, tok, h, T, d, d_ff, s);
    return;
  }
  // one stage per consumer warp holding R gate+up row pairs (R <= 4), as many as fit next to
  // x (kept in shared memory when a one-pair stage per warp still fits in 224 KB)
  const uint32_t unit = 4u * d;
  const size_t xb = (size_t)T * d * 2, xr = (xb + 127) & ~(size_t)127;
  const bool xs = xr + (size_t)kGemvWarps * unit <= (224u << 10);
  const uint32_t ring = xs ? (uint32_t)std::min<size_t>(kRingBytes, (224u << 10) - xr) : kRingBytes;
  const int R = std::max(1, std::min({d_ff, 4, (int)(ring / kGemvWarps / unit)}));
  const uint32_t sb = (uint32_t)R * unit;
  const size_t smem = ring_smem_bytes(xs ? xb : 0, sb, ring);
  auto go = [&](auto kern) {
    allow_smem(kern, smem);
    launch_pdl(kern, dim3(sm_count()), dim3(kGemvThreads), smem, s, work, ctr, x, tok, h, T, d,
               d_ff, R, sb, ring);
  };
  if (xs)
    go(k_gateup_tma<true>);
  else
    go(k_gateup_tma<false>);
}

// out[t][i] = sum_j w[t][j] * y[inv[t*k+j]][i] (j ascending) + y[P+t][i] for the shared
// expert; fixed order, so the result is deterministic.  8 features per thread.
__global__ void k_combine(const float *__restrict__ y, const float *__restrict__ w,
                          const int32_t *__restrict__ inv, const DevCounters *__restrict__ ctr,
                          uint16_t *__restrict__ out, int T, int k, int d, int shared) {
  pdl_trigger();
  pdl_wait();
  if (ctr->call_status != 0) return;
  const int n8 = d >> 3;
  const int gidx = blockIdx.x * blockDim.x + threadIdx.x;
  if (gidx >= T * n8) return;
  const int t = gidx / n8, c = gidx - t * n8;
  float acc[8];
#pragma unroll
  for (int v = 0; v < 8; ++v) acc[v] = 0.f;
  // groups of 8 ranks: all row addresses, then all row loads, then the sums in rank order
  for (int j0 = 0; j0 < k; j0 += 8) {
    const int nj = min(8, k - j0);
    float wj[8];
    int rj[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      wj[u] = u < nj ? w[t * k + j0 + u] : 0.f;
      rj[u] = u < nj ? inv[t * k + j0 + u] : 0;
    }
    float4 ra[8], rb[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (u < nj) {
        const float4 *row = reinterpret_cast<const float4 *>(y + (size_t)rj[u] * d) + 2 * c;
        ra[u] = row[0];
        rb[u] = row[1];
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (u < nj) {
        acc[0] = fmaf(wj[u], ra[u].x, acc[0]);
        acc[1] = fmaf(wj[u], ra[u].y, acc[1]);
        acc[2] = fmaf(wj[u], ra[u].z, acc[2]);
        acc[3] = fmaf(wj[u], ra[u].w, acc[3]);
        acc[4] = fmaf(wj[u], rb[u].x, acc[4]);
        acc[5] = fmaf(wj[u], rb[u].y, acc[5]);
        acc[6] = fmaf(wj[u], rb[u].z, acc[6]);
        acc[7] = fmaf(wj[u], rb[u].w, acc[7]);
      }
    }
  }
  if (shared) {
    const float4 *row = reinterpret_cast<const float4 *>(y + (size_t)(T * k + t) * d) + 2 * c;
    const float4 a = row[0], b = row[1];
    acc[0] += a.x;
    acc[1] += a.y;
    acc[2] += a.z;
    acc[3] += a.w;
    acc[4] += b.x;
    acc[5] += b.y;
    acc[6] += b.z;
    acc[7] += b.w;
  }
  uint4 o;
  o.x = (uint32_t)f32_to_bf16(acc[0]) | ((uint32_t)f32_to_bf16(acc[1]) << 16);
  o.y = (uint32_t)f32_to_bf16(acc[2]) | ((uint32_t)f32_to_bf16(acc[3]) << 16);
  o.z = (uint32_t)f32_to_bf16(acc[4]) | ((uint32_t)f32_to_bf16(acc[5]) << 16);
  o.w = (uint32_t)f32_to_bf16(acc[6]) | ((uint32_t)f32_to_bf16(acc[7]) << 16);
  reinterpret_cast<uint4 *>(out + (size_t)t * d)[c] = o;
}

void launch_down_gemv(const WorkItem *work, DevCounters *ctr, int max_work, const uint16_t *h,
                      float *y, int T, int d, int d_ff, bool fp4, cudaStream_t s) {
  (void)T;
  (void)max_work;
  if (fp4) {
    launch_down_fp4(work, ctr, h, y, d, d_ff, s);
    return;
  }
  const uint32_t unit = 2u * d_ff;
  const int R = std::max(1, std::min({d, kDownRows, (int)(kRingBytes / kGemvWarps / unit)}));
  const uint32_t sb = (uint32_t)R * unit;
  const size_t smem = ring_smem_bytes(0, sb, kRingBytes);
  allow_smem(k_down_tma, smem);
  launch_pdl(k_down_tma, dim3(sm_count()), dim3(kGemvThreads), smem, s, work, ctr, h, y, d, d_ff,
             R, sb, kRingBytes);
}

void launch_combine(const float *y, const float *w, const int32_t *inv, const DevCounters *ctr,
                    uint16_t *out, int T, int k, int d, int shared, cudaStream_t s) {
  const int n = T * (d >> 3);
  launch_pdl(k_combine, dim3((n + 127) / 128), dim3(128), 0, s, y, w, inv, ctr, out, T, k, d,
             shared);
}

// ---------------------------------------------------------------------------------------
// Larger T: gather the permuted activation rows, grouped GEMMs, fp32 combine, cast.
// ---------------------------------------------------------------------------------------
__global__ void k_gather_rows(const uint16_t *__restrict__ x, const int32_t *__restrict__ tok,
                              uint16_t *__restrict__ xp, int rows, int d,
                              const DevCounters *__restrict__ ctr) {
  if (ctr->call_status != 0) return;  // refused call: tok is not this call's
  const int nchunk = d >> 3;
  const size_t n = (size_t)rows * nchunk;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = i / nchunk, ch = i - r * nchunk;
    reinterpret_cast<uint4 *>(xp)[i] =
        __ldg(reinterpret_cast<const uint4 *>(x + (size_t)tok[r] * d) + ch);
  }
}

void launch_gather_rows(const uint16_t *x, const int32_t *tok, uint16_t *xp, int rows, int d,
                        const DevCounters *ctr,
                        cudaStream_t s) {
  if (rows <= 0) return;
  const size_t n = (size_t)rows * (d >> 3);
  const int threads = 256;
  const unsigned blocks = (unsigned)std::min<size_t>((n + threads - 1) / threads, 148 * 16);
  k_gather_rows<<<blocks, threads, 0, s>>>(x, tok, xp, rows, d, ctr);
}

__global__ void k_cast_out(const float *__restrict__ acc, uint16_t *__restrict__ out, size_t n,
                           const DevCounters *__restrict__ ctr) {
  if (ctr->call_status != 0) return;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    out[i] = f32_to_bf16(acc[i]);
}

void launch_cast_out(const float *acc, uint16_t *out, size_t n, const DevCounters *ctr,
                     cudaStream_t s) {
  if (n == 0) return;
  const unsigned blocks = (unsigned)std::min<size_t>((n + 255) / 256, 148 * 16);
  k_cast_out<<<blocks, 256, 0, s>>>(acc, out, n, ctr);
}

}  // namespace ftm
