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

#include "internal.h"

namespace ftm {

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// ---------------------------------------------------------------------------------------
// Miss fill: every fill-list entry (slot, layer, expert) is copied from the mapped pinned
// host pool to its slot by SM loads over the host link.  The grid is fixed; the count is
// read on the device, so the launch needs no host round trip and can be captured.
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(512) k_fill(const uint4 *__restrict__ pool, uint4 *slots,
                                              const int32_t *__restrict__ fills,
                                              const DevCounters *__restrict__ ctr,
                                              size_t entry_vec, int E) {
  const int n = ctr->n_fill;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t t0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int f = 0; f < n; ++f) {
    const int slot = fills[3 * f], l = fills[3 * f + 1], e = fills[3 * f + 2];
    const uint4 *src = pool + ((size_t)l * E + e) * entry_vec;
    uint4 *dst = slots + (size_t)slot * entry_vec;
    size_t i = t0;
    for (; i + 3 * stride < entry_vec; i += 4 * stride) {
      const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride],
                  d = src[i + 3 * stride];
      dst[i] = a;
      dst[i + stride] = b;
      dst[i + 2 * stride] = c;
      dst[i + 3 * stride] = d;
    }
    for (; i < entry_vec; i += stride) dst[i] = src[i];
  }
}

void launch_fill(const uint16_t *pool_dev, uint16_t *slots, const int32_t *fills,
                 const DevCounters *ctr, size_t entry_bytes, int E, int max_fill,
                 cudaStream_t s) {
  (void)max_fill;
  k_fill<<<148 * 2, 512, 0, s>>>(reinterpret_cast<const uint4 *>(pool_dev),
                                 reinterpret_cast<uint4 *>(slots), fills, ctr, entry_bytes / 16,
                                 E);
}

// ---------------------------------------------------------------------------------------
// Decode gate/up GEMV + SwiGLU.  CTA (feature block, work item): 8 warps, one output
// feature j per warp; the warp streams W_gate row j and W_up row j once (16-byte loads,
// 8 per lane in flight per row) and dots them with the item's <= 16 token rows staged in
// shared memory.  h[q][j] = silu(g) * u, rounded to bf16.
// ---------------------------------------------------------------------------------------
constexpr int kGemvWarps = 8;
constexpr int kNB = 8;  // 16-byte chunks per lane per row per batch

template <int MAXT>
__global__ void __launch_bounds__(kGemvWarps * 32) k_gateup_gemv(
    const WorkItem *__restrict__ work, const DevCounters *__restrict__ ctr,
    const uint16_t *__restrict__ x, const int32_t *__restrict__ tok, uint16_t *__restrict__ h,
    int d, int d_ff) {
  const int u = blockIdx.y;
  if (u >= ctr->n_work) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = blockIdx.x * kGemvWarps + warp;
  if (j >= d_ff) return;
  const WorkItem wi = work[u];
  const int c = min(wi.count, MAXT);
  const int nchunk = d >> 3;
  const uint4 *xr[MAXT];  // the item's token rows (read through L1: shared by the CTA's warps)
#pragma unroll
  for (int t = 0; t < MAXT; ++t)
    xr[t] = reinterpret_cast<const uint4 *>(x + (size_t)(t < c ? tok[wi.q0 + t] : 0) * d);
  const uint16_t *grow = wi.W + (size_t)j * d;
  const uint16_t *urow = wi.W + (size_t)(d_ff + j) * d;
  float ag[MAXT], au[MAXT];
#pragma unroll
  for (int t = 0; t < MAXT; ++t) ag[t] = au[t] = 0.f;
  for (int cb = 0; cb < nchunk; cb += 32 * kNB) {
    uint4 gv[kNB], uv[kNB];
#pragma unroll
    for (int b = 0; b < kNB; ++b) {
      const int ch = cb + b * 32 + lane;
      gv[b] = ch < nchunk ? ld_stream(grow + (size_t)ch * 8) : make_uint4(0, 0, 0, 0);
      uv[b] = ch < nchunk ? ld_stream(urow + (size_t)ch * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int b = 0; b < kNB; ++b) {
      const int ch = cb + b * 32 + lane;
      if (ch < nchunk) {
#pragma unroll
        for (int t = 0; t < MAXT; ++t) {
          if (t < c) {
            const uint4 xv = __ldg(xr[t] + ch);
            ag[t] = dot8_seq(gv[b], xv, ag[t]);
            au[t] = dot8_seq(uv[b], xv, au[t]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < MAXT; ++t) {
    if (t < c) {
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        ag[t] += __shfl_xor_sync(0xffffffffu, ag[t], off);
        au[t] += __shfl_xor_sync(0xffffffffu, au[t], off);
      }
      if (lane == t) h[(size_t)(wi.q0 + t) * d_ff + j] = f32_to_bf16(silu_mul(ag[t], au[t]));
    }
  }
}

void launch_gateup_gemv(const WorkItem *work, const DevCounters *ctr, int max_work,
                        const uint16_t *x, const int32_t *tok, uint16_t *h, int T, int d,
                        int d_ff, cudaStream_t s) {
  dim3 grid((d_ff + kGemvWarps - 1) / kGemvWarps, max_work);
  if (T <= 1)
    k_gateup_gemv<1><<<grid, kGemvWarps * 32, 0, s>>>(work, ctr, x, tok, h, d, d_ff);
  else if (T <= 4)
    k_gateup_gemv<4><<<grid, kGemvWarps * 32, 0, s>>>(work, ctr, x, tok, h, d, d_ff);
  else
    k_gateup_gemv<16><<<grid, kGemvWarps * 32, 0, s>>>(work, ctr, x, tok, h, d, d_ff);
}

// ---------------------------------------------------------------------------------------
// Decode down GEMV fused with the weighted combine.  One warp per output feature i: for
// every work item (ascending expert id, then the shared expert) it streams W_down row i,
// dots it with the item's h rows and adds w[q] * y into the accumulator of token tok[q],
// which lane tok[q] holds.  The sum over a token's experts therefore runs in a fixed order
// and the result is deterministic; out[t][i] = bf16(acc).
// ---------------------------------------------------------------------------------------
template <int MAXT>
__global__ void __launch_bounds__(kGemvWarps * 32) k_down_gemv(
    const WorkItem *__restrict__ work, const DevCounters *__restrict__ ctr,
    const uint16_t *__restrict__ h, const int32_t *__restrict__ tok, const float *__restrict__ wq,
    uint16_t *__restrict__ out, int T, int d, int d_ff) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * kGemvWarps + warp;
  if (i >= d) return;
  if (ctr->call_status != 0) return;
  const int n_work = ctr->n_work;
  const int nchunk = d_ff >> 3;
  float acc = 0.f;
  for (int u = 0; u < n_work; ++u) {
    const WorkItem wi = work[u];
    const uint16_t *row = wi.W + (size_t)2 * d_ff * d + (size_t)i * d_ff;
    const int c = min(wi.count, MAXT);
    float part[MAXT];
#pragma unroll
    for (int r = 0; r < MAXT; ++r) part[r] = 0.f;
    for (int cb = 0; cb < nchunk; cb += 32 * kNB) {
      uint4 wv[kNB];
#pragma unroll
      for (int b = 0; b < kNB; ++b) {
        const int ch = cb + b * 32 + lane;
        wv[b] = ch < nchunk ? ld_stream(row + (size_t)ch * 8) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int r = 0; r < MAXT; ++r) {
        if (r < c) {
          const uint4 *hr = reinterpret_cast<const uint4 *>(h + (size_t)(wi.q0 + r) * d_ff);
#pragma unroll
          for (int b = 0; b < kNB; ++b) {
            const int ch = cb + b * 32 + lane;
            if (ch < nchunk) part[r] = dot8_seq(wv[b], __ldg(hr + ch), part[r]);
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < MAXT; ++r) {
      if (r < c) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) part[r] += __shfl_xor_sync(0xffffffffu, part[r], off);
        const int q = wi.q0 + r;
        if (lane == tok[q]) acc = fmaf(wq[q], part[r], acc);
      }
    }
  }
  if (lane < T) out[(size_t)lane * d + i] = f32_to_bf16(acc);
}

void launch_down_gemv(const WorkItem *work, const DevCounters *ctr, int max_work,
                      const uint16_t *h, const int32_t *tok, const float *wq, uint16_t *out, int T,
                      int d, int d_ff, cudaStream_t s) {
  (void)max_work;
  dim3 grid((d + kGemvWarps - 1) / kGemvWarps);
  if (T <= 1)
    k_down_gemv<1><<<grid, kGemvWarps * 32, 0, s>>>(work, ctr, h, tok, wq, out, T, d, d_ff);
  else if (T <= 4)
    k_down_gemv<4><<<grid, kGemvWarps * 32, 0, s>>>(work, ctr, h, tok, wq, out, T, d, d_ff);
  else
    k_down_gemv<16><<<grid, kGemvWarps * 32, 0, s>>>(work, ctr, h, tok, wq, out, T, d, d_ff);
}

// ---------------------------------------------------------------------------------------
// Larger T: gather the permuted activation rows, grouped GEMMs, fp32 combine, cast.
// ---------------------------------------------------------------------------------------
__global__ void k_gather_rows(const uint16_t *__restrict__ x, const int32_t *__restrict__ tok,
                              uint16_t *__restrict__ xp, int rows, int d) {
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
                        cudaStream_t s) {
  if (rows <= 0) return;
  const size_t n = (size_t)rows * (d >> 3);
  const int threads = 256;
  const unsigned blocks = (unsigned)std::min<size_t>((n + threads - 1) / threads, 148 * 16);
  k_gather_rows<<<blocks, threads, 0, s>>>(x, tok, xp, rows, d);
}

// CUDA-core tiled GEMM, 64 x 64 output tile, K step 32, 4 x 4 outputs per thread.
// GATEUP: h[q][j] = silu(xp[q] . Wg[j]) * (xp[q] . Wu[j])          (K = d)
// DOWN:   acc[tok[q]][i] += wq[q] * (h[q] . Wd[i])  (fp32 atomics)  (K = d_ff)
constexpr int kTM = 64, kTN = 64, kTK = 32;

template <bool GATEUP>
__global__ void __launch_bounds__(256) k_gemm_simt(const WorkItem *__restrict__ work,
                                                   const DevCounters *__restrict__ ctr,
                                                   const uint16_t *__restrict__ A,
                                                   uint16_t *__restrict__ h,
                                                   const int32_t *__restrict__ tok,
                                                   const float *__restrict__ wq,
                                                   float *__restrict__ acc, int d, int d_ff) {
  const int u = blockIdx.z;
  if (u >= ctr->n_work) return;
  if (ctr->call_status != 0) return;
  const WorkItem wi = work[u];
  const int m0 = blockIdx.y * kTM;
  if (m0 >= wi.count) return;
  const int n0 = blockIdx.x * kTN;
  const int K = GATEUP ? d : d_ff;
  const int Nout = GATEUP ? d_ff : d;
  if (n0 >= Nout) return;
  const uint16_t *B0 = GATEUP ? wi.W : wi.W + (size_t)2 * d_ff * d;  // rows [Nout][K]
  const uint16_t *B1 = wi.W + (size_t)d_ff * d;                        // W_up rows (GATEUP)
  __shared__ float As[kTK][kTM + 4];
  __shared__ float Bs[kTK][kTN + 4];
  __shared__ float Us[GATEUP ? kTK : 1][kTN + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float cg[4][4] = {}, cu[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += kTK) {
    for (int i = threadIdx.x; i < kTM * kTK; i += 256) {
      const int r = i / kTK, kk = i % kTK;
      const int m = m0 + r;
      As[kk][r] = (m < wi.count) ? bf16_to_f32(A[(size_t)(wi.q0 + m) * K + k0 + kk]) : 0.f;
      const int n = n0 + r;
      Bs[kk][r] = (n < Nout) ? bf16_to_f32(B0[(size_t)n * K + k0 + kk]) : 0.f;
      if (GATEUP) Us[kk][r] = (n < Nout) ? bf16_to_f32(B1[(size_t)n * K + k0 + kk]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kTK; ++kk) {
      float a[4], b[4], bu[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b[i] = Bs[kk][tx * 4 + i];
        if (GATEUP) bu[i] = Us[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          cg[i][j] = fmaf(a[i], b[j], cg[i][j]);
          if (GATEUP) cu[i][j] = fmaf(a[i], bu[j], cu[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= wi.count) continue;
    const int q = wi.q0 + m;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= Nout) continue;
      if (GATEUP)
        h[(size_t)q * d_ff + n] = f32_to_bf16(silu_mul(cg[i][j], cu[i][j]));
      else
        atomicAdd(&acc[(size_t)tok[q] * d + n], wq[q] * cg[i][j]);
    }
  }
}

void launch_gemm_gateup(const WorkItem *work, const DevCounters *ctr, int max_work, int max_rows,
                        const uint16_t *xp, uint16_t *h, int d, int d_ff, cudaStream_t s) {
  const unsigned my = (unsigned)((max_rows + kTM - 1) / kTM);
  dim3 g1((d_ff + kTN - 1) / kTN, my, max_work);
  k_gemm_simt<true><<<g1, 256, 0, s>>>(work, ctr, xp, h, nullptr, nullptr, nullptr, d, d_ff);
}

void launch_gemm_down(const WorkItem *work, const DevCounters *ctr, int max_work, int max_rows,
                      const uint16_t *h, const int32_t *tok, const float *wq, float *acc, int d,
                      int d_ff, cudaStream_t s) {
  const unsigned my = (unsigned)((max_rows + kTM - 1) / kTM);
  dim3 g2((d + kTN - 1) / kTN, my, max_work);
  k_gemm_simt<false><<<g2, 256, 0, s>>>(work, ctr, h, nullptr, tok, wq, acc, d, d_ff);
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
