// Expert-side kernels of calls with more tokens than the decode path takes: miss fills from
// the host pool, the gather of the permuted activation rows and the final cast (the grouped
// GEMMs themselves are in gemm_tc.cu; the decode path is decode.cu).
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

// ---------------------------------------------------------------------------------------
// MXFP4 entries for the grouped GEMMs: each work item's entry is expanded to bf16 in the
// scratch entry of the same index (the GEMMs then address their B rows by item).  The codes
// of W_gate, W_up and W_down are contiguous and so are their scales, one byte per 32-input
// block in the same order, so block b of the entry has its 16 code bytes at 16*b, its scale at
// (3*d*d_ff/2) + b and its 32 outputs at 32*b: out = e2m1(code) * 2^(scale - 127), exact in
// bf16 (input 2i of a block is the low nibble of byte i).
// ---------------------------------------------------------------------------------------
__global__ void k_dequant_work(const WorkItem *__restrict__ work, const DevCounters *__restrict__ ctr,
                               uint16_t *__restrict__ scratch, size_t entry_elems, size_t n_blocks) {
  if (ctr->call_status != 0) return;
  const int n_work = ctr->n_work;
  const size_t total = (size_t)n_work * n_blocks;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int u = (int)(i / n_blocks);
    const size_t b = i - (size_t)u * n_blocks;
    const uint8_t *src = reinterpret_cast<const uint8_t *>(work[u].W);
    const uint4 q = __ldg(reinterpret_cast<const uint4 *>(src) + b);
    const float sc = e8m0_f32(src[16 * n_blocks + b]);  // the scale region follows the codes
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    uint4 *dst = reinterpret_cast<uint4 *>(scratch + (size_t)u * entry_elems + 32 * b);
#pragma unroll
    for (int v = 0; v < 4; ++v) {  // 8 inputs per code word -> one uint4 of bf16
      uint32_t o[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const float lo = e2m1_f32(w[v] >> (8 * p)) * sc, hi = e2m1_f32(w[v] >> (8 * p + 4)) * sc;
        o[p] = (uint32_t)f32_to_bf16(lo) | ((uint32_t)f32_to_bf16(hi) << 16);
      }
      dst[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

void launch_dequant_work(const WorkItem *work, const DevCounters *ctr, uint16_t *scratch, int d,
                         int d_ff, int max_items, cudaStream_t s) {
  const size_t n_blocks = (size_t)3 * d * d_ff / 32;
  const size_t total = (size_t)max_items * n_blocks;
  const unsigned blocks = (unsigned)std::min<size_t>((total + 255) / 256, 148 * 16);
  k_dequant_work<<<blocks, 256, 0, s>>>(work, ctr, scratch, (size_t)3 * d * d_ff, n_blocks);
}

// out = bf16(acc); with `next`, also the residual stream's next layer input
// next = bf16(x + out) (an fp32 add of the two bf16 values, then round to nearest even).
// 8 elements per thread (n % 8 == 0).
__global__ void k_cast_out(const float *__restrict__ acc, uint16_t *__restrict__ out, size_t n,
                           const uint16_t *__restrict__ x, uint16_t *__restrict__ next,
                           const DevCounters *__restrict__ ctr) {
  if (ctr->call_status != 0) return;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n / 8;
       i += (size_t)gridDim.x * blockDim.x) {
    const float4 a0 = reinterpret_cast<const float4 *>(acc)[2 * i];
    const float4 a1 = reinterpret_cast<const float4 *>(acc)[2 * i + 1];
    const float v[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    uint16_t o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = f32_to_bf16(v[j]);
    uint4 ov;
    ov.x = (uint32_t)o[0] | ((uint32_t)o[1] << 16);
    ov.y = (uint32_t)o[2] | ((uint32_t)o[3] << 16);
    ov.z = (uint32_t)o[4] | ((uint32_t)o[5] << 16);
    ov.w = (uint32_t)o[6] | ((uint32_t)o[7] << 16);
    reinterpret_cast<uint4 *>(out)[i] = ov;
    if (next) {
      const uint4 xv = reinterpret_cast<const uint4 *>(x)[i];
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
      uint32_t nw[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float s0 = bf16_to_f32((uint16_t)(xw[j] & 0xFFFFu)) + bf16_to_f32(o[2 * j]);
        const float s1 = bf16_to_f32((uint16_t)(xw[j] >> 16)) + bf16_to_f32(o[2 * j + 1]);
        nw[j] = (uint32_t)f32_to_bf16(s0) | ((uint32_t)f32_to_bf16(s1) << 16);
      }
      reinterpret_cast<uint4 *>(next)[i] = make_uint4(nw[0], nw[1], nw[2], nw[3]);
    }
  }
}

void launch_cast_out(const float *acc, uint16_t *out, size_t n, const uint16_t *x, uint16_t *next,
                     const DevCounters *ctr, cudaStream_t s) {
  if (n == 0) return;
  const unsigned blocks = (unsigned)std::min<size_t>((n / 8 + 255) / 256, 148 * 8);
  k_cast_out<<<blocks, 256, 0, s>>>(acc, out, n, x, next, ctr);
}

}  // namespace ftm
