// Grouped GEMMs of the expert FFN on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by tiled TMA, for calls with more tokens than the decode GEMVs handle (prefill).
//
//   gate/up:  H[q][j] = silu(X[q] . Wg[j]) * (X[q] . Wu[j])       (K = d)
//   down:     acc[tok[q]][i] += w[q] * (H[q] . Wd[i])              (K = d_ff)
//
// Rows q of X / H are the (token, expert) pairs grouped by expert (one work item per expert);
// each expert's weights come from one complete (layer, expert) entry: a cache slot, the
// prefill double buffer, or the shared-expert array (FreeToken RTX 4090, "how the MoE memory
// hierarchy works": an expert executes from its complete entry).
//
// Tile: M = 128 pair rows (TMEM lanes) x N = 256 accumulator columns, K in steps of 64 (one
// 128-byte swizzle row).  For gate/up the 256 B-rows of a tile are 128 W_gate rows followed by
// the same 128 W_up rows, so a thread's TMEM lane holds both halves of SwiGLU for 128 output
// features.  Warp roles: warp 0 issues TMA loads into a 4-stage ring, warp 1 allocates TMEM
// (2 x 256 columns: the epilogue of one tile overlaps the MMAs of the next) and issues
// tcgen05.mma, warps 2..5 drain TMEM.  Persistent CTAs (one per SM) walk the tile list; the
// M-tiles that share a weight block are consecutive, so the block is re-read from L2.  All
// waits are bounded (FT_ERR_TIMEOUT).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace ftm {

constexpr int kTcM = 128;
constexpr int kTcK = 64;
constexpr int kTcStages = 4;
constexpr int kTcThreads = 192;
constexpr uint32_t kTcA = kTcM * kTcK * 2;  // 16 KB

__device__ __forceinline__ float silu_mul_tc(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// prefix[u] = tiles of work items 0..u-1 (u = 0..n_work); tiles per item =
// ceil(count / 128) * n_blocks.
__global__ void k_tile_prefix(const WorkItem *__restrict__ work, const DevCounters *__restrict__ ctr,
                              int n_blocks, int *__restrict__ prefix) {
  if (threadIdx.x != 0) return;
  const int n = ctr->call_status ? 0 : ctr->n_work;
  int acc = 0;
  prefix[0] = 0;
  for (int u = 0; u < n; ++u) {
    acc += ((work[u].count + kTcM - 1) / kTcM) * n_blocks;
    prefix[u + 1] = acc;
  }
  prefix[kMaxE + 2] = n;  // n_work, read by the GEMM
}

struct TcArgs {
  const WorkItem *work;
  const int *prefix;  // [kMaxE + 3]; prefix[kMaxE + 2] = n_work
  DevCounters *ctr;
  int K;              // reduction length (d or d_ff)
  int n_blocks;       // N blocks per work item
  int rows_per_entry; // rows of one entry in the B view (3*d_ff for gate/up, 3*d for down)
  int b_row_off;      // first B row of the matrix inside an entry (0 or 2*d)
  int up_off;         // gate/up: row offset of W_up from W_gate (d_ff)
  int shared_entry;   // entry index of the shared expert in its array (layer)
  int by_item;        // 1: item u's weights are entry u of the B view (expanded MXFP4 scratch)
  int d, d_ff;
  uint16_t *h;        // gate/up output [rows][d_ff]
  const int32_t *tok; // down: token of each pair row
  const float *wq;    // down: gate weight of each pair row
  float *acc;         // down: fp32 [T][d]
};

__device__ __forceinline__ void decode_tile(const TcArgs &a, int n_work, int t, int &u, int &nb,
                                            int &mt, int &mtiles) {
  int lo = 0, hi = n_work - 1;
  while (lo < hi) {  // last u with prefix[u] <= t
    const int mid = (lo + hi + 1) >> 1;
    if (a.prefix[mid] <= t) lo = mid; else hi = mid - 1;
  }
  u = lo;
  const int local = t - a.prefix[u];
  mtiles = (a.work[u].count + kTcM - 1) / kTcM;
  nb = local / mtiles;
  mt = local - nb * mtiles;
}

template <bool GATEUP, int BN>
__global__ void __launch_bounds__(kTcThreads, 1)
    k_tc_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmBs, const TcArgs a) {
  constexpr uint32_t kB = (uint32_t)BN * kTcK * 2;
  constexpr uint32_t kStage = kTcA + kB;
  constexpr uint32_t kIdesc = idesc_bf16(kTcM, BN);
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~(uintptr_t)1023);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + kTcStages * kStage);
  uint64_t *empty = full + kTcStages;
  uint64_t *tfull = empty + kTcStages;
  uint64_t *tempty = tfull + 2;
  uint64_t *done = tempty + 2;
  uint32_t *tmem_base_p = reinterpret_cast<uint32_t *>(done + 1);
  int *abort_flag = reinterpret_cast<int *>(tmem_base_p + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_base_p, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_p;
  const int n_work = a.prefix[kMaxE + 2];
  const int n_tiles = n_work > 0 ? a.prefix[n_work] : 0;
  const int n_kb = a.K / kTcK;

  if (warp == 0) {
    if (lane == 0) {  // ---------------- TMA producer
      long it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
        int u, nb, mt, mtiles;
        decode_tile(a, n_work, t, u, nb, mt, mtiles);
        const WorkItem wi = a.work[u];
        const bool sh = wi.expert < 0;
        const int entry = sh ? a.shared_entry : (a.by_item ? u : wi.slot);
        const void *mapB = sh ? (const void *)&tmBs : (const void *)&tmB;
        const int row_a = wi.q0 + mt * kTcM;
        const int row_b = entry * a.rows_per_entry + a.b_row_off + nb * (GATEUP ? 128 : BN);
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int s = (int)(it % kTcStages);
          const uint32_t ph = (uint32_t)((it / kTcStages) & 1);
          if (it >= kTcStages && !mbar_wait(&empty[s], ph ^ 1u)) {
            ok = false;
            break;
          }
          uint8_t *sa = smem + s * kStage;
          uint8_t *sb = sa + kTcA;
          mbar_arrive_expect_tx(&full[s], kStage);
          tma_load_2d(sa, &tmA, kb * kTcK, row_a, &full[s]);
          if (GATEUP) {
            tma_load_2d(sb, mapB, kb * kTcK, row_b, &full[s]);
            tma_load_2d(sb + kB / 2, mapB, kb * kTcK, row_b + a.up_off, &full[s]);
          } else {
            tma_load_2d(sb, mapB, kb * kTcK, row_b, &full[s]);
          }
        }
      }
      if (!ok) *abort_flag = 1;
      for (long i = (it > kTcStages ? it - kTcStages : 0); i < it; ++i)
        mbar_wait(&full[i % kTcStages], (uint32_t)((i / kTcStages) & 1));
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---------------- MMA issuer
      long it = 0;
      int tc = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++tc) {
        const int acc_i = tc & 1;
        const uint32_t aph = (uint32_t)((tc >> 1) & 1);
        if (tc >= 2 && !mbar_wait(&tempty[acc_i], aph ^ 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc_i * 256);
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int s = (int)(it % kTcStages);
          const uint32_t ph = (uint32_t)((it / kTcStages) & 1);
          if (!mbar_wait(&full[s], ph)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * kStage);
          const uint64_t adesc = sw128_desc(sa);
          const uint64_t bdesc = sw128_desc(sa + kTcA);
#pragma unroll
          for (int ks = 0; ks < kTcK / 16; ++ks)
            umma_bf16(d_tmem, adesc + 2 * ks, bdesc + 2 * ks, kIdesc, (kb | ks) != 0);
          umma_commit(&empty[s]);
        }
        if (!ok) break;
        umma_commit(&tfull[acc_i]);
      }
      if (!ok) *abort_flag = 1;
      umma_commit(done);  // every MMA issued above has completed once this arrives
      mbar_wait(done, 0);
    }
  } else {  // ---------------- epilogue warps 2..5: TMEM lanes 32*(warp%4) ..
    const int quad = warp & 3;
    const int m = quad * 32 + lane;
    int tc = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++tc) {
      const int acc_i = tc & 1;
      const uint32_t aph = (uint32_t)((tc >> 1) & 1);
      if (!mbar_wait(&tfull[acc_i], aph)) {
        ok = false;
        break;
      }
      tc_fence_after();
      int u, nb, mt, mtiles;
      decode_tile(a, n_work, t, u, nb, mt, mtiles);
      const WorkItem wi = a.work[u];
      const int ql = mt * kTcM + m;
      const bool valid = ql < wi.count;
      const int q = wi.q0 + ql;
      const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc_i * 256);
      if (GATEUP) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], v[32];
          tmem_ld32(taddr + 32 * c, g);
          tmem_ld32(taddr + 128 + 32 * c, v);
          tmem_ld_wait();
          if (valid) {
            uint4 *dst = reinterpret_cast<uint4 *>(a.h + (size_t)q * a.d_ff + nb * 128 + 32 * c);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint32_t pk[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int e = 8 * i + 2 * j;
                const float h0 = silu_mul_tc(__uint_as_float(g[e]), __uint_as_float(v[e]));
                const float h1 = silu_mul_tc(__uint_as_float(g[e + 1]), __uint_as_float(v[e + 1]));
                pk[j] = (uint32_t)f32_to_bf16(h0) | ((uint32_t)f32_to_bf16(h1) << 16);
              }
              dst[i] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
          }
        }
      } else {
        const float wgt = valid ? a.wq[q] : 0.f;
        float *dst = valid ? a.acc + (size_t)a.tok[q] * a.d + nb * BN : nullptr;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t y[32];
          tmem_ld32(taddr + 32 * c, y);
          tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              red_add_v4(dst + 32 * c + 4 * i, wgt * __uint_as_float(y[4 * i]),
                         wgt * __uint_as_float(y[4 * i + 1]), wgt * __uint_as_float(y[4 * i + 2]),
                         wgt * __uint_as_float(y[4 * i + 3]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc_i]);
    }
    if (!ok && lane == 0) *abort_flag = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) set_status(a.ctr, FT_ERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// ---------------------------------------------------------------------------------------
// Host side: tensor maps and launches.
// ---------------------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 view [rows][inner] of `base`, box [box_rows][64], 128-byte swizzle.
bool make_tmap(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto enc = get_encode();
  if (!enc || !base) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kTcK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int tc_sms() {
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
static void tc_smem_attr(K kern, size_t smem) {
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

void launch_tc_ffn(const TcMaps &maps, const WorkItem *work, DevCounters *ctr, int *prefix,
                   uint16_t *h, const int32_t *tok, const float *wq, float *acc, int d, int d_ff,
                   int shared_entry, bool by_item, cudaStream_t s) {
  TcArgs a{};
  a.by_item = by_item ? 1 : 0;
  a.work = work;
  a.prefix = prefix;
  a.ctr = ctr;
  a.d = d;
  a.d_ff = d_ff;
  a.shared_entry = shared_entry;
  a.h = h;
  a.tok = tok;
  a.wq = wq;
  a.acc = acc;
  const int grid = tc_sms();
  // gate/up
  a.K = d;
  a.n_blocks = d_ff / 128;
  a.rows_per_entry = 3 * d_ff;
  a.b_row_off = 0;
  a.up_off = d_ff;
  k_tile_prefix<<<1, 32, 0, s>>>(work, ctr, a.n_blocks, prefix);
  {
    constexpr size_t smem = kTcStages * (kTcA + 256 * kTcK * 2) + 1024 + 256;
    tc_smem_attr(k_tc_gemm<true, 256>, smem);
    k_tc_gemm<true, 256><<<grid, kTcThreads, smem, s>>>(maps.a_x, maps.b_gu, maps.bs_gu, a);
  }
  // down
  a.K = d_ff;
  a.rows_per_entry = 3 * d;
  a.b_row_off = 2 * d;
  a.up_off = 0;
  if (d % 256 == 0) {
    a.n_blocks = d / 256;
    k_tile_prefix<<<1, 32, 0, s>>>(work, ctr, a.n_blocks, prefix);
    constexpr size_t smem = kTcStages * (kTcA + 256 * kTcK * 2) + 1024 + 256;
    tc_smem_attr(k_tc_gemm<false, 256>, smem);
    k_tc_gemm<false, 256><<<grid, kTcThreads, smem, s>>>(maps.a_h, maps.b_dn256, maps.bs_dn256, a);
  } else {
    a.n_blocks = d / 128;
    k_tile_prefix<<<1, 32, 0, s>>>(work, ctr, a.n_blocks, prefix);
    constexpr size_t smem = kTcStages * (kTcA + 128 * kTcK * 2) + 1024 + 256;
    tc_smem_attr(k_tc_gemm<false, 128>, smem);
    k_tc_gemm<false, 128><<<grid, kTcThreads, smem, s>>>(maps.a_h, maps.b_dn128, maps.bs_dn128, a);
  }
}

}  // namespace ftm
