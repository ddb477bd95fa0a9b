// Shared definitions of the ft_moe CUDA library (device state layout, small helpers).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ft_moe.h"

namespace ftm {

// Launch `kern` on `s` with programmatic stream serialization, so it may begin while the
// previous kernel on the stream finishes; the kernel calls pdl_wait() before reading that
// kernel's results.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

constexpr int kMaxE = 1024;        // experts per layer
constexpr int kMaxK = 32;          // routed experts per token
constexpr int kGemvMaxTokens = 16; // forward calls with T <= this use the GEMV kernels
constexpr double kNearTie = 1e-6;  // top-k gap reported as a near-tie (exact fp32 difference)
// Default limit of a cross-CTA wait in the decode expert kernel.  The longest legitimate wait
// is for the last fill of a call, behind every other fill of that call over the host link
// (about 0.1 s for 96 misses of 50 MB); a wait that runs out records FT_ERR_TIMEOUT.
constexpr unsigned long long kDefaultWaitNs = 4000000000ull;

// Device counters and the status word.  One instance per handle, in device memory.
struct DevCounters {
  unsigned long long calls, hits, misses, fill_bytes, evictions, near_ties;
  unsigned long long tick;       // global LRU clock
  unsigned long long bypasses;   // misses staged without entering the cache (admission)
  unsigned long long acc;        // admission: accesses since the counts were last halved
  int status;                    // first device-side error (FT_ERR_*), 0 = none
  int n_fill;                    // fills of the most recent forward call
  int n_work;                    // work items of the most recent call
  int occupied;                  // slots holding an entry
  int call_status;               // 0, or FT_ERR_CAPACITY if the current call was refused
  unsigned route_arrive;         // CTAs of the fused routing kernel that have finished
  int n_hit;                     // work items 0 .. n_hit-1 are cached hits; the n_fill
                                 // misses follow (item n_hit + m uses fill m), then the
                                 // shared expert
  int hold_fills;                // debug: the decode expert kernel never reports its fills
                                 // done, so its waits for them run out (timeout tests)
  int pad;
  unsigned long long wait_ns;    // limit of every cross-CTA wait of the decode expert kernel
};

// Where the cache's slot state lives.  Kept in device memory and read by the kernels on
// every call, so that a graph captured before ft_cache_resize (which reallocates the slot
// storage) stays valid after it.
struct CacheDesc {
  uint16_t *slots;              // [n_slots][entry]
  int32_t *owner;               // [n_slots]
  unsigned long long *stamps;   // [n_slots]
  int n_slots;
  int pad;
};

// One group of rows of the expert FFN: the rows q0 .. q0+count-1 of the permuted
// activations all use the weights of one complete entry W (W_gate | W_up | W_down).
struct WorkItem {
  const uint16_t *W;
  int q0;
  int count;
  int expert;  // expert id, or -1 for the shared expert
  int slot;    // cache slot (decode), expert id (prefill buffer) or -1 (shared)
};

// Arguments of the routing/control stage for one call.
struct ControlArgs {
  const int32_t *idx;   // [T][k]
  const float *w;       // [T][k]
  const uint8_t *tie;   // [T]
  int T, k, E, P;       // P = T*k
  int d;                // hidden size (fused decode routing)
  int layer, L;
  int32_t *counts;      // [E]
  int32_t *offsets;     // [E+1]
  int32_t *perm;        // [P]
  int32_t *inv;         // [P]
  int32_t *tok;         // [P + T] token of FFN row q
  float *wq;            // [P + T] gate weight of FFN row q
  WorkItem *work;       // [E + 1]
  // cache (decode mode); null slot_table selects prefill mode
  int32_t *slot_table;  // [L][E]
  const CacheDesc *cache;      // slot storage, owners, stamps, capacity (device)
  int32_t *fills;       // [max_fill][3]
  uint32_t *freq;       // admission counts [L][E], or null for the plain LRU
  int32_t *sync;        // decode expert kernel counters, zeroed here ([n_sync])
  int n_sync;
  const uint16_t *buffer;      // prefill: E entries of this layer
  const uint16_t *shared;      // shared entry of this layer or null
  size_t entry_elems;
  DevCounters *ctr;
};

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

// Round to nearest even (no NaNs arise on this path).
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

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

// Programmatic dependent launch: let the next kernel on the stream start launching now, and
// wait here until the previous kernel has completed and its writes are visible.  Both are
// no-ops for kernels launched without the programmatic-serialization attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Pull one line of global memory into L2 (no register result).
__device__ __forceinline__ void prefetch_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void set_status(DevCounters *c, int code) {
  atomicCAS(&c->status, 0, code);
}

// Streaming 16-byte load that bypasses L1 allocation (weights are read once).  Not volatile:
// the data is read-only for the kernel's lifetime, so the compiler may hoist these loads and
// keep many in flight.
__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// Dot of 8 bf16 pairs packed in two uint4, accumulated sequentially in feature order.
__device__ __forceinline__ float dot8_seq(uint4 a, uint4 b, float acc) {
  const uint32_t av[4] = {a.x, a.y, a.z, a.w};
  const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc = fmaf(__uint_as_float(av[i] << 16), __uint_as_float(bv[i] << 16), acc);
    acc = fmaf(__uint_as_float(av[i] & 0xFFFF0000u), __uint_as_float(bv[i] & 0xFFFF0000u), acc);
  }
  return acc;
}

}  // namespace ftm
