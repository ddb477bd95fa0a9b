// Routing (router logits + top-k + gates) for callers that cannot allocate device memory.
//
// The regular path keeps the router logits in scratch that ft_moe_create allocates.  Some
// callers cannot allocate at all: code that runs while a global-mode stream capture is open
// (cudaMalloc is refused there), serving loops that must never pay for an allocation (which
// can synchronise the device), and host frameworks that own all device memory through their
// own pool and forbid side allocations.  For them ft_route_topk_noalloc keeps its scratch in a
// fixed array compiled into this library instead.
//
// The scratch lives in the file-scope array below.  Every GPU that loads the library holds it
// (1 MiB) until the process exits.  Host code cannot pass the array's name to a kernel: on the
// host that name is only a stand-in, not a device address.  So a call asks the runtime for the
// array's device address on the current device (cudaGetSymbolAddress) whenever its stream is
// not capturing, and keeps it per device; a call on a capturing stream uses the kept address,
// so the first call on each device must come before any stream capture.  Looking the address
// up again on every uncaptured call keeps it right after cudaDeviceReset or a new context.
//
// All calls share the one array, which keeps the previous call's logits; a call overwrites all
// T*E logits it reads, so nothing needs to start at zero.  Calls that overlap on the GPU (on
// different streams, or from different threads) race on the array and may return each
// other's results: order them.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "ft_moe.h"
#include "internal.h"

namespace {

constexpr size_t kMaxLogits = (size_t)1 << 18;  // T * E <= 262,144 fp32 values (1 MiB)
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_route_scratch[kMaxLogits];

std::mutex g_mu;
float *g_scratch_addr[kMaxDevices] = {};

// Device address of g_route_scratch on the current device: looked up again when `s` is not
// capturing (the runtime call may load the module, which a capture forbids), else the address
// kept from the last uncaptured call on this device.
int scratch_address(cudaStream_t s, float **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return ftm::report_error(FT_ERR_CUDA, "cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices)
    return ftm::report_error(FT_ERR_INVALID, "device index out of range", cudaSuccess);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return ftm::report_error(FT_ERR_CUDA, "cudaStreamIsCapturing", e);
  std::lock_guard<std::mutex> lock(g_mu);
  if (cs == cudaStreamCaptureStatusNone) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess)
      return ftm::report_error(FT_ERR_CUDA, "cudaGetSymbolAddress(routing scratch)", e);
    g_scratch_addr[dev] = static_cast<float *>(p);
  } else if (!g_scratch_addr[dev]) {
    return ftm::report_error(FT_ERR_STATE,
                             "the first routing call on a device must come before any stream "
                             "capture (it looks up the scratch address)",
                             cudaSuccess);
  }
  *out = g_scratch_addr[dev];
  return FT_OK;
}

}  // namespace

extern "C" int ft_route_topk_noalloc(const void *x, const void *Wr, const float *bias, int T,
                                     int E, int d, int k, int32_t *idx, float *w, uint8_t *tie,
                                     ft_stream_t stream) {
  if (!x || !Wr || !idx || !w || !tie)
    return ftm::report_error(FT_ERR_INVALID, "x, Wr, idx, w and tie must not be NULL",
                             cudaSuccess);
  if (T < 1 || E < 1 || E > ftm::kMaxE || k < 1 || k > E || k > ftm::kMaxK || d < 8 || d % 8)
    return ftm::report_error(FT_ERR_INVALID,
                             "need T >= 1, 1 <= k <= E <= 1024, k <= 32, d a multiple of 8",
                             cudaSuccess);
  if ((size_t)T * (size_t)E > kMaxLogits)
    return ftm::report_error(FT_ERR_INVALID,
                             "T * E exceeds the fixed routing scratch of 262144 logits",
                             cudaSuccess);
  if ((((uintptr_t)x) | ((uintptr_t)Wr)) & 15)
    return ftm::report_error(FT_ERR_INVALID, "x and Wr must be 16-byte aligned", cudaSuccess);
  float *scratch = nullptr;
  cudaStream_t s = (cudaStream_t)stream;
  if (int r = scratch_address(s, &scratch)) return r;
  ftm::launch_router(static_cast<const uint16_t *>(x), static_cast<const uint16_t *>(Wr), bias,
                     scratch, T, E, d, s);
  ftm::launch_topk(scratch, idx, w, tie, T, E, k, s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return ftm::report_error(FT_ERR_CUDA, "routing launch", e);
  return FT_OK;
}
