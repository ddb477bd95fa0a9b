// GPU implementation of the seeded input generator defined in ft_synth/__init__.py
// (splitmix64 counters, Irwin-Hall sum of 12 uniforms, one fp32 multiply by sigma, bf16
// round to nearest even).  Integer arithmetic only, so it reproduces the host generator bit
// for bit.  Used to fill multi-GB expert pools quickly; holds none of the layer's arithmetic.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kG = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint16_t gen_one(uint64_t key, uint64_t i, float sigma) {
  int tot = 0;
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const uint64_t s = mix64(key + (3 * i + j + 1) * kG);
    tot += (int)(s & 0xFFFF) + (int)((s >> 16) & 0xFFFF) + (int)((s >> 32) & 0xFFFF) +
           (int)(s >> 48);
  }
  float z = (float)(tot - 393210) / 65536.0f;  // exact
  if (sigma != 1.0f) z = __fmul_rn(sigma, z);
  uint32_t u = __float_as_uint(z);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

// keys[k] generates dst[k * per_key + i], i in [start, start + n).
__global__ void k_gen(const uint64_t *__restrict__ keys, int n_keys, uint64_t per_key,
                      uint64_t start, uint64_t n, float sigma, uint16_t *__restrict__ dst) {
  const uint64_t total = (uint64_t)n_keys * n;
  for (uint64_t t = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; t * 8 < total;
       t += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t g0 = t * 8;
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const uint64_t g = g0 + v;
      if (g >= total) break;
      const uint64_t k = g / n, i = g - k * n;
      dst[k * per_key + i] = gen_one(keys[k], start + i, sigma);
    }
  }
}

// 4-bit entries (ft_synth.expert_entry_fp4): entry k is `nc` code bytes (the little-endian
// bytes of draws 0 .. nc/8 - 1 of keys[k]) then `ns` scale bytes (118 + draw(nc/8 + j) % 3).
__global__ void k_gen_fp4(const uint64_t *__restrict__ keys, int n_keys, uint64_t nc,
                          uint64_t ns, uint8_t *__restrict__ dst) {
  const uint64_t per = nc + ns, nd = nc / 8, units = nd + ns;
  const uint64_t total = (uint64_t)n_keys * units;
  for (uint64_t t = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t k = t / units, i = t - k * units;
    const uint64_t v = mix64(keys[k] + (i + 1) * kG);
    if (i < nd)
      *reinterpret_cast<uint64_t *>(dst + k * per + 8 * i) = v;  // little-endian bytes
    else
      dst[k * per + nc + (i - nd)] = (uint8_t)(118 + v % 3);
  }
}

}  // namespace

extern "C" {

// Fill a host buffer with n_keys consecutive 4-bit entries (nc code bytes + ns scale bytes
// each, nc a multiple of 16), staged through two device buffers like fts_fill_host.
int fts_fill_host_fp4(const uint64_t *keys_host, int n_keys, uint64_t nc, uint64_t ns,
                      void *dst_host, int stage_entries) {
  if (n_keys <= 0) return 0;
  if (stage_entries < 1) stage_entries = 1;
  const uint64_t per = nc + ns;
  cudaStream_t st[2];
  uint8_t *buf[2] = {nullptr, nullptr};
  uint64_t *dk = nullptr;
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaStreamCreate(&st[i]);
  for (int i = 0; i < 2 && e == cudaSuccess; ++i)
    e = cudaMalloc(&buf[i], (size_t)stage_entries * per);
  if (e == cudaSuccess) e = cudaMalloc(&dk, (size_t)n_keys * 8);
  if (e == cudaSuccess) e = cudaMemcpy(dk, keys_host, (size_t)n_keys * 8, cudaMemcpyHostToDevice);
  for (int c = 0, it = 0; e == cudaSuccess && c < n_keys; c += stage_entries, ++it) {
    const int b = it & 1;
    const int m = (n_keys - c) < stage_entries ? (n_keys - c) : stage_entries;
    k_gen_fp4<<<148 * 8, 256, 0, st[b]>>>(dk + c, m, nc, ns, buf[b]);
    e = cudaGetLastError();
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(static_cast<uint8_t *>(dst_host) + (size_t)c * per, buf[b],
                          (size_t)m * per, cudaMemcpyDeviceToHost, st[b]);
  }
  for (int i = 0; i < 2; ++i) {
    cudaError_t e2 = cudaStreamSynchronize(st[i]);
    if (e == cudaSuccess) e = e2;
  }
  for (int i = 0; i < 2; ++i) {
    if (buf[i]) cudaFree(buf[i]);
    cudaStreamDestroy(st[i]);
  }
  if (dk) cudaFree(dk);
  return (int)e;
}


// Generate n_keys streams of `n` bf16 values each (elements start..start+n-1) into device
// memory dst_dev, stream k at dst_dev + k * per_key.  Returns a cudaError_t value.
int fts_generate_device(const uint64_t *keys_host, int n_keys, uint64_t per_key, uint64_t start,
                        uint64_t n, float sigma, void *dst_dev, cudaStream_t s) {
  uint64_t *dk = nullptr;
  cudaError_t e = cudaMallocAsync(&dk, (size_t)n_keys * 8, s);
  if (e != cudaSuccess) return (int)e;
  e = cudaMemcpyAsync(dk, keys_host, (size_t)n_keys * 8, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) {
    k_gen<<<148 * 8, 256, 0, s>>>(dk, n_keys, per_key, start, n, sigma,
                                   static_cast<uint16_t *>(dst_dev));
    e = cudaGetLastError();
  }
  cudaFreeAsync(dk, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return (int)e;
}

// Fill a host buffer (pinned for speed) with n_keys consecutive entries of per_key values
// each, entry k generated from keys_host[k]; staged through two device buffers of
// `stage_entries` entries so generation overlaps the device-to-host copies.
int fts_fill_host(const uint64_t *keys_host, int n_keys, uint64_t per_key, float sigma,
                  void *dst_host, int stage_entries) {
  if (n_keys <= 0) return 0;
  if (stage_entries < 1) stage_entries = 1;
  cudaStream_t st[2];
  uint16_t *buf[2] = {nullptr, nullptr};
  uint64_t *dk = nullptr;
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaStreamCreate(&st[i]);
  for (int i = 0; i < 2 && e == cudaSuccess; ++i)
    e = cudaMalloc(&buf[i], (size_t)stage_entries * per_key * 2);
  if (e == cudaSuccess) e = cudaMalloc(&dk, (size_t)n_keys * 8);
  if (e == cudaSuccess) e = cudaMemcpy(dk, keys_host, (size_t)n_keys * 8, cudaMemcpyHostToDevice);
  for (int c = 0, it = 0; e == cudaSuccess && c < n_keys; c += stage_entries, ++it) {
    const int b = it & 1;
    const int m = (n_keys - c) < stage_entries ? (n_keys - c) : stage_entries;
    k_gen<<<148 * 8, 256, 0, st[b]>>>(dk + c, m, per_key, 0, per_key, sigma, buf[b]);
    e = cudaGetLastError();
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(static_cast<uint16_t *>(dst_host) + (size_t)c * per_key, buf[b],
                          (size_t)m * per_key * 2, cudaMemcpyDeviceToHost, st[b]);
  }
  for (int i = 0; i < 2; ++i) {
    cudaError_t e2 = cudaStreamSynchronize(st[i]);
    if (e == cudaSuccess) e = e2;
  }
  for (int i = 0; i < 2; ++i) {
    if (buf[i]) cudaFree(buf[i]);
    cudaStreamDestroy(st[i]);
  }
  if (dk) cudaFree(dk);
  return (int)e;
}

}  // extern "C"
