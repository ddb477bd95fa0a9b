// ft_moe C ABI: handle lifetime, pool attachment, the per-layer forward, prefill with
// full-layer double buffering, elastic resize and counters.  See include/ft_moe.h.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <numeric>
#include <string>
#include <vector>

#include "ft_moe.h"
#include "internal.h"

using namespace ftm;

namespace {

thread_local std::string g_err;

int fail(int code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

#define FT_CUDA(call)                                                                   \
  do {                                                                                  \
    cudaError_t e_ = (call);                                                            \
    if (e_ != cudaSuccess)                                                              \
      return fail(e_ == cudaErrorMemoryAllocation ? FT_ERR_OOM : FT_ERR_CUDA, "%s: %s (%s:%d)", \
                  #call, cudaGetErrorString(e_), __FILE__, __LINE__);                   \
  } while (0)

bool inject(const char *what) {
  const char *v = getenv("FT_FAULT_INJECT");
  return v && strstr(v, what) != nullptr;
}

}  // namespace

int ftm::report_error(int code, const char *what, cudaError_t e) {
  if (e != cudaSuccess) return fail(code, "%s: %s", what, cudaGetErrorString(e));
  return fail(code, "%s", what);
}

struct ft_moe {
  int L = 0, E = 0, k = 0, d = 0, d_ff = 0, n_slots = 0, max_tokens = 0, n_shared = 0;
  int prewarm = 1, debug = 0;
  size_t entry_elems = 0, entry_bytes = 0;
  int device = 0;
  std::vector<void *> allocs;  // fixed-size device allocations

  uint16_t *wr = nullptr;  // [L][E][d]
  float *bias = nullptr;   // [L][E]
  std::vector<char> has_bias;
  uint16_t *shared = nullptr;  // [L][entry]
  uint16_t *slots = nullptr;   // [n_slots][entry]
  int32_t *slot_table = nullptr;
  int32_t *owner = nullptr;
  unsigned long long *stamps = nullptr;
  DevCounters *ctr = nullptr;
  CacheDesc *cache = nullptr;  // device copy of {slots, owner, stamps, n_slots}
  float *logits = nullptr;
  int32_t *idx = nullptr;
  float *w = nullptr;
  uint8_t *tie = nullptr;
  int32_t *counts = nullptr, *offsets = nullptr, *perm = nullptr, *inv = nullptr;
  int32_t *tok = nullptr;
  float *wq = nullptr;
  WorkItem *work = nullptr;
  int32_t *fills = nullptr;
  uint16_t *hbuf = nullptr;
  uint16_t *xp = nullptr;
  float *acc = nullptr;
  float *ybuf = nullptr;  // decode: fp32 rows of the down projection [(16k + 16)][d]
  int32_t *sync = nullptr;  // decode expert kernel completion counters [kSyncInts(d)]
  int32_t *chunk = nullptr;
  int *tile_prefix = nullptr;  // tcgen05 tile scheduler [kMaxE + 3]
  TcMaps maps_slots{};         // tensor maps over the slot storage
  TcMaps maps_dbuf[2]{};       // ... over the prefill double buffer
  uint16_t *fp4_scratch = nullptr;  // MXFP4 entries expanded to bf16 for the grouped GEMMs [E]
  TcMaps maps_fp4{};                // ... and its tensor maps
  uint64_t resizes = 0;

  // pool
  const uint16_t *pool_host = nullptr;
  const uint16_t *pool_dev = nullptr;
  size_t pool_bytes = 0;
  bool pool_registered = false;

  // prefill
  uint16_t *dbuf[2] = {nullptr, nullptr};
  uint16_t *chain[2] = {nullptr, nullptr};  // residual stream inputs of layers 1.. [max_tokens][d]
  cudaStream_t copy_stream = nullptr;
  std::vector<cudaEvent_t> ev_cs, ev_ce, ev_ks, ev_ke;  // copy start/end, compute start/end
  int last_prefill_layers = 0;
  int prefill_topup = 0;
  int admission = 0;          // frequency admission (see ft_moe_opts)
  bool fp4 = false;           // MXFP4 entries (decode calls only)
  int n_stage = 0;            // staging entries after the slots: E with admission, else 0
  uint32_t *freq = nullptr;   // admission counts [L][E]
  uint64_t last_h2d_bytes = 0, last_d2d_bytes = 0;  // moved by the last prefill
  std::vector<int32_t> table_host;                  // slot table read by the top-up

  // host staging for decode_host
  uint16_t *xstage = nullptr, *ostage = nullptr;
  size_t xstage_bytes = 0, ostage_bytes = 0;

  // most recent call, for the debug getters
  int last_T = 0;
  cudaStream_t last_stream = nullptr;

  // kernel timing (ft_moe_profile)
  bool prof_on = false;
  bool prof_keep = false;                     // graph mode: keep the recorded pairs
  std::vector<cudaEvent_t> prof_events;       // pool; pairs (begin, end)
  std::vector<int> prof_class;                // class of pair i
  int32_t *prof_rec = nullptr;                // device [pairs][2]: (n_fill, n_work) of the
                                              // call of a decode expert launch
  size_t prof_rec_cap = 0;
  int64_t prof_items[FT_PROF_N] = {};
  double prof_ms[FT_PROF_N] = {};
  int64_t prof_n[FT_PROF_N] = {};
};

namespace {

int dev_alloc(ft_moe *h, void **p, size_t bytes) {
  if (bytes == 0) bytes = 16;
  if (inject("create_alloc")) return fail(FT_ERR_OOM, "injected allocation failure");
  cudaError_t e = cudaMalloc(p, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(FT_ERR_OOM, "cudaMalloc(%zu) failed: %s", bytes, cudaGetErrorString(e));
  }
  h->allocs.push_back(*p);
  return FT_OK;
}

template <typename T>
int alloc_n(ft_moe *h, T **p, size_t n) {
  return dev_alloc(h, reinterpret_cast<void **>(p), n * sizeof(T));
}

// Sum the recorded event pairs into prof_ms / prof_n and clear the record (in graph mode
// the pairs are kept: every replay of the captured graph records them again).
void prof_flush(ft_moe *h) {
  if (h->prof_class.empty()) return;
  cudaEventSynchronize(h->prof_events[2 * h->prof_class.size() - 1]);
  std::vector<int32_t> rec;
  if (h->prof_rec) {
    rec.resize(2 * std::min(h->prof_class.size(), h->prof_rec_cap));
    if (cudaMemcpy(rec.data(), h->prof_rec, rec.size() * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
      rec.clear();
  }
  for (size_t i = 0; i < h->prof_class.size(); ++i) {
    float ms = 0.f;
    int cls = h->prof_class[i];
    int64_t items = 0;
    if (cls == FT_PROF_EXPERTS_HIT && 2 * i + 1 < rec.size()) {
      if (rec[2 * i] > 0) cls = FT_PROF_EXPERTS_MISS;
      items = rec[2 * i + 1];
    }
    if (cudaEventElapsedTime(&ms, h->prof_events[2 * i], h->prof_events[2 * i + 1]) == cudaSuccess) {
      h->prof_ms[cls] += ms;
      h->prof_n[cls] += 1;
      h->prof_items[cls] += items;
    }
  }
  cudaGetLastError();
  if (!h->prof_keep) h->prof_class.clear();
}

// Brackets one kernel launch with timing events while profiling is on.
struct ProfScope {
  ft_moe *h;
  cudaStream_t s;
  int idx = -1;
  ProfScope(ft_moe *h_, int cls, cudaStream_t s_) : h(h_), s(s_) {
    if (!h->prof_on) return;
    if (2 * (h->prof_class.size() + 1) > h->prof_events.size()) {
      if (h->prof_keep) return;  // graph mode: the pool was sized when profiling was enabled
      if (h->prof_events.size() < 16384) {
        for (int i = 0; i < 512; ++i) {
          cudaEvent_t e;
          if (cudaEventCreate(&e) != cudaSuccess) break;
          h->prof_events.push_back(e);
        }
      }
      if (2 * (h->prof_class.size() + 1) > h->prof_events.size()) prof_flush(h);
    }
    idx = (int)h->prof_class.size();
    h->prof_class.push_back(cls);
    record(h->prof_events[2 * idx]);
  }
  ~ProfScope() {
    if (idx < 0) return;
    record(h->prof_events[2 * idx + 1]);
    // the decode expert kernel's call: its fill and item counts, read back at the flush
    if (h->prof_class[idx] == FT_PROF_EXPERTS_HIT && h->prof_rec && (size_t)idx < h->prof_rec_cap)
      cudaMemcpyAsync(h->prof_rec + 2 * idx, &h->ctr->n_fill, 2 * sizeof(int32_t),
                      cudaMemcpyDeviceToDevice, s);
  }
  // In graph mode the records are captured as external event nodes, which keep timing.
  void record(cudaEvent_t e) {
    if (h->prof_keep)
      cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
    else
      cudaEventRecord(e, s);
  }
};

void free_all(ft_moe *h) {
  for (void *p : h->allocs) cudaFree(p);
  h->allocs.clear();
  if (h->slots) cudaFree(h->slots);
  if (h->owner) cudaFree(h->owner);
  if (h->stamps) cudaFree(h->stamps);
  if (h->fp4_scratch) cudaFree(h->fp4_scratch);
  for (int i = 0; i < 2; ++i) {
    if (h->dbuf[i]) cudaFree(h->dbuf[i]);
    if (h->chain[i]) cudaFree(h->chain[i]);
  }
  if (h->xstage) cudaFree(h->xstage);
  if (h->ostage) cudaFree(h->ostage);
  for (auto *v : {&h->ev_cs, &h->ev_ce, &h->ev_ks, &h->ev_ke})
    for (cudaEvent_t e : *v) cudaEventDestroy(e);
  if (h->copy_stream) cudaStreamDestroy(h->copy_stream);
  if (h->pool_registered) cudaHostUnregister(const_cast<uint16_t *>(h->pool_host));
  for (cudaEvent_t e : h->prof_events) cudaEventDestroy(e);
  if (h->prof_rec) cudaFree(h->prof_rec);
}

bool capturing(cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &st) != cudaSuccess) {
    cudaGetLastError();
    return true;  // querying failed: treat as unsafe
  }
  return st != cudaStreamCaptureStatusNone;
}

ControlArgs control_args(ft_moe *h, int layer, int T, bool decode, const uint16_t *buffer) {
  ControlArgs a{};
  a.idx = h->idx;
  a.w = h->w;
  a.tie = h->tie;
  a.T = T;
  a.k = h->k;
  a.E = h->E;
  a.P = T * h->k;
  a.layer = layer;
  a.L = h->L;
  a.counts = h->counts;
  a.offsets = h->offsets;
  a.perm = h->perm;
  a.inv = h->inv;
  a.tok = h->tok;
  a.wq = h->wq;
  a.work = h->work;
  a.slot_table = decode ? h->slot_table : nullptr;
  a.cache = h->cache;
  a.fills = h->fills;
  a.freq = h->freq;
  a.sync = decode ? h->sync : nullptr;
  a.n_sync = decode ? kSyncInts(h->d) : 0;
  a.buffer = buffer;
  a.shared = h->n_shared ? h->shared + (size_t)layer * h->entry_elems : nullptr;
  a.entry_elems = h->entry_elems;
  a.ctr = h->ctr;
  a.d = h->d;
  return a;
}

// Publish the current slot storage to the device-side descriptor the kernels read.
int upload_cache_desc(ft_moe *h) {
  CacheDesc d{h->slots, h->owner, h->stamps, h->n_slots, 0};
  cudaError_t e = cudaMemcpy(h->cache, &d, sizeof(d), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return fail(FT_ERR_CUDA, "cache descriptor: %s", cudaGetErrorString(e));
  return FT_OK;
}

// Tensor maps for the tcgen05 GEMMs over `buffer` (n_entries complete entries).
int build_maps(ft_moe *h, TcMaps *m, const uint16_t *buffer, int n_entries) {
  const uint64_t R = (uint64_t)h->max_tokens * h->k + h->max_tokens;
  const uint64_t d = h->d, f = h->d_ff;
  const uint16_t *sh = h->shared ? h->shared : buffer;
  const uint64_t nsh = h->shared ? (uint64_t)h->L : (uint64_t)n_entries;
  bool ok = make_tmap(&m->a_x, h->xp, d, R, 128) && make_tmap(&m->a_h, h->hbuf, f, R, 128) &&
            make_tmap(&m->b_gu, buffer, d, (uint64_t)n_entries * 3 * f, 128) &&
            make_tmap(&m->bs_gu, sh, d, nsh * 3 * f, 128) &&
            make_tmap(&m->b_dn128, buffer, f, (uint64_t)n_entries * 3 * d, 128) &&
            make_tmap(&m->bs_dn128, sh, f, nsh * 3 * d, 128);
  if (ok && d % 256 == 0)
    ok = make_tmap(&m->b_dn256, buffer, f, (uint64_t)n_entries * 3 * d, 256) &&
         make_tmap(&m->bs_dn256, sh, f, nsh * 3 * d, 256);
  if (!ok) return fail(FT_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  return FT_OK;
}

// bf16 scratch for the MXFP4 entries of one grouped-GEMM call (E entries) and its maps.
int ensure_fp4_scratch(ft_moe *h) {
  if (h->fp4_scratch) return FT_OK;
  const size_t bytes = (size_t)h->E * 6 * h->d * h->d_ff;
  cudaError_t e = cudaMalloc(&h->fp4_scratch, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    h->fp4_scratch = nullptr;
    return fail(FT_ERR_OOM, "MXFP4 expansion scratch (%zu bytes): %s", bytes, cudaGetErrorString(e));
  }
  return build_maps(h, &h->maps_fp4, h->fp4_scratch, h->E);
}

// Router, top-k, permutation and control for one layer.
void route_layer(ft_moe *h, int layer, const uint16_t *x, int T, bool decode,
                 const uint16_t *buffer, cudaStream_t s) {
  if (decode && T <= kGemvMaxTokens) {
    // router, top-k, grouping and the LRU update in one launch
    ControlArgs a = control_args(h, layer, T, decode, buffer);
    ProfScope p(h, FT_PROF_ROUTER, s);
    launch_route_decode(x, h->wr + (size_t)layer * h->E * h->d,
                        h->has_bias[layer] ? h->bias + (size_t)layer * h->E : nullptr, h->logits,
                        a, s);
    return;
  }
  {
    ProfScope p(h, FT_PROF_ROUTER, s);
    launch_router(x, h->wr + (size_t)layer * h->E * h->d,
                  h->has_bias[layer] ? h->bias + (size_t)layer * h->E : nullptr, h->logits, T,
                  h->E, h->d, s);
  }
  {
    ProfScope p(h, FT_PROF_TOPK, s);
    launch_topk(h->logits, h->idx, h->w, h->tie, T, h->E, h->k, s);
  }
  ControlArgs a = control_args(h, layer, T, decode, buffer);
  ProfScope p(h, FT_PROF_CONTROL, s);
  if (a.P > kPermSingleMax) {
    launch_perm_multi(a, h->chunk, s);
    launch_control(a, true, s);
  } else {
    launch_control(a, false, s);
  }
}

// Expert FFN + combine for one layer after routing; `maps` view the weights' buffer.
// Decode calls (T <= kGemvMaxTokens) run the fills and the whole expert path in one launch;
// larger calls fill first (decode forward) and then run the grouped GEMMs, as does every
// prefill layer (whose cast also writes the residual stream's next input).
int experts_layer(ft_moe *h, const uint16_t *x, int T, uint16_t *out, const TcMaps &maps,
                  int layer, bool decode, cudaStream_t s, uint16_t *next = nullptr) {
  const int P = T * h->k;
  if (decode && T <= kGemvMaxTokens) {
    DecodeArgs a{};
    a.work = h->work;
    a.ctr = h->ctr;
    a.fills = h->fills;
    a.pool = reinterpret_cast<const uint4 *>(h->pool_dev);
    a.cache = h->cache;
    a.x = x;
    a.tok = h->tok;
    a.w = h->w;
    a.inv = h->inv;
    a.h = h->hbuf;
    a.y = h->ybuf;
    a.out = out;
    a.sync = h->sync;
    a.T = T;
    a.k = h->k;
    a.d = h->d;
    a.d_ff = h->d_ff;
    a.E = h->E;
    a.shared = h->n_shared;
    a.entry_bytes = h->entry_bytes;
    ProfScope p(h, FT_PROF_EXPERTS_HIT, s);
    return launch_decode_experts(a, h->fp4, s);
  }
  if (decode) {
    ProfScope p(h, FT_PROF_FILL, s);
    launch_fill(h->pool_dev, h->cache, h->fills, h->ctr, h->entry_bytes, h->E,
                std::min(h->E, P), s);
  }
  const int rows = P + (h->n_shared ? T : 0);
  {
    ProfScope p(h, FT_PROF_OTHER, s);
    launch_gather_rows(x, h->tok, h->xp, rows, h->d, h->ctr, s);
    cudaMemsetAsync(h->acc, 0, (size_t)T * h->d * sizeof(float), s);
  }
  if (h->fp4) {
    ProfScope p(h, FT_PROF_OTHER, s);
    launch_dequant_work(h->work, h->ctr, h->fp4_scratch, h->d, h->d_ff, std::min(h->E, P), s);
  }
  {
    ProfScope p(h, FT_PROF_GATEUP, s);  // gate/up and down GEMMs on the tensor cores
    launch_tc_ffn(h->fp4 ? h->maps_fp4 : maps, h->work, h->ctr, h->tile_prefix, h->hbuf, h->tok,
                  h->wq, h->acc, h->d, h->d_ff, layer, h->fp4, s);
  }
  ProfScope p(h, FT_PROF_OTHER, s);
  launch_cast_out(h->acc, out, (size_t)T * h->d, x, next, h->ctr, s);
  return FT_OK;
}

int check_handle(ft_moe *h) {
  if (!h) return fail(FT_ERR_INVALID, "null handle");
  return FT_OK;
}

}  // namespace

extern "C" {

const char *ft_last_error(void) { return g_err.c_str(); }

int ft_moe_create(int L, int E, int k, int d, int d_ff, int n_slots, const ft_moe_opts *opts,
                  ft_moe **out) {
  if (!out) return fail(FT_ERR_INVALID, "out is NULL");
  *out = nullptr;
  if (L < 1 || E < 1 || E > kMaxE || k < 1 || k > E || k > kMaxK)
    return fail(FT_ERR_INVALID, "need L >= 1, 1 <= k <= E <= %d, k <= %d (got L=%d E=%d k=%d)",
                kMaxE, kMaxK, L, E, k);
  if (d < 128 || d % 128 || d > 4096 || d_ff < 128 || d_ff % 128 || d_ff > 8192)
    return fail(FT_ERR_INVALID,
                "need d in [128, 4096] and d_ff in [128, 8192], multiples of 128 (got %d, %d)", d,
                d_ff);
  if (n_slots < 1) return fail(FT_ERR_INVALID, "n_slots must be >= 1 (got %d)", n_slots);
  ft_moe_opts o{0, 1, 4096, 0, 0, 0, FT_WEIGHTS_BF16};
  if (opts) o = *opts;
  if (o.max_tokens < 1 || o.max_tokens > (1 << 20))
    return fail(FT_ERR_INVALID, "max_tokens out of range (%d)", o.max_tokens);
  if (o.n_shared != 0 && o.n_shared != 1) return fail(FT_ERR_INVALID, "n_shared must be 0 or 1");
  if (o.weight_format != FT_WEIGHTS_BF16 && o.weight_format != FT_WEIGHTS_MXFP4)
    return fail(FT_ERR_INVALID, "unknown weight_format %d", o.weight_format);
  if (o.weight_format == FT_WEIGHTS_MXFP4 && o.n_shared)
    return fail(FT_ERR_INVALID, "MXFP4 entries: n_shared must be 0");

  ft_moe *h = new ft_moe();
  h->L = L;
  h->E = E;
  h->k = k;
  h->d = d;
  h->d_ff = d_ff;
  h->n_slots = n_slots;
  h->max_tokens = o.max_tokens;
  h->n_shared = o.n_shared;
  h->prewarm = o.prewarm;
  h->debug = o.debug_checks;
  h->prefill_topup = o.prefill_topup != 0;
  h->admission = o.admission != 0;
  h->n_stage = h->admission ? E : 0;
  h->fp4 = o.weight_format == FT_WEIGHTS_MXFP4;
  // entry_elems counts 16-bit units (pointer arithmetic on uint16_t), whatever the format
  h->entry_bytes = h->fp4 ? (size_t)3 * d * d_ff * 17 / 32 : (size_t)3 * d * d_ff * 2;
  h->entry_elems = h->entry_bytes / 2;
  h->has_bias.assign(L, 0);
  cudaGetDevice(&h->device);

  const size_t T = (size_t)o.max_tokens, P = T * k, R = P + T;
  int rc = FT_OK;
  auto A = [&](int r) {
    if (rc == FT_OK) rc = r;
  };
  A(alloc_n(h, &h->wr, (size_t)L * E * d));
  A(alloc_n(h, &h->bias, (size_t)L * E));
  if (o.n_shared) A(alloc_n(h, &h->shared, (size_t)L * h->entry_elems));
  A(alloc_n(h, &h->slot_table, (size_t)L * E));
  A(alloc_n(h, &h->ctr, 1));
  A(alloc_n(h, &h->cache, 1));
  A(alloc_n(h, &h->logits, T * E));
  A(alloc_n(h, &h->idx, P));
  A(alloc_n(h, &h->w, P));
  A(alloc_n(h, &h->tie, T));
  A(alloc_n(h, &h->counts, (size_t)E));
  A(alloc_n(h, &h->offsets, (size_t)E + 1));
  A(alloc_n(h, &h->perm, P));
  A(alloc_n(h, &h->inv, P));
  A(alloc_n(h, &h->tok, R));
  A(alloc_n(h, &h->wq, R));
  A(alloc_n(h, &h->work, (size_t)E + 1));
  A(alloc_n(h, &h->fills, (size_t)E * 3));
  A(alloc_n(h, &h->hbuf, R * d_ff));
  A(alloc_n(h, &h->xp, R * d));
  A(alloc_n(h, &h->acc, T * d));
  A(alloc_n(h, &h->ybuf, (size_t)(kGemvMaxTokens * k + kGemvMaxTokens) * d));
  A(alloc_n(h, &h->sync, (size_t)kSyncInts(d)));
  A(alloc_n(h, &h->chunk, perm_multi_scratch_ints((int)P, E)));
  A(alloc_n(h, &h->tile_prefix, (size_t)kMaxE + 3));
  if (h->admission) A(alloc_n(h, &h->freq, (size_t)L * E));
  if (rc == FT_OK) {
    cudaError_t e = cudaMalloc(&h->slots, (size_t)(n_slots + h->n_stage) * h->entry_bytes);
    if (e == cudaSuccess) e = cudaMalloc(&h->owner, (size_t)n_slots * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMalloc(&h->stamps, (size_t)n_slots * sizeof(unsigned long long));
    if (e != cudaSuccess) {
      cudaGetLastError();
      rc = fail(FT_ERR_OOM, "slot storage (%d x %zu bytes): %s", n_slots, h->entry_bytes,
                cudaGetErrorString(e));
    }
  }
  if (rc == FT_OK) {
    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess) e = cudaMemset(h->bias, 0, (size_t)L * E * sizeof(float));
    if (e == cudaSuccess) e = cudaMemset(h->slot_table, 0xFF, (size_t)L * E * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMemset(h->owner, 0xFF, (size_t)n_slots * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMemset(h->stamps, 0, (size_t)n_slots * sizeof(unsigned long long));
    if (e == cudaSuccess) e = cudaMemset(h->ctr, 0, sizeof(DevCounters));
    if (e == cudaSuccess) e = cudaMemset(h->sync, 0, (size_t)kSyncInts(d) * sizeof(int32_t));
    if (e == cudaSuccess) {
      const unsigned long long limit = kDefaultWaitNs;
      e = cudaMemcpy(&h->ctr->wait_ns, &limit, sizeof(limit), cudaMemcpyHostToDevice);
    }
    if (e == cudaSuccess && h->freq) e = cudaMemset(h->freq, 0, (size_t)L * E * sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemset(h->wr, 0, (size_t)L * E * d * 2);
    if (e == cudaSuccess && h->shared) e = cudaMemset(h->shared, 0, (size_t)L * h->entry_bytes);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->copy_stream, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) rc = fail(FT_ERR_CUDA, "initialisation: %s", cudaGetErrorString(e));
  }
  if (rc == FT_OK && !h->fp4) rc = build_maps(h, &h->maps_slots, h->slots, n_slots + h->n_stage);
  // MXFP4 calls with more tokens than the decode path takes expand their entries to bf16
  // first; the scratch exists from creation so that such calls can be captured
  if (rc == FT_OK && h->fp4 && h->max_tokens > kGemvMaxTokens) rc = ensure_fp4_scratch(h);
  if (rc == FT_OK) rc = upload_cache_desc(h);
  if (rc != FT_OK) {
    free_all(h);
    delete h;
    return rc;
  }
  *out = h;
  return FT_OK;
}

void ft_moe_destroy(ft_moe *h) {
  if (!h) return;
  cudaDeviceSynchronize();
  free_all(h);
  delete h;
}

int ft_moe_get_dims(ft_moe *h, int32_t dims[8]) {
  if (int r = check_handle(h)) return r;
  if (!dims) return fail(FT_ERR_INVALID, "dims is NULL");
  const int32_t v[8] = {h->L, h->E, h->k, h->d, h->d_ff, h->n_slots, h->max_tokens, h->n_shared};
  memcpy(dims, v, sizeof(v));
  return FT_OK;
}

int ft_moe_load_router(ft_moe *h, int layer, const void *Wr_bf16, const float *bias) {
  if (int r = check_handle(h)) return r;
  if (layer < 0 || layer >= h->L) return fail(FT_ERR_INVALID, "layer %d out of range", layer);
  if (!Wr_bf16) return fail(FT_ERR_INVALID, "Wr is NULL");
  FT_CUDA(cudaMemcpy(h->wr + (size_t)layer * h->E * h->d, Wr_bf16, (size_t)h->E * h->d * 2,
                     cudaMemcpyDefault));
  if (bias) {
    FT_CUDA(cudaMemcpy(h->bias + (size_t)layer * h->E, bias, (size_t)h->E * sizeof(float),
                       cudaMemcpyDefault));
    h->has_bias[layer] = 1;
  } else {
    FT_CUDA(cudaMemset(h->bias + (size_t)layer * h->E, 0, (size_t)h->E * sizeof(float)));
    h->has_bias[layer] = 0;
  }
  return FT_OK;
}

int ft_moe_set_router_bias(ft_moe *h, int layer, const float *bias, ft_stream_t stream) {
  if (int r = check_handle(h)) return r;
  if (!bias) return fail(FT_ERR_INVALID, "bias is NULL");
  cudaStream_t s = (cudaStream_t)stream;
  if (layer == -1) {
    FT_CUDA(cudaMemcpyAsync(h->bias, bias, (size_t)h->L * h->E * sizeof(float),
                            cudaMemcpyDefault, s));
    std::fill(h->has_bias.begin(), h->has_bias.end(), 1);
  } else {
    if (layer < 0 || layer >= h->L) return fail(FT_ERR_INVALID, "layer %d out of range", layer);
    FT_CUDA(cudaMemcpyAsync(h->bias + (size_t)layer * h->E, bias, (size_t)h->E * sizeof(float),
                            cudaMemcpyDefault, s));
    h->has_bias[layer] = 1;
  }
  return FT_OK;
}

int ft_moe_load_pool(ft_moe *h, void *host_pool, size_t bytes) {
  if (int r = check_handle(h)) return r;
  if (h->pool_host) return fail(FT_ERR_STATE, "pool already loaded");
  if (!host_pool) return fail(FT_ERR_INVALID, "pool is NULL");
  const size_t want = (size_t)h->L * h->E * h->entry_bytes;
  if (bytes != want) return fail(FT_ERR_INVALID, "pool bytes %zu != L*E*entry = %zu", bytes, want);
  if (((uintptr_t)host_pool) & 15) return fail(FT_ERR_INVALID, "pool must be 16-byte aligned");
  cudaPointerAttributes at{};
  cudaError_t e = cudaPointerGetAttributes(&at, host_pool);
  if (e != cudaSuccess) cudaGetLastError();
  bool registered = false;
  if (e != cudaSuccess || at.type == cudaMemoryTypeUnregistered) {
    FT_CUDA(cudaHostRegister(host_pool, bytes, cudaHostRegisterMapped | cudaHostRegisterPortable));
    registered = true;
  } else if (at.type != cudaMemoryTypeHost) {
    return fail(FT_ERR_INVALID, "pool must be host memory (got memory type %d)", (int)at.type);
  }
  void *dptr = nullptr;
  e = cudaHostGetDevicePointer(&dptr, host_pool, 0);
  if (e != cudaSuccess) {
    cudaGetLastError();
    if (registered) cudaHostUnregister(host_pool);
    return fail(FT_ERR_CUDA, "pool is not mapped into the device: %s", cudaGetErrorString(e));
  }
  h->pool_host = static_cast<const uint16_t *>(host_pool);
  h->pool_dev = static_cast<const uint16_t *>(dptr);
  h->pool_bytes = bytes;
  h->pool_registered = registered;
  if (h->prewarm) {
    const int n = std::min(h->n_slots, h->L * h->E);
    FT_CUDA(cudaMemcpy(h->slots, host_pool, (size_t)n * h->entry_bytes, cudaMemcpyHostToDevice));
    std::vector<int32_t> table((size_t)h->L * h->E, -1), owner(h->n_slots, -1);
    std::vector<unsigned long long> stamps(h->n_slots, 0);
    for (int key = 0; key < n; ++key) {
      table[key] = key;
      owner[key] = key;
      stamps[key] = (unsigned long long)key + 1;
    }
    FT_CUDA(cudaMemcpy(h->slot_table, table.data(), table.size() * 4, cudaMemcpyHostToDevice));
    FT_CUDA(cudaMemcpy(h->owner, owner.data(), owner.size() * 4, cudaMemcpyHostToDevice));
    FT_CUDA(cudaMemcpy(h->stamps, stamps.data(), stamps.size() * 8, cudaMemcpyHostToDevice));
    DevCounters c{};
    FT_CUDA(cudaMemcpy(&c, h->ctr, sizeof(c), cudaMemcpyDeviceToHost));
    c.tick = (unsigned long long)n;
    c.occupied = n;
    FT_CUDA(cudaMemcpy(h->ctr, &c, sizeof(c), cudaMemcpyHostToDevice));
  }
  return FT_OK;
}

int ft_moe_load_shared(ft_moe *h, int layer, const void *entry_bf16) {
  if (int r = check_handle(h)) return r;
  if (!h->n_shared) return fail(FT_ERR_STATE, "handle was created without a shared expert");
  if (layer < 0 || layer >= h->L) return fail(FT_ERR_INVALID, "layer %d out of range", layer);
  if (!entry_bf16) return fail(FT_ERR_INVALID, "entry is NULL");
  FT_CUDA(cudaMemcpy(h->shared + (size_t)layer * h->entry_elems, entry_bf16, h->entry_bytes,
                     cudaMemcpyDefault));
  return FT_OK;
}

int ft_moe_forward(ft_moe *h, int layer, const void *x, int T, void *out, ft_stream_t stream) {
  if (int r = check_handle(h)) return r;
  if (!h->pool_host) return fail(FT_ERR_STATE, "forward before ft_moe_load_pool");
  if (layer < 0 || layer >= h->L) return fail(FT_ERR_INVALID, "layer %d out of range", layer);
  if (T < 1 || T > h->max_tokens)
    return fail(FT_ERR_INVALID, "T=%d outside [1, max_tokens=%d]", T, h->max_tokens);
  if (!x || !out) return fail(FT_ERR_INVALID, "x or out is NULL");
  if ((((uintptr_t)x) | ((uintptr_t)out)) & 15)
    return fail(FT_ERR_INVALID, "x and out must be 16-byte aligned");
  cudaStream_t s = (cudaStream_t)stream;
  const uint16_t *xb = static_cast<const uint16_t *>(x);
  route_layer(h, layer, xb, T, true, nullptr, s);
  if (int r = experts_layer(h, xb, T, static_cast<uint16_t *>(out), h->maps_slots, layer, true, s))
    return r;
  h->last_T = T;
  h->last_stream = s;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(FT_ERR_CUDA, "forward launch: %s", cudaGetErrorString(e));
  return FT_OK;
}

int ft_moe_decode_host(ft_moe *h, int layer0, int n_layers, const void *x_host, int T,
                       void *out_host, ft_stream_t stream) {
  if (int r = check_handle(h)) return r;
  if (n_layers < 1 || layer0 < 0 || layer0 + n_layers > h->L)
    return fail(FT_ERR_INVALID, "layers [%d, %d) out of range", layer0, layer0 + n_layers);
  if (T < 1 || T > h->max_tokens) return fail(FT_ERR_INVALID, "T=%d out of range", T);
  if (!x_host || !out_host) return fail(FT_ERR_INVALID, "x or out is NULL");
  cudaStream_t s = (cudaStream_t)stream;
  const size_t xb = (size_t)T * h->d * 2, ob = xb * n_layers;
  if (xb > h->xstage_bytes || ob > h->ostage_bytes) {
    if (capturing(s)) return fail(FT_ERR_STATE, "staging must grow outside stream capture");
    FT_CUDA(cudaStreamSynchronize(s));
    if (xb > h->xstage_bytes) {
      if (h->xstage) cudaFree(h->xstage);
      h->xstage = nullptr;
      h->xstage_bytes = 0;
      FT_CUDA(cudaMalloc(&h->xstage, xb));
      h->xstage_bytes = xb;
    }
    if (ob > h->ostage_bytes) {
      if (h->ostage) cudaFree(h->ostage);
      h->ostage = nullptr;
      h->ostage_bytes = 0;
      FT_CUDA(cudaMalloc(&h->ostage, ob));
      h->ostage_bytes = ob;
    }
  }
  FT_CUDA(cudaMemcpyAsync(h->xstage, x_host, xb, cudaMemcpyHostToDevice, s));
  for (int i = 0; i < n_layers; ++i) {
    int r = ft_moe_forward(h, layer0 + i, h->xstage, T, h->ostage + (size_t)i * T * h->d, stream);
    if (r != FT_OK) return r;
  }
  FT_CUDA(cudaMemcpyAsync(out_host, h->ostage, ob, cudaMemcpyDeviceToHost, s));
  return FT_OK;
}

int ft_moe_prefill_stream(ft_moe *h, int layer0, int n_layers, const void *x, int T, void *out,
                          ft_stream_t stream) {
  if (int r = check_handle(h)) return r;
  if (!h->pool_host) return fail(FT_ERR_STATE, "prefill before ft_moe_load_pool");
  if (n_layers < 1 || layer0 < 0 || layer0 + n_layers > h->L)
    return fail(FT_ERR_INVALID, "layers [%d, %d) out of range", layer0, layer0 + n_layers);
  if (T < 1 || T > h->max_tokens)
    return fail(FT_ERR_INVALID, "T=%d outside [1, max_tokens=%d]", T, h->max_tokens);
  if (!x || !out) return fail(FT_ERR_INVALID, "x or out is NULL");
  if ((((uintptr_t)x) | ((uintptr_t)out)) & 15)
    return fail(FT_ERR_INVALID, "x and out must be 16-byte aligned");
  cudaStream_t s = (cudaStream_t)stream;
  if (capturing(s)) return fail(FT_ERR_STATE, "prefill cannot be captured");
  const size_t layer_bytes = (size_t)h->E * h->entry_bytes;
  for (int i = 0; i < 2; ++i) {
    if (!h->dbuf[i]) {
      if (inject("prefill_alloc")) return fail(FT_ERR_OOM, "injected allocation failure");
      cudaError_t e = cudaMalloc(&h->dbuf[i], layer_bytes);
      if (e != cudaSuccess) {
        cudaGetLastError();
        h->dbuf[i] = nullptr;
        return fail(FT_ERR_OOM, "double buffer (%zu bytes): %s", layer_bytes,
                    cudaGetErrorString(e));
      }
      if (!h->fp4)
        if (int r = build_maps(h, &h->maps_dbuf[i], h->dbuf[i], h->E)) return r;
    }
    if (!h->chain[i]) {
      cudaError_t e = cudaMalloc(&h->chain[i], (size_t)h->max_tokens * h->d * 2);
      if (e != cudaSuccess) {
        cudaGetLastError();
        h->chain[i] = nullptr;
        return fail(FT_ERR_OOM, "residual stream buffer: %s", cudaGetErrorString(e));
      }
    }
  }
  if (h->fp4)
    if (int r = ensure_fp4_scratch(h)) return r;
  while ((int)h->ev_cs.size() < n_layers) {
    cudaEvent_t a, b, c, d;
    FT_CUDA(cudaEventCreate(&a));
    FT_CUDA(cudaEventCreate(&b));
    FT_CUDA(cudaEventCreate(&c));
    FT_CUDA(cudaEventCreate(&d));
    h->ev_cs.push_back(a);
    h->ev_ce.push_back(b);
    h->ev_ks.push_back(c);
    h->ev_ke.push_back(d);
  }
  const uint8_t *pool = reinterpret_cast<const uint8_t *>(h->pool_host);
  const uint16_t *xb = static_cast<const uint16_t *>(x);
  uint16_t *ob = static_cast<uint16_t *>(out);
  // the copy stream starts after everything already queued on `stream` (earlier users of
  // the buffers)
  cudaEvent_t start = h->ev_ks[0];
  FT_CUDA(cudaEventRecord(start, s));
  FT_CUDA(cudaStreamWaitEvent(h->copy_stream, start, 0));
  // top-up: the slot table as of everything already queued on `stream`
  if (h->prefill_topup) {
    FT_CUDA(cudaStreamSynchronize(s));
    h->table_host.resize((size_t)h->L * h->E);
    FT_CUDA(cudaMemcpy(h->table_host.data(), h->slot_table, h->table_host.size() * sizeof(int32_t),
                       cudaMemcpyDeviceToHost));
  }
  h->last_h2d_bytes = h->last_d2d_bytes = 0;
  const size_t eb = h->entry_bytes;
  auto enqueue_copy = [&](int i) -> int {
    const int l = layer0 + i;
    uint8_t *dst = reinterpret_cast<uint8_t *>(h->dbuf[i & 1]);
    const uint8_t *src = pool + (size_t)l * layer_bytes;
    if (i >= 2) FT_CUDA(cudaStreamWaitEvent(h->copy_stream, h->ev_ke[i - 2], 0));
    FT_CUDA(cudaEventRecord(h->ev_cs[i], h->copy_stream));
    if (!h->prefill_topup) {
      FT_CUDA(cudaMemcpyAsync(dst, src, layer_bytes, cudaMemcpyHostToDevice, h->copy_stream));
      h->last_h2d_bytes += layer_bytes;
    } else {
      const int32_t *row = h->table_host.data() + (size_t)l * h->E;
      const uint8_t *slots = reinterpret_cast<const uint8_t *>(h->slots);
      for (int e = 0; e < h->E;) {
        const int sl = row[e];
        if (sl >= 0) {  // resident: slot -> buffer
          FT_CUDA(cudaMemcpyAsync(dst + (size_t)e * eb, slots + (size_t)sl * eb, eb,
                                  cudaMemcpyDeviceToDevice, h->copy_stream));
          h->last_d2d_bytes += eb;
          ++e;
        } else {        // a maximal run of absent experts: one host -> device copy
          int e1 = e + 1;
          while (e1 < h->E && row[e1] < 0) ++e1;
          const size_t n = (size_t)(e1 - e) * eb;
          FT_CUDA(cudaMemcpyAsync(dst + (size_t)e * eb, src + (size_t)e * eb, n,
                                  cudaMemcpyHostToDevice, h->copy_stream));
          h->last_h2d_bytes += n;
          e = e1;
        }
      }
    }
    FT_CUDA(cudaEventRecord(h->ev_ce[i], h->copy_stream));
    return FT_OK;
  };
  if (int r = enqueue_copy(0)) return r;
  for (int i = 0; i < n_layers; ++i) {
    if (i + 1 < n_layers)
      if (int r = enqueue_copy(i + 1)) return r;
    FT_CUDA(cudaStreamWaitEvent(s, h->ev_ce[i], 0));
    FT_CUDA(cudaEventRecord(h->ev_ks[i], s));
    // residual stream: layer i reads x_i (x_0 = x), and writes out[i] = y_i and
    // x_{i+1} = bf16(x_i + y_i) for the next layer
    const uint16_t *xi = i == 0 ? xb : h->chain[i & 1];
    uint16_t *xnext = i + 1 < n_layers ? h->chain[(i + 1) & 1] : nullptr;
    route_layer(h, layer0 + i, xi, T, false, h->dbuf[i & 1], s);
    if (int r = experts_layer(h, xi, T, ob + (size_t)i * T * h->d, h->maps_dbuf[i & 1], layer0 + i,
                              false, s, xnext))
      return r;
    FT_CUDA(cudaEventRecord(h->ev_ke[i], s));
  }
  h->last_prefill_layers = n_layers;
  h->last_T = T;
  h->last_stream = s;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(FT_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
  return FT_OK;
}

int ft_moe_prefill_bytes(ft_moe *h, uint64_t *h2d_bytes, uint64_t *d2d_bytes) {
  if (int r = check_handle(h)) return r;
  if (h->last_prefill_layers == 0) return fail(FT_ERR_STATE, "no prefill has run");
  if (h2d_bytes) *h2d_bytes = h->last_h2d_bytes;
  if (d2d_bytes) *d2d_bytes = h->last_d2d_bytes;
  return FT_OK;
}

int ft_moe_prefill_timing(ft_moe *h, float *copy_ms, float *compute_ms, float *wall_ms) {
  if (int r = check_handle(h)) return r;
  const int n = h->last_prefill_layers;
  if (n == 0) return fail(FT_ERR_STATE, "no prefill has run");
  FT_CUDA(cudaEventSynchronize(h->ev_ke[n - 1]));
  float c = 0, k = 0, w = 0, t;
  for (int i = 0; i < n; ++i) {
    FT_CUDA(cudaEventElapsedTime(&t, h->ev_cs[i], h->ev_ce[i]));
    c += t;
    FT_CUDA(cudaEventElapsedTime(&t, h->ev_ks[i], h->ev_ke[i]));
    k += t;
  }
  FT_CUDA(cudaEventElapsedTime(&w, h->ev_cs[0], h->ev_ke[n - 1]));
  if (copy_ms) *copy_ms = c;
  if (compute_ms) *compute_ms = k;
  if (wall_ms) *wall_ms = w;
  return FT_OK;
}

int ft_cache_resize(ft_moe *h, int n_new) {
  if (int r = check_handle(h)) return r;
  if (n_new < 1) return fail(FT_ERR_INVALID, "n_slots must be >= 1 (got %d)", n_new);
  if (capturing(h->last_stream) || capturing(cudaStreamLegacy))
    return fail(FT_ERR_STATE, "resize during stream capture");
  FT_CUDA(cudaDeviceSynchronize());  // safe point
  const int n_old = h->n_slots;
  std::vector<int32_t> owner(n_old);
  std::vector<unsigned long long> stamps(n_old);
  FT_CUDA(cudaMemcpy(owner.data(), h->owner, (size_t)n_old * 4, cudaMemcpyDeviceToHost));
  FT_CUDA(cudaMemcpy(stamps.data(), h->stamps, (size_t)n_old * 8, cudaMemcpyDeviceToHost));
  std::vector<int> occ;
  for (int s = 0; s < n_old; ++s)
    if (owner[s] >= 0) occ.push_back(s);
  std::stable_sort(occ.begin(), occ.end(), [&](int a, int b) { return stamps[a] > stamps[b]; });
  const int m = std::min<int>(n_new, (int)occ.size());

  uint16_t *nslots = nullptr;
  int32_t *nowner = nullptr;
  unsigned long long *nstamps = nullptr;
  cudaError_t e = cudaSuccess;
  if (inject("resize_alloc")) e = cudaErrorMemoryAllocation;
  if (e == cudaSuccess) e = cudaMalloc(&nslots, (size_t)(n_new + h->n_stage) * h->entry_bytes);
  if (e == cudaSuccess) e = cudaMalloc(&nowner, (size_t)n_new * 4);
  if (e == cudaSuccess) e = cudaMalloc(&nstamps, (size_t)n_new * 8);
  if (e != cudaSuccess) {
    cudaGetLastError();
    if (nslots) cudaFree(nslots);
    if (nowner) cudaFree(nowner);
    if (nstamps) cudaFree(nstamps);
    return fail(FT_ERR_OOM, "resize to %d slots: %s", n_new, cudaGetErrorString(e));
  }
  std::vector<int32_t> o2(n_new, -1), table((size_t)h->L * h->E, -1);
  std::vector<unsigned long long> s2(n_new, 0);
  for (int r = 0; r < m; ++r) {
    const int old = occ[r];
    o2[r] = owner[old];
    s2[r] = stamps[old];
    table[owner[old]] = r;
    e = cudaMemcpyAsync(nslots + (size_t)r * h->entry_elems, h->slots + (size_t)old * h->entry_elems,
                        h->entry_bytes, cudaMemcpyDeviceToDevice, h->copy_stream);
    if (e != cudaSuccess) break;
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(h->copy_stream);
  if (e == cudaSuccess) e = cudaMemcpy(nowner, o2.data(), (size_t)n_new * 4, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(nstamps, s2.data(), (size_t)n_new * 8, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(nslots);
    cudaFree(nowner);
    cudaFree(nstamps);
    return fail(FT_ERR_CUDA, "resize copy: %s", cudaGetErrorString(e));
  }
  // commit: from here on the new storage is the cache
  FT_CUDA(cudaMemcpy(h->slot_table, table.data(), table.size() * 4, cudaMemcpyHostToDevice));
  cudaFree(h->slots);
  cudaFree(h->owner);
  cudaFree(h->stamps);
  h->slots = nslots;
  h->owner = nowner;
  h->stamps = nstamps;
  h->n_slots = n_new;
  if (int r = upload_cache_desc(h)) return r;
  if (!h->fp4)
    if (int r = build_maps(h, &h->maps_slots, h->slots, n_new + h->n_stage)) return r;
  DevCounters c{};
  FT_CUDA(cudaMemcpy(&c, h->ctr, sizeof(c), cudaMemcpyDeviceToHost));
  c.occupied = m;
  FT_CUDA(cudaMemcpy(h->ctr, &c, sizeof(c), cudaMemcpyHostToDevice));
  h->resizes += 1;
  return FT_OK;
}

int ft_cache_stats(ft_moe *h, ft_cache_stats_t *out) {
  if (int r = check_handle(h)) return r;
  if (!out) return fail(FT_ERR_INVALID, "out is NULL");
  FT_CUDA(cudaDeviceSynchronize());
  DevCounters c{};
  FT_CUDA(cudaMemcpy(&c, h->ctr, sizeof(c), cudaMemcpyDeviceToHost));
  memset(out, 0, sizeof(*out));
  out->calls = c.calls;
  out->hits = c.hits;
  out->misses = c.misses;
  out->fill_bytes = c.fill_bytes;
  out->evictions = c.evictions;
  out->near_ties = c.near_ties;
  out->resizes = h->resizes;
  out->tick = c.tick;
  out->bypasses = c.bypasses;
  out->n_slots = h->n_slots;
  out->occupied = c.occupied;
  out->status = c.status;
  return FT_OK;
}

int ft_cache_stats_reset(ft_moe *h) {
  if (int r = check_handle(h)) return r;
  FT_CUDA(cudaDeviceSynchronize());
  DevCounters c{};
  FT_CUDA(cudaMemcpy(&c, h->ctr, sizeof(c), cudaMemcpyDeviceToHost));
  c.calls = c.hits = c.misses = c.fill_bytes = c.evictions = c.near_ties = c.bypasses = 0;
  c.status = 0;
  FT_CUDA(cudaMemcpy(h->ctr, &c, sizeof(c), cudaMemcpyHostToDevice));
  h->resizes = 0;
  return FT_OK;
}

int ft_moe_status(ft_moe *h, int *status) {
  if (int r = check_handle(h)) return r;
  if (!status) return fail(FT_ERR_INVALID, "status is NULL");
  FT_CUDA(cudaDeviceSynchronize());
  DevCounters c{};
  FT_CUDA(cudaMemcpy(&c, h->ctr, sizeof(c), cudaMemcpyDeviceToHost));
  *status = c.status;
  return FT_OK;
}

int ft_moe_get_routing(ft_moe *h, int32_t *idx, float *w, uint8_t *tie) {
  if (int r = check_handle(h)) return r;
  FT_CUDA(cudaDeviceSynchronize());
  const size_t P = (size_t)h->last_T * h->k;
  if (idx) FT_CUDA(cudaMemcpy(idx, h->idx, P * 4, cudaMemcpyDeviceToHost));
  if (w) FT_CUDA(cudaMemcpy(w, h->w, P * 4, cudaMemcpyDeviceToHost));
  if (tie) FT_CUDA(cudaMemcpy(tie, h->tie, (size_t)h->last_T, cudaMemcpyDeviceToHost));
  return FT_OK;
}

int ft_moe_get_logits(ft_moe *h, float *logits) {
  if (int r = check_handle(h)) return r;
  if (!logits) return fail(FT_ERR_INVALID, "logits is NULL");
  FT_CUDA(cudaDeviceSynchronize());
  FT_CUDA(cudaMemcpy(logits, h->logits, (size_t)h->last_T * h->E * 4, cudaMemcpyDeviceToHost));
  return FT_OK;
}

int ft_moe_get_perm(ft_moe *h, int32_t *counts, int32_t *offsets, int32_t *perm) {
  if (int r = check_handle(h)) return r;
  FT_CUDA(cudaDeviceSynchronize());
  if (counts) FT_CUDA(cudaMemcpy(counts, h->counts, (size_t)h->E * 4, cudaMemcpyDeviceToHost));
  if (offsets)
    FT_CUDA(cudaMemcpy(offsets, h->offsets, (size_t)(h->E + 1) * 4, cudaMemcpyDeviceToHost));
  if (perm)
    FT_CUDA(cudaMemcpy(perm, h->perm, (size_t)h->last_T * h->k * 4, cudaMemcpyDeviceToHost));
  return FT_OK;
}

int ft_moe_get_cache_state(ft_moe *h, int32_t *slot_table, int32_t *owner, uint64_t *stamps,
                           uint64_t *tick) {
  if (int r = check_handle(h)) return r;
  FT_CUDA(cudaDeviceSynchronize());
  if (slot_table)
    FT_CUDA(cudaMemcpy(slot_table, h->slot_table, (size_t)h->L * h->E * 4, cudaMemcpyDeviceToHost));
  if (owner) FT_CUDA(cudaMemcpy(owner, h->owner, (size_t)h->n_slots * 4, cudaMemcpyDeviceToHost));
  if (stamps)
    FT_CUDA(cudaMemcpy(stamps, h->stamps, (size_t)h->n_slots * 8, cudaMemcpyDeviceToHost));
  if (tick) {
    DevCounters c{};
    FT_CUDA(cudaMemcpy(&c, h->ctr, sizeof(c), cudaMemcpyDeviceToHost));
    *tick = c.tick;
  }
  return FT_OK;
}

int ft_moe_get_fills(ft_moe *h, int32_t *n_fill, int32_t *fills, int cap) {
  if (int r = check_handle(h)) return r;
  FT_CUDA(cudaDeviceSynchronize());
  DevCounters c{};
  FT_CUDA(cudaMemcpy(&c, h->ctr, sizeof(c), cudaMemcpyDeviceToHost));
  if (n_fill) *n_fill = c.n_fill;
  if (fills && c.n_fill > 0) {
    const int n = std::min(cap, c.n_fill);
    FT_CUDA(cudaMemcpy(fills, h->fills, (size_t)n * 3 * 4, cudaMemcpyDeviceToHost));
  }
  return FT_OK;
}

int ft_moe_profile(ft_moe *h, int enable) {
  if (int r = check_handle(h)) return r;
  if (enable && (capturing(h->last_stream) || capturing(cudaStreamLegacy)))
    return fail(FT_ERR_STATE, "profiling cannot be enabled during stream capture");
  if (!enable) {
    h->prof_keep = false;
    prof_flush(h);
    h->prof_class.clear();
  } else {
    h->prof_class.clear();
    if (enable == 2) {  // graph mode: events for up to 4096 launches, created now
      while (h->prof_events.size() < 8192) {
        cudaEvent_t e;
        FT_CUDA(cudaEventCreate(&e));
        h->prof_events.push_back(e);
      }
    }
    if (!h->prof_rec) {  // one record per event pair, for every pair the pool can hold
      h->prof_rec_cap = 8192;
      FT_CUDA(cudaMalloc(&h->prof_rec, h->prof_rec_cap * 2 * sizeof(int32_t)));
      FT_CUDA(cudaMemset(h->prof_rec, 0, h->prof_rec_cap * 2 * sizeof(int32_t)));
    }
    h->prof_keep = enable == 2;
  }
  h->prof_on = enable != 0;
  return FT_OK;
}

int ft_moe_profile_read(ft_moe *h, double *ms, int64_t *launches, int64_t *items) {
  if (int r = check_handle(h)) return r;
  prof_flush(h);
  for (int i = 0; i < FT_PROF_N; ++i) {
    if (ms) ms[i] += h->prof_ms[i];
    if (launches) launches[i] += h->prof_n[i];
    if (items) items[i] += h->prof_items[i];
    h->prof_ms[i] = 0;
    h->prof_n[i] = 0;
    h->prof_items[i] = 0;
  }
  return FT_OK;
}

int ft_moe_debug_set(ft_moe *h, int what, int64_t value) {
  if (int r = check_handle(h)) return r;
  FT_CUDA(cudaDeviceSynchronize());
  if (what == FT_DEBUG_HOLD_FILLS) {
    const int v = value != 0;
    FT_CUDA(cudaMemcpy(&h->ctr->hold_fills, &v, sizeof(v), cudaMemcpyHostToDevice));
  } else if (what == FT_DEBUG_WAIT_NS) {
    if (value < 1) return fail(FT_ERR_INVALID, "wait limit must be >= 1 ns");
    const unsigned long long v = (unsigned long long)value;
    FT_CUDA(cudaMemcpy(&h->ctr->wait_ns, &v, sizeof(v), cudaMemcpyHostToDevice));
  } else {
    return fail(FT_ERR_INVALID, "unknown debug setting %d", what);
  }
  return FT_OK;
}

}  // extern "C"
