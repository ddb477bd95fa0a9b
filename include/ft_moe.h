/*
 * ft_moe.h - routed Mixture-of-Experts layer forward with a device-resident LRU
 * expert-slot cache, for one NVIDIA B300 (sm_103a).
 *
 * The system follows the FreeToken pages:
 *   - "FreeToken benchmark", section "how FreeToken serves large MoE models": the full
 *     routed-expert pool lives in host memory as the source of truth; the GPU holds an
 *     elastic expert cache; prefill double-buffers whole layers (layer l+1 is copied while
 *     layer l computes); decode uses a shared LRU expert cache; device-resident control
 *     data keeps routing-dependent decisions compatible with captured CUDA execution
 *     ("graph compatibility" blurb).
 *   - "FreeToken RTX 4090", section "how the MoE memory hierarchy works": a cache entry is
 *     one complete logical (layer, expert) pair, identified by one mapping on CPU and GPU;
 *     the LRU is shared across layers and tokens and follows routing.
 *   - "FreeToken vram": the GPU expert cache can be rebuilt at scheduler safe points
 *     without restarting or reloading the host pool.
 * The pages print no formulas.  The layer computed here (a reading, stated once):
 *   logits l[t,e] = sum_i x[t,i] W_r[e,i] (+ bias[e]) in one fixed fp32 order;
 *   top-k by (logit descending, expert id ascending);
 *   gates = softmax over the k selected logits (= full softmax renormalised over top-k);
 *   y_e(x) = W_down^T (silu(W_gate^T x) * (W_up^T x));
 *   out[t] = sum_j w[t,j] y_{idx[t,j]}(x_t) (+ the shared expert with weight 1).
 *
 * Conventions for every call:
 *   - Returns FT_OK (0) or a negative-free error code below; ft_last_error() gives a
 *     thread-local message for the last failing call of this thread.
 *   - "device" pointers are CUDA device memory of the current device; "host" pointers are
 *     ordinary or pinned host memory as stated.
 *   - bf16 tensors are row-major arrays of uint16 bit patterns.
 *   - A handle is not thread-safe; calls on one handle must not overlap.
 *   - Asynchronous calls (forward, set_router_bias) only enqueue work on the given stream;
 *     device-side failures (capacity exceeded, a bad index caught by a kernel) are recorded
 *     in a device status word read by ft_cache_stats() / ft_moe_status().
 *   - No kernel traps, asserts or spins: kernels that meet an error set the status word and
 *     return.
 */
#ifndef FT_MOE_H
#define FT_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *ft_stream_t; /* a cudaStream_t; NULL = legacy default stream */

enum {
  FT_OK = 0,
  FT_ERR_INVALID = 1,  /* bad argument (shape, pointer, layer index, alignment)         */
  FT_ERR_STATE = 2,    /* call not allowed now (no pool loaded, stream capture active)   */
  FT_ERR_CUDA = 3,     /* a CUDA runtime call failed; message in ft_last_error()         */
  FT_ERR_OOM = 4,      /* device or pinned allocation failed; state unchanged            */
  FT_ERR_CAPACITY = 5, /* a call touched more distinct experts than there are slots      */
  FT_ERR_TIMEOUT = 6   /* reserved for bounded device waits                              */
};

typedef struct ft_moe ft_moe;

/* Options for ft_moe_create; pass NULL for the defaults given in brackets. */
typedef struct {
  int n_shared;     /* [0] 1 = one always-active shared expert per layer, outside the LRU */
  int prewarm;      /* [1] fill the cache at ft_moe_load_pool with entries (l,e) in
                           lexicographic order, slots 0..min(n_slots,L*E)-1, stamps 1..n  */
  int max_tokens;   /* [4096] largest T accepted by forward / prefill (sizes scratch)     */
  int debug_checks; /* [0] kernels re-check slot indices and record violations           */
  int prefill_topup; /* [0] 1 = prefill copies entries already resident in cache slots
                            device -> device and streams only the rest from the host      */
  int admission;     /* [0] 1 = frequency admission: a miss that finds no free slot replaces
                            the next LRU victim only if its access count is at least the
                            victim's, else it is staged for the one call (see below)       */
  int weight_format; /* [FT_WEIGHTS_BF16] expert entry format, see below                  */
} ft_moe_opts;

/*
 * Expert entry formats (ft_moe_opts.weight_format).
 *   FT_WEIGHTS_BF16:  Wg [d_ff][d] | Wu [d_ff][d] | Wd [d][d_ff], bf16, every row one output
 *                     feature contiguous over its inputs; 6*d*d_ff bytes.
 *   FT_WEIGHTS_MXFP4: the same matrices in MXFP4 - the format the pages deploy routed
 *                     experts in (FreeToken benchmark, "benchmark results", model table),
 *                     read as OCP Microscaling MXFP4: E2M1 codes, one E8M0 power-of-two
 *                     scale per 32 inputs of a row.  Codes Wg [d_ff][d/2] | codes Wu
 *                     [d_ff][d/2] | codes Wd [d][d_ff/2] | scales Wg [d_ff][d/32] | scales Wu
 *                     [d_ff][d/32] | scales Wd [d][d_ff/32]; input 2i of a row is the low
 *                     nibble of byte i, 2i+1 the high nibble; 3*d*d_ff*17/32 bytes.  Decode
 *                     calls (T <= 16) read the 4-bit entries directly; forward with T > 16
 *                     and prefill expand each touched entry to bf16 (exact) before the
 *                     tensor-core grouped GEMMs, in a scratch of E bf16 entries allocated at
 *                     create (max_tokens > 16) or at the first prefill.  n_shared must be 0.
 */
enum { FT_WEIGHTS_BF16 = 0, FT_WEIGHTS_MXFP4 = 1 };

/* Cache counters, accumulated on the device since creation or the last reset. */
typedef struct {
  uint64_t calls;      /* forward calls that reached the cache                            */
  uint64_t hits;       /* sum over calls of |touched experts already resident|            */
  uint64_t misses;     /* sum over calls of |touched experts not resident| (= fills)      */
  uint64_t fill_bytes; /* misses * entry bytes copied host -> slot                        */
  uint64_t evictions;  /* resident entries replaced by a miss                             */
  uint64_t near_ties;  /* tokens whose top-k decision had a logit gap <= 1e-6             */
  uint64_t resizes;    /* successful ft_cache_resize calls                                */
  uint64_t tick;       /* global LRU clock (last stamp handed out)                        */
  uint64_t bypasses;   /* misses staged for one call without entering the cache          */
  int32_t n_slots;     /* current capacity in entries                                     */
  int32_t occupied;    /* slots holding an entry                                          */
  int32_t status;      /* first device-side error code since the last reset (0 = none)    */
  int32_t reserved;
} ft_cache_stats_t;

/* Message for the last failing call on this thread ("" if none). */
const char *ft_last_error(void);

/*
 * Create a layer stack: L layers, E routed experts per layer, top-k routing, hidden size d,
 * expert FFN size d_ff, and a cache of n_slots complete (layer, expert) entries.
 * (FreeToken RTX 4090, "how the MoE memory hierarchy works": each token routes to a few of a
 * layer's experts - 6 of 256 in its example - and the GPU holds one cache of complete
 * (layer, expert) entries shared by all layers; FreeToken vram: n_slots is the elastic size
 * of that cache.)
 * Requires 1 <= k <= E <= 1024, k <= 32, 1 <= n_slots, d and d_ff multiples of 128 with
 * d <= 4096 and d_ff <= 8192.  The multiples of 128 come from the tensor-core grouped GEMM:
 * K runs in steps of 64 (d for gate/up, d_ff for down) and N in blocks of 128 W_gate/W_up rows
 * (d_ff) and 128 or 256 W_down rows (d); d <= 4096 lets a W_gate + W_up row pair fit one
 * 16 KB shared-memory stage of the decode kernel.
 * One entry is 3*d*d_ff bf16: W_gate rows [d_ff][d], W_up rows [d_ff][d], W_down rows
 * [d][d_ff] (each row one output feature, contiguous over input features).  The library
 * allocates and owns all device state (router weights, slot storage, tables, scratch).
 * *out receives the handle; on failure *out is NULL and nothing stays allocated.
 */
int ft_moe_create(int L, int E, int k, int d, int d_ff, int n_slots, const ft_moe_opts *opts,
                  ft_moe **out);

/* Free every device allocation; unregister the host pool if this library registered it.
 * Synchronises the library's streams first.  NULL is ignored.  (The state released is what
 * the pages' runtime keeps per model: the GPU expert cache and its mapping - FreeToken
 * benchmark, "how FreeToken serves large MoE models", runtime-layer table.) */
void ft_moe_destroy(ft_moe *h);

/*
 * Router weights of one layer: Wr = device bf16 [E][d] (copied), bias = device fp32 [E] or
 * NULL (bias 0).  Synchronous.  The bias is added to the logits before top-k and before the
 * gate softmax.  (FreeToken RTX 4090, "how the MoE memory hierarchy works": the router picks
 * each token's experts per layer; scores, selection and gates follow the reading at the top
 * of this file.)
 */
int ft_moe_load_router(ft_moe *h, int layer, const void *Wr_bf16, const float *bias);

/*
 * Replace router biases on `stream` (device-to-device, so it may sit inside a captured
 * graph): layer >= 0 sets that layer from device fp32 [E]; layer == -1 sets all layers from
 * device fp32 [L][E].  (Same routing passage as ft_moe_load_router; per-step biases let a
 * captured decode step follow drifting expert popularity - FreeToken benchmark, "graph
 * compatibility": routing-dependent data stays on the device.)
 */
int ft_moe_set_router_bias(ft_moe *h, int layer, const float *bias, ft_stream_t stream);

/*
 * Attach the host expert pool (FreeToken benchmark, "how FreeToken serves large MoE models":
 * the full routed-expert pool lives in host memory as the source of truth, loaded straight
 * into its final layout; FreeToken RTX 4090: one mapping names each (layer, expert) entry
 * wherever it lives): `host_pool` holds L*E entries in [L][E][entry] order,
 * `bytes` == L*E*entry bytes.  The caller owns the pool and keeps it alive and unchanged
 * until ft_moe_destroy.  Pinned memory (cudaHostAlloc / cudaHostRegister) is used as is;
 * pageable memory is registered here (mapped) and unregistered at destroy.  Kernels read
 * missed entries straight from the mapped pool over the host link.  With prewarm, copies
 * the first min(n_slots, L*E) entries into slots 0.. in (layer, expert) order.
 * Synchronous.  Must be called once, before forward / prefill.
 */
int ft_moe_load_pool(ft_moe *h, void *host_pool, size_t bytes);

/* Shared expert of one layer (opts.n_shared = 1): one entry, device or host bf16, copied.
 * It runs for every token with gate weight 1 and lives outside the cache (the always-active
 * expert of the large-expert models the pages serve, FreeToken benchmark, "benchmark
 * results", model table). */
int ft_moe_load_shared(ft_moe *h, int layer, const void *entry_bf16);

/*
 * Decode / general forward of one layer (FreeToken benchmark, "how FreeToken serves large MoE
 * models": decode uses the shared LRU expert cache, missed experts cross the host link into
 * it and every expert executes on the GPU; "graph compatibility": the routing-dependent
 * control stays on the device so the step can be captured): x = device bf16 [T][d],
 * out = device bf16 [T][d], 1 <= T <= max_tokens.  Runs router, top-k, permutation, the LRU update, fills of missed
 * entries from the host pool, the SwiGLU experts through the slot table, and the weighted
 * combine, all on `stream`, with no host synchronisation, so a sequence of calls can be
 * captured into a CUDA graph (for a fixed T).  If the call touches more distinct experts
 * than n_slots, the device status becomes FT_ERR_CAPACITY, the cache is unchanged and
 * out is left unwritten; a call whose logits leave some token without k rankable experts
 * (non-finite activations) is refused the same way with FT_ERR_INVALID.  x and out may not
 * overlap.
 */
int ft_moe_forward(ft_moe *h, int layer, const void *x, int T, void *out, ft_stream_t stream);

/*
 * Decode step over consecutive layers from host buffers (the forward passage above, with the
 * activations crossing the host link as in the pages' end-to-end serving): copies x (host
 * bf16 [T][d],
 * pinned for full speed) to the device, runs ft_moe_forward for layers layer0 ..
 * layer0+n_layers-1 on the same x, and copies the outputs to out (host bf16
 * [n_layers][T][d]).  Enqueued on `stream`; synchronise before reading `out`.
 */
int ft_moe_decode_host(ft_moe *h, int layer0, int n_layers, const void *x_host, int T,
                       void *out_host, ft_stream_t stream);

/*
 * Prefill with full-layer double buffering (FreeToken benchmark, "how FreeToken serves large
 * MoE models", prefill paragraph: whole layers are double-buffered, layer l+1's experts copied
 * while layer l computes).  The layers form a residual stream with attention omitted:
 * x_0 = x (device bf16 [T][d]); for i = 0 .. n_layers-1, out[i] = y_i = MoE layer (layer0+i)
 * applied to x_i, and x_{i+1} = bf16(x_i + y_i) (an fp32 add of the two bf16 values, rounded
 * to nearest even); out is device bf16 [n_layers][T][d].  All E experts of layer l+1 are copied
 * into the back buffer (host -> device, or from cache slots with the top-up option below) on
 * an internal copy stream while layer l computes on `stream`.  Prefill reads the double buffer
 * only: it neither reads nor updates the LRU cache.  Allocates the 2 x E-entry double buffer
 * and two [max_tokens][d] residual-stream buffers on first use.  Returns after enqueueing;
 * `stream` waits for all of it.  Not capturable (FT_ERR_STATE during capture).
 */
int ft_moe_prefill_stream(ft_moe *h, int layer0, int n_layers, const void *x, int T, void *out,
                          ft_stream_t stream);
/*
 * Prefill top-up (opts.prefill_topup = 1), an extension beyond the pages: FreeToken's
 * full-layer streaming ("Prefill double-buffering") copies every expert of a layer over the
 * host link even when the decode cache ("FreeToken pages" LRU) already holds some of them.
 * With the option set, ft_moe_prefill_stream synchronises `stream` once, reads the slot
 * table, and fills each layer's back buffer with a device -> device copy from the slot of
 * every resident (layer, expert) and host -> device copies of the maximal runs of absent
 * experts.  The buffer contents, and so the results, are the same as without the option;
 * the LRU stays untouched (no stamps, no counters).  Forward calls on other streams must
 * not be in flight during the prefill (the handle is single-stream, as everywhere).
 */

/* Bytes the most recent prefill moved into the double buffer: host -> device and
 * slot -> buffer (device -> device).  Either pointer may be NULL.  (The prefill passage
 * above; the bytes are what bounds it on the host link.) */
int ft_moe_prefill_bytes(ft_moe *h, uint64_t *h2d_bytes, uint64_t *d2d_bytes);

/* Timing of the most recent prefill (milliseconds, from CUDA events): per-layer copy and
 * compute spans, summed, and the wall time from first copy to last compute - how well the
 * double buffer hides the copies (prefill passage above). */
int ft_moe_prefill_timing(ft_moe *h, float *copy_ms, float *compute_ms, float *wall_ms);

/*
 * Elastic resize at a safe point (FreeToken vram, elastic-cache paragraph, and FreeToken
 * benchmark, "elastic cache": the GPU expert cache is rebuilt at scheduler safe points without
 * restarting or reloading the host pool): synchronises the library's work, keeps the
 * min(n_slots, occupied) most recently used entries (moved device-to-device into slots 0..
 * in descending stamp order, stamps kept), frees the old slot storage.  Never reads the
 * host pool.  FT_ERR_STATE while a stream capture is active; FT_ERR_OOM leaves the cache
 * exactly as it was.  Graphs of decode calls (T <= 16) captured before a resize stay valid:
 * their kernels find the slot storage through a device-side descriptor that the resize
 * updates.  Graphs of calls with T > 16 hold tensor maps of the old storage and must be
 * captured again.
 */
int ft_cache_resize(ft_moe *h, int n_slots);

/* Synchronise and copy the counters; ft_cache_stats_reset zeroes counters and status.
 * (The hits and misses behind the pages' miss-rate comparison of a global LRU with static
 * placement - FreeToken benchmark, "benchmark results" - and the fill bytes that cross the
 * host link.) */
int ft_cache_stats(ft_moe *h, ft_cache_stats_t *out);
int ft_cache_stats_reset(ft_moe *h);

/* Synchronise and read the device status word (0 = no device-side error); the device-side
 * failures are those listed at the top of this file. */
int ft_moe_status(ft_moe *h, int *status);

/*
 * Debug getters for the most recent forward / prefill layer (synchronise; host outputs), the
 * device-resident control data of the "graph compatibility" blurb (FreeToken benchmark) read
 * back for bit-exact checks:
 *   routing:     idx int32 [T][k], w fp32 [T][k], tie uint8 [T]  (any may be NULL)
 *   logits:      fp32 [T][E]
 *   perm:        counts int32 [E], offsets int32 [E+1], perm int32 [T*k]
 *   cache state: slot_table int32 [L][E] (-1 = absent), owner int32 [n_slots]
 *                (layer*E+expert, -1 = free), stamps uint64 [n_slots], tick
 *   fills:       n_fill, and fills int32 [n_fill][3] = (slot, layer, expert) in order;
 *                `cap` = room in `fills` (entries)
 */
int ft_moe_get_routing(ft_moe *h, int32_t *idx, float *w, uint8_t *tie);
int ft_moe_get_logits(ft_moe *h, float *logits);
int ft_moe_get_perm(ft_moe *h, int32_t *counts, int32_t *offsets, int32_t *perm);
int ft_moe_get_cache_state(ft_moe *h, int32_t *slot_table, int32_t *owner, uint64_t *stamps,
                           uint64_t *tick);
int ft_moe_get_fills(ft_moe *h, int32_t *n_fill, int32_t *fills, int cap);

/* Sizes of a handle: [L, E, k, d, d_ff, n_slots, max_tokens, n_shared]. */
int ft_moe_get_dims(ft_moe *h, int32_t dims[8]);

/*
 * Kernel timing for roofline measurement.  While enabled, forward and prefill bracket every
 * kernel launch with a pair of CUDA events on the launching stream.  enable = 1: eager calls;
 * ft_moe_profile_read synchronises, adds the elapsed time and launch count of each kernel
 * class to ms[] / launches[] (arrays of FT_PROF_N, zeroed by the caller) and clears the
 * record.  enable = 2: graph mode; the events (for up to 4096 launches) are created now, the
 * calls are then captured into a CUDA graph (their event records become graph nodes), and
 * ft_moe_profile_read after each replay adds that replay's times, keeping the record.
 * enable = 0 stops.  Recording adds a little time per launch; time throughput with it off.
 * The decode expert kernel (T <= 16) is one launch per call that runs the call's fills and
 * its whole expert path; its launches are split by whether the call had misses
 * (FT_PROF_EXPERTS_MISS) or not (FT_PROF_EXPERTS_HIT), and items[] (may be NULL) receives the
 * number of expert entries those launches processed (touched experts plus the shared one).
 */
enum {
  FT_PROF_ROUTER = 0,       /* router logits (decode: with top-k and control)   */
  FT_PROF_TOPK = 1,         /* top-k + gates                                     */
  FT_PROF_CONTROL = 2,      /* grouping by expert + LRU update / buffer mapping  */
  FT_PROF_FILL = 3,         /* miss fills over the host link (T > 16)            */
  FT_PROF_GATEUP = 4,       /* grouped GEMMs on the tensor cores (T > 16)        */
  FT_PROF_DOWN = 5,         /* reserved                                          */
  FT_PROF_OTHER = 6,        /* gather, clear, cast                               */
  FT_PROF_EXPERTS_HIT = 7,  /* decode expert kernel, calls without misses        */
  FT_PROF_EXPERTS_MISS = 8, /* decode expert kernel, calls with misses           */
  FT_PROF_N = 9
};
int ft_moe_profile(ft_moe *h, int enable);
int ft_moe_profile_read(ft_moe *h, double *ms, int64_t *launches, int64_t *items);

/*
 * Test hooks (synchronise, then set a device-side value; not for production use):
 *   FT_DEBUG_HOLD_FILLS  value != 0: the decode expert kernel copies its fills but never
 *                        reports them done, so the work that waits for them runs out of time
 *                        and the call records FT_ERR_TIMEOUT (checks that every wait is
 *                        bounded and that the context stays usable); 0 restores.
 *   FT_DEBUG_WAIT_NS     limit in nanoseconds of each cross-CTA wait of the decode expert
 *                        kernel (default 4e9).
 */
enum { FT_DEBUG_HOLD_FILLS = 1, FT_DEBUG_WAIT_NS = 2 };
int ft_moe_debug_set(ft_moe *h, int what, int64_t value);

/*
 * Routing that allocates nothing.  No counterpart in the paper (the FreeToken pages): it is a
 * deployment aid for callers that cannot allocate device memory - code running while a
 * global-mode stream capture is open (cudaMalloc is refused there), serving loops that must
 * not pay for an allocation, and hosts whose framework owns all device memory.
 *
 * Computes, for one layer, what ft_moe_forward computes first: router logits in the same
 * fixed fp32 order, top-k by (logit descending, expert id ascending), gates (softmax over the
 * k selected logits) and near-tie flags.  Inputs: x = device bf16 [T][d], Wr = device bf16
 * [E][d] (both 16-byte aligned), bias = device fp32 [E] or NULL.  Outputs (device, caller
 * owned): idx int32 [T][k], w fp32 [T][k], tie uint8 [T].  Enqueued on `stream`.
 * Limits: 1 <= k <= E <= 1024, k <= 32, d a multiple of 8, and T*E <= 262144; larger sizes
 * return FT_ERR_INVALID.  The logits live in a fixed 1 MiB device array inside this library
 * that every GPU using the library keeps until the process exits.  A call whose stream is not
 * capturing looks up that array's device address on the current device and keeps it; a call
 * on a capturing stream uses the kept address, so make the first call on each device before
 * any stream capture (otherwise FT_ERR_STATE).  All calls share the array: calls that overlap
 * on the GPU race and must be ordered by the caller.
 */
int ft_route_topk_noalloc(const void *x, const void *Wr, const float *bias, int T, int E, int d,
                          int k, int32_t *idx, float *w, uint8_t *tie, ft_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* FT_MOE_H */
