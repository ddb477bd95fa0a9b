#!/usr/bin/env python3
"""MoE-layer throughput on one B300: routed MoE layers with the device LRU expert-slot cache.

Default workload ("decode24"): the decode trace of 24 layers, d=2048, d_ff=768, E=128
routed experts, top-8, a global LRU pool of 768 slots (25% of the 3,072 layer-expert
entries), router logits biased by a per-layer Zipf(1.1) popularity plus a slowly drifting
random walk, misses filled from the pinned host pool.  A step is one decode step: the
batch of b tokens through all 24 layers (router, top-k, grouping, LRU update, miss fills,
SwiGLU experts, combine), captured once as a CUDA graph and replayed.  b = 1 is the headline;
b = 4 and 16 are reported in ``config.per_batch``.  Inputs (activations, per-step biases)
are resident in HBM before the timed region; every step streams >1.8 GB of expert weights,
more than L2 (126 MB), so no flush is needed.

Other workloads: ``--workload large8`` (8 layers, d=4096, d_ff=2048, E=256, top-6 + shared
expert, 640 slots = 30 GiB), ``--workload prefill8`` (prefill streaming, 8 layers, T=4096 and
16384), ``--workload prefill8_topup`` (the same prefill with the full 640-slot decode cache
feeding the double buffer device -> device; only absent experts cross the host link).

``--impl reference`` times the CPU oracle (the slow, plain reference implementation) on the
same workload; each step is one layer call of the b=1 trace.
"""
from __future__ import annotations

import argparse
import json
import os
import signal
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = {
    "decode24": dict(L=24, E=128, k=8, d=2048, d_ff=768, n_slots=768, zipf=1.1, shared=0,
                     batches=(1, 4, 16), headline_b=1),
    "large8": dict(L=8, E=256, k=6, d=4096, d_ff=2048, n_slots=640, zipf=1.0, shared=1,
                   batches=(1, 4, 16), headline_b=1),
    "prefill8": dict(L=8, E=256, k=6, d=4096, d_ff=2048, n_slots=16, shared=0,
                     tokens=(4096, 16384)),
    # prefill top-up: the 640-slot (30 GiB) decode cache, full, feeds the double buffer
    "prefill8_topup": dict(L=8, E=256, k=6, d=4096, d_ff=2048, n_slots=640, shared=0,
                           tokens=(4096, 16384), topup=1),
    "policy": dict(L=24, E=128, k=8, d=2048, d_ff=768, n_slots=768, zipf=1.1, shared=0,
                   batches=(1, 16), steps=2000, refresh=500),
    "elastic": dict(L=24, E=128, k=8, d=2048, d_ff=768, n_slots=768, zipf=1.1, shared=0,
                    steps=10000, phase=1000, resizes=((3500, 307), (6500, 1228))),
}
SEED = 0
# DRAM bytes per launch of the decode expert kernel on an all-hit b=1 call of the 24-layer trace
# (8 entries of 9.44 MB): mean of dram__bytes_read.sum + dram__bytes_write.sum over three
# launches of that shape in one ncu capture of the 4-layer, 512-slot, b = 1 case.  None: the
# kernel has changed since the last capture (76.0 MB per launch), so no figure is claimed.
TRAFFIC_DECODE24_B1 = None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=d["hbm_gbs"], bf16=d["bf16_tflops"],
                    bf16_sustained=d.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm_gbs=6400.0, bf16=1800.0, bf16_sustained=1400.0, source="fallback")


# ----------------------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0):
        self.dev = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.send_signal(signal.SIGTERM)
            self.proc.wait()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) >= 9:
                    rows.append(f)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(rows[0][2]) if rows[0][2].replace(".", "").isdigit() else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------------------
# distributed plumbing (N > 1: independent replicas, no data-path collective)
# ----------------------------------------------------------------------------------------
def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------------------
# workload construction
# ----------------------------------------------------------------------------------------
def entry_bytes(wl):
    """Bytes of one (layer, expert) entry: bf16, or MXFP4 codes + block scales."""
    n = 3 * wl["d"] * wl["d_ff"]
    return n * 17 // 32 if wl.get("fp4") else 2 * n


def build_pool(wl, seed):
    import torch
    import ft_synth.gpu as sg
    sg.build()
    if wl.get("fp4"):
        pool = torch.empty(wl["L"] * wl["E"] * entry_bytes(wl), dtype=torch.uint8,
                           pin_memory=True)
        sg.fill_pool_fp4(pool.data_ptr(), seed, wl["L"], wl["E"], wl["d"], wl["d_ff"])
        return pool
    n = wl["L"] * wl["E"] * 3 * wl["d"] * wl["d_ff"]
    pool = torch.empty(n, dtype=torch.int16, pin_memory=True)
    sg.fill_pool(pool.data_ptr(), seed, wl["L"], wl["E"], wl["d"], wl["d_ff"])
    return pool


def make_stack(wl, pool, seed, max_tokens, n_slots=None):
    import torch
    import ft_synth
    from expert_cached_routed_router_b300 import MoELayerStack
    st = MoELayerStack(wl["L"], wl["E"], wl["k"], wl["d"], wl["d_ff"],
                       n_slots or wl["n_slots"], n_shared=wl["shared"], max_tokens=max_tokens,
                       prefill_topup=wl.get("topup", 0), admission=wl.get("admission", 0),
                       weight_format=1 if wl.get("fp4") else 0)
    for l in range(wl["L"]):
        wr = ft_synth.router_weight(seed, l, wl["E"], wl["d"])
        st.load_router(l, torch.from_numpy(wr.view(np.int16)).cuda())
        if wl["shared"]:
            sh = ft_synth.shared_entry(seed, l, wl["d"], wl["d_ff"])
            st.load_shared(l, torch.from_numpy(sh.view(np.int16)).cuda())
    st.load_pool(pool, pool.numel() * pool.element_size())
    torch.cuda.synchronize()
    return st


def decode_trace(wl, b, n_steps, seed):
    """Device-resident (x [n][b][d] bf16, bias [n][L][E] fp32) for steps 1..n."""
    import torch
    import ft_synth
    import ft_synth.gpu as sg
    gen = ft_synth.DriftingZipfBias(seed, wl["L"], wl["E"], s=wl["zipf"])
    bias = np.empty((n_steps, wl["L"], wl["E"]), np.float32)
    for t in range(n_steps):
        gen.advance()
        for l in range(wl["L"]):
            bias[t, l] = gen.bias(l)
    x = torch.empty((n_steps, b, wl["d"]), dtype=torch.int16, device="cuda")
    sg.activations_device(x.data_ptr(), seed, [1_000_000 * b + t for t in range(n_steps)], b,
                          wl["d"], torch.cuda.current_stream().cuda_stream)
    return x, torch.from_numpy(bias).cuda(), bias


# ----------------------------------------------------------------------------------------
# decode benchmark
# ----------------------------------------------------------------------------------------
def bench_decode_batch(wl, pool, b, W, K, seed, world):
    import torch
    L, d = wl["L"], wl["d"]
    x_all, bias_all, _ = decode_trace(wl, b, W + K, seed)
    st = make_stack(wl, pool, seed, max_tokens=max(16, b))
    xs = torch.empty((b, d), dtype=torch.int16, device="cuda")
    bs = torch.empty((L, wl["E"]), dtype=torch.float32, device="cuda")
    out = torch.empty((L, b, d), dtype=torch.int16, device="cuda")

    def step_body():
        st.set_router_bias(-1, bs)
        for l in range(L):
            st.forward(l, xs, out[l])

    # capture one decode step
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        xs.copy_(x_all[0])
        bs.copy_(bias_all[0])
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    st.stats_reset()
    # capture performs no work; the state only changes on replay
    with torch.cuda.graph(g):
        step_body()
    torch.cuda.synchronize()

    def run(t):
        xs.copy_(x_all[t])
        bs.copy_(bias_all[t])
        g.replay()

    for t in range(W):
        run(t)
    torch.cuda.synchronize()
    st0 = st.stats()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        e0.record()
        for t in range(W, W + K):
            run(t)
        e1.record()
        torch.cuda.synchronize()
    barrier(world)
    ms = e0.elapsed_time(e1)
    st1 = st.stats()
    assert st1["status"] == 0, f"device status {st1['status']}"
    dh = st1["hits"] - st0["hits"]
    dm = st1["misses"] - st0["misses"]
    res = dict(b=b, ms=ms, ms_per_step=ms / K, tok_s=b * K / (ms / 1e3), hits=dh, misses=dm,
               hit_rate=dh / max(1, dh + dm), fill_bytes=st1["fill_bytes"] - st0["fill_bytes"],
               bypasses=st1["bypasses"] - st0["bypasses"], clocks=clk.summary())
    del g
    st.close()
    return res, x_all, bias_all


def profile_decode_batch(wl, pool, b, x_all, bias_all, W, K, seed):
    """Per-kernel device time over the same trace steps: the decode step is captured into a
    CUDA graph with an event-record node before and after every kernel, replayed step by step."""
    import torch
    L, d = wl["L"], wl["d"]
    st = make_stack(wl, pool, seed, max_tokens=max(16, b))
    xs = torch.empty((b, d), dtype=torch.int16, device="cuda")
    bs = torch.empty((L, wl["E"]), dtype=torch.float32, device="cuda")
    out = torch.empty((L, b, d), dtype=torch.int16, device="cuda")
    st.profile(2)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st.set_router_bias(-1, bs)
        for l in range(L):
            st.forward(l, xs, out[l])
    torch.cuda.synchronize()

    def run(t):
        xs.copy_(x_all[t])
        bs.copy_(bias_all[t])
        g.replay()

    for t in range(W):
        run(t)
    torch.cuda.synchronize()
    st.profile_read()
    s0 = st.stats()
    from expert_cached_routed_router_b300 import PROF_CLASSES
    prof = {c: (0.0, 0, 0) for c in PROF_CLASSES}
    for t in range(W, W + K):
        run(t)
        p = st.profile_read()
        prof = {c: tuple(a + b for a, b in zip(prof[c], p[c])) for c in PROF_CLASSES}
    s1 = st.stats()
    st.profile(False)
    touched = (s1["hits"] - s0["hits"]) + (s1["misses"] - s0["misses"])
    fill_bytes = s1["fill_bytes"] - s0["fill_bytes"]
    del g
    st.close()
    return prof, touched, fill_bytes, K * L


def bench_decode_e2e(wl, pool, b, x_all, bias_all, W, K, seed, world):
    """Same trace through ft_moe_decode_host: x from pinned host memory each step, outputs
    read back to pinned host memory each step, copies inside the timed region."""
    import torch
    L, d = wl["L"], wl["d"]
    st = make_stack(wl, pool, seed, max_tokens=max(16, b))
    xh = x_all[:W + K].cpu().pin_memory()
    oh = torch.empty((L, b, d), dtype=torch.int16, pin_memory=True)
    for t in range(W):
        st.set_router_bias(-1, bias_all[t])
        st.decode_host(0, L, xh[t], oh)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for t in range(W, W + K):
        st.set_router_bias(-1, bias_all[t])
        st.decode_host(0, L, xh[t], oh)
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    ms = e0.elapsed_time(e1)
    st.close()
    return dict(ms=ms, tok_s=b * K / (ms / 1e3), h2d=b * d * 2, d2h=L * b * d * 2)


def cpu_oracle_decode(wl, pool, b, bias_np, seed, budget_s=15.0, max_calls=None):
    """The oracle as it stands on layer calls of the trace, in order, until ``budget_s``."""
    import ft_synth
    from oracle import lru as olru
    from oracle import moe as omoe
    from oracle import fp4 as ofp4
    L, E, k, d, d_ff = wl["L"], wl["E"], wl["k"], wl["d"], wl["d_ff"]
    fp4 = bool(wl.get("fp4"))
    ent = entry_bytes(wl) if fp4 else 3 * d * d_ff      # pool elements per entry
    pv = pool.numpy() if fp4 else pool.numpy().view(np.uint16)
    sim = olru.SlotCacheSim(L, E, wl["n_slots"], entry_bytes(wl), prewarm=True,
                            admission=bool(wl.get("admission")))
    routers = {}
    calls = 0
    t0 = time.perf_counter()
    step = 0
    while True:
        x = ft_synth.activations(seed, 1_000_000 * b + step, b, d)
        for l in range(L):
            if l not in routers:
                routers[l] = ft_synth.router_weight(seed, l, E, d)
            r = omoe.moe_layer(x, routers[l], k,
                               lambda e, l=l: pv[(l * E + e) * ent:(l * E + e + 1) * ent],
                               d, d_ff, bias=bias_np[step, l],
                               shared_entry=(ft_synth.shared_entry(seed, l, d, d_ff)
                                             if wl["shared"] else None),
                               ffn=ofp4.expert_ffn_fp4 if fp4 else None)
            sim.access(l, r["idx"].ravel())
            calls += 1
            el = time.perf_counter() - t0
            if (max_calls and calls >= max_calls) or (not max_calls and el >= budget_s):
                return calls, el
        step += 1


def measure_h2d(nbytes=1 << 30, reps=5):
    """Pinned host -> device cudaMemcpyAsync GB/s (best of ``reps``), in this run."""
    import torch
    src = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    best = 0.0
    for _ in range(reps + 1):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        dst.copy_(src, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        best = max(best, nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9)
    del src, dst
    return best


def roofline_decode(wl, prof, pk):
    """HBM rooflines of the decode step from the per-launch record.

    experts_hit: the decode expert kernel on calls without misses, HBM bound: bytes = the
    entries it streams (touched experts + shared) x entry bytes.  experts_miss: the same kernel
    on calls with misses, bound by the host link (its fills) with the hit experts overlapped.
    step_m2: touched bytes (entries + router weights) over routing + expert-kernel time of the
    calls without misses (the survey's decode metric with fills excluded)."""
    eb = entry_bytes(wl)
    router_bytes = wl["E"] * wl["d"] * 2
    out = {}
    h_ms, h_n, h_items = prof["experts_hit"]
    m_ms, m_n, m_items = prof["experts_miss"]
    r_ms, r_n, _ = prof["router"]
    out["experts_hit"] = dict(ms=h_ms, launches=h_n, bytes=h_items * eb,
                              achieved=(h_items * eb / (h_ms / 1e3) / 1e9) if h_ms > 0 else 0.0)
    out["experts_miss"] = dict(ms=m_ms, launches=m_n, hbm_bytes=m_items * eb)
    route_per_call = r_ms / r_n if r_n else 0.0
    t_m2 = h_ms + route_per_call * h_n
    b_m2 = h_items * eb + h_n * router_bytes
    out["step_m2"] = dict(bytes=b_m2, ms=t_m2,
                          achieved=(b_m2 / (t_m2 / 1e3) / 1e9) if t_m2 > 0 else 0.0)
    out["route_us_per_call"] = route_per_call * 1e3
    return out


def run_decode(args, wl, rank, world):
    import torch
    pk = peaks()
    seed = SEED + rank
    pool = build_pool(wl, seed)
    h2d_gbs = measure_h2d()
    per_batch = {}
    head = None
    eb = entry_bytes(wl)
    for b in wl["batches"]:
        res, x_all, bias_all = bench_decode_batch(wl, pool, b, args.warmup, args.steps, seed,
                                                  world)
        res["ms"] = max_over_ranks(res["ms"], world)
        res["tok_s_all"] = world * b * args.steps / (res["ms"] / 1e3)
        prof_k = min(args.steps, args.profile_steps)
        prof, touched, fill_bytes, n_calls = profile_decode_batch(
            wl, pool, b, x_all, bias_all, args.warmup, prof_k, seed)
        rl = roofline_decode(wl, prof, pk)
        res["kernels_ms_per_step"] = {c: v[0] / prof_k for c, v in prof.items() if v[1]}
        res["launches_per_step"] = {c: v[1] / prof_k for c, v in prof.items() if v[1]}
        res["experts_hit_gbs"] = rl["experts_hit"]["achieved"]
        res["step_m2_gbs"] = rl["step_m2"]["achieved"]
        res["route_us_per_call"] = rl["route_us_per_call"]
        miss_ms = rl["experts_miss"]["ms"]
        res["fill_gbs"] = fill_bytes / (miss_ms / 1e3) / 1e9 if miss_ms > 0 else None
        e2e = bench_decode_e2e(wl, pool, b, x_all, bias_all, args.warmup, args.steps, seed, world)
        e2e["ms"] = max_over_ranks(e2e["ms"], world)
        res["e2e_tok_s_all"] = world * b * args.steps / (e2e["ms"] / 1e3)
        res["e2e"] = e2e
        per_batch[b] = res
        if b == wl["headline_b"]:
            head = (res, rl, prof, prof_k, bias_all, fill_bytes)
        del x_all, bias_all
        torch.cuda.empty_cache()
    res, rl, prof, prof_k, bias_all, fill_bytes = head
    b = wl["headline_b"]
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        calls, el = cpu_oracle_decode(wl, pool, b, bias_all.cpu().numpy(), seed,
                                      budget_s=args.cpu_budget)
        cpu = {"value": b * calls / wl["L"] / el, "unit": "tokens/s", "cores": 1,
               "kind": "oracle", "host_cores": os.cpu_count(),
               "sample": f"first {calls} layer calls of the b={b} trace "
                         f"({calls / wl['L']:.2f} decode steps), {el:.1f} s, numpy fp32 router "
                         f"+ fp64 experts, single thread (the box has {os.cpu_count()} cores)"}
    eh = rl["experts_hit"]
    kname = "k_decode_experts<mxfp4>" if wl.get("fp4") else "k_decode_experts"
    traffic = None
    if args.workload == "decode24" and b == 1 and not wl.get("fp4") and TRAFFIC_DECODE24_B1:
        traffic = TRAFFIC_DECODE24_B1
    roof = {"bound": "hbm",
            "kernel": f"{kname} (gate/up + SwiGLU + down + combine; fills when the call misses), "
                      "launches of calls without misses",
            "achieved": round(eh["achieved"], 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": round(eh["achieved"] / pk["hbm_gbs"], 4), "traffic": traffic,
            "peak_source": pk["source"],
            "frac_of_8tbs": round(eh["achieved"] / 8000.0, 4),
            "launches": eh["launches"],
            "algorithmic_bytes": ("entries streamed x 3*d*d_ff*17/32 B (MXFP4 codes + scales)"
                                  if wl.get("fp4") else
                                  f"entries streamed x 3*d*d_ff*2 B = {eb / 1e6:.2f} MB per entry"
                                  " (touched experts + shared)")}
    m2 = rl["step_m2"]
    fill = {"fill_gbs": round(fill_bytes / (rl["experts_miss"]["ms"] / 1e3) / 1e9, 2)
            if rl["experts_miss"]["ms"] > 0 else None,
            "h2d_gbs": round(h2d_gbs, 2),
            "h2d_how": "pinned cudaMemcpyAsync host -> device of 1 GiB, best of 5, this run",
            "fill_how": "missed-entry bytes over the time of the expert launches of calls with "
                        "misses (their hit experts overlap the fills)"}
    if fill["fill_gbs"]:
        fill["frac"] = round(fill["fill_gbs"] / h2d_gbs, 4)
    line = {
        "metric": "MoE-layer tokens/s (decode trace, b=1"
                  + (", MXFP4 experts" if wl.get("fp4") else "")
                  + (", frequency admission)" if wl.get("admission") else ")"),
        "value": round(res["tok_s_all"], 2), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(res["ms"] / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "mxfp4 weights, bf16 activations, fp32 accumulate" if wl.get("fp4") else "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "layers": wl["L"], "d": wl["d"],
                   "d_ff": wl["d_ff"], "experts": wl["E"], "top_k": wl["k"],
                   "n_slots": wl["n_slots"], "batch": b, "graph": True,
                   "admission": bool(wl.get("admission")),
                   "weights": "mxfp4" if wl.get("fp4") else "bf16",
                   "l2": "inputs larger than L2 (every step streams "
                         f">{wl['L'] * wl['k'] * eb / 1e9:.2f} GB of experts)",
                   "parallelism": f"replicas x{world}",
                   "per_batch": {str(bb): {k: (round(v, 4) if isinstance(v, float) else v)
                                           for k, v in r.items()
                                           if k not in ("clocks", "e2e")}
                                 for bb, r in per_batch.items()}},
        "roofline": roof,
        "decode_step_m2": {"achieved": round(m2["achieved"], 1), "unit": "GB/s",
                           "frac": round(m2["achieved"] / pk["hbm_gbs"], 4),
                           "frac_of_8tbs": round(m2["achieved"] / 8000.0, 4),
                           "what": "touched entries + router weights over routing + expert "
                                   "kernel time, calls without misses"},
        "fill": fill,
        "cpu_baseline": cpu,
        "e2e": {"value": round(res["e2e_tok_s_all"], 2), "unit": "tokens/s",
                "h2d_bytes_per_step": res["e2e"]["h2d"], "d2h_bytes_per_step": res["e2e"]["d2h"]},
        # kernels per decode layer call: routing + control, and the expert kernel
        "gpu_launches": int(sum(v[1] for v in prof.values()) / prof_k * args.steps),
        "clocks": res["clocks"],
    }
    if args.workload == "decode24" and not args.no_prefill and not wl.get("fp4"):
        del pool
        import gc
        gc.collect()
        if hasattr(torch._C, "_host_emptyCache"):
            torch._C._host_emptyCache()
        pl = run_prefill(args, dict(WORKLOADS["prefill8"]), rank, world, steps=1)
        line["prefill"] = {t: {k: v for k, v in r.items()
                               if k in ("tok_s", "ms_per_prefill", "gemm_ms_per_layer",
                                        "gemm_tflops", "tc_frac", "tc_frac_sustained",
                                        "overlap", "h2d_gbs", "copy_ms", "compute_ms",
                                        "wall_ms", "router_ms_per_layer")}
                           for t, r in pl["config"]["per_T"].items()}
        line["prefill"]["workload"] = "prefill8: 8 layers, d=4096, d_ff=2048, E=256, top-6"
        line["prefill"]["peak_tflops"] = pk["bf16"]
        line["prefill"]["peak_tflops_sustained"] = pk["bf16_sustained"]
    return line


# ----------------------------------------------------------------------------------------
# prefill benchmark
# ----------------------------------------------------------------------------------------
def run_prefill(args, wl, rank, world, steps=None):
    """Prefill streaming: every layer's full expert set is copied host -> device into the back
    buffer while the previous layer computes.  A step is one prefill over all L layers."""
    import torch
    import ft_synth.gpu as sg
    pk = peaks()
    seed = SEED + rank
    pool = build_pool(wl, seed)
    L, d, d_ff, k = wl["L"], wl["d"], wl["d_ff"], wl["k"]
    K = steps or max(1, min(args.steps, args.prefill_steps))
    W = 1
    per_T = {}
    for T in wl["tokens"]:
        st = make_stack(wl, pool, seed, max_tokens=T)
        x = torch.empty((T, d), dtype=torch.int16, device="cuda")
        sg.activations_device(x.data_ptr(), seed, [7_000_000 + T], T, d,
                              torch.cuda.current_stream().cuda_stream)
        out = torch.empty((L, T, d), dtype=torch.int16, device="cuda")
        for _ in range(W):
            st.prefill(0, L, x, out)
        torch.cuda.synchronize()
        barrier(world)
        copy_ms = comp_ms = wall_ms = 0.0
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(torch.cuda.current_device()) as clk:
            e0.record()
            for _ in range(K):
                st.prefill(0, L, x, out)
                c, kk, w = st.prefill_timing()
                copy_ms += c
                comp_ms += kk
                wall_ms += w
            e1.record()
            torch.cuda.synchronize()
        ms = max_over_ranks(e0.elapsed_time(e1), world)
        # GEMM time alone (one profiled prefill)
        st.profile(True)
        st.profile_read()
        st.prefill(0, L, x, out)
        prof = st.profile_read()
        st.profile(False)
        flops = 2.0 * 3 * d * d_ff * T * k * L
        gemm_ms = prof["gateup"][0] + prof["down"][0]
        tflops = flops / (gemm_ms / 1e3) / 1e12 if gemm_ms > 0 else 0.0
        router_ms = prof["router"][0] + prof["topk"][0] + prof["control"][0]
        overlap = (copy_ms + comp_ms - wall_ms) / max(1e-9, min(copy_ms, comp_ms))
        h2d_b, d2d_b = st.prefill_bytes()
        per_T[T] = dict(ms_per_prefill=ms / K, tok_s=world * T * K / (ms / 1e3),
                        gemm_ms_per_layer=gemm_ms / L, gemm_tflops=tflops,
                        tc_frac=tflops / pk["bf16"],
                        tc_frac_sustained=tflops / pk["bf16_sustained"]
                        if pk.get("bf16_sustained") else None,
                        router_ms_per_layer=router_ms / L, copy_ms=copy_ms / K,
                        compute_ms=comp_ms / K, wall_ms=wall_ms / K, overlap=overlap,
                        h2d_gbs=h2d_b / (copy_ms / K / 1e3) / 1e9,
                        h2d_gb_per_prefill=h2d_b / 1e9, d2d_gb_per_prefill=d2d_b / 1e9,
                        kernels_ms={c: v[0] for c, v in prof.items()}, clocks=clk.summary())
        st.close()
        del x, out
        torch.cuda.empty_cache()
    Th = wl["tokens"][-1]
    r = per_T[Th]
    return {
        "metric": f"MoE-layer prefill tokens/s (T={Th}, 8 layers streamed"
                  + (", cache top-up)" if wl.get("topup") else ")"),
        "value": round(r["tok_s"], 1), "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(r["ms_per_prefill"], 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "layers": L, "d": d, "d_ff": d_ff,
                   "experts": wl["E"], "top_k": k, "tokens": list(wl["tokens"]),
                   "per_T": {str(t): {kk: (round(v, 4) if isinstance(v, float) else v)
                                      for kk, v in rr.items()} for t, rr in per_T.items()}},
        "roofline": {"bound": "tensor", "kernel": "grouped GEMM gate/up + down",
                     "achieved": round(r["gemm_tflops"], 1), "peak": pk["bf16"],
                     "unit": "TFLOP/s", "frac": round(r["tc_frac"], 4), "traffic": None,
                     "peak_source": pk["source"]},
        "e2e": None, "clocks": r["clocks"],
    }


# ----------------------------------------------------------------------------------------
# placement-policy replay
# ----------------------------------------------------------------------------------------
def run_policy(args, wl, rank, world):
    """Miss rates of the device LRU against a static layer split and a hot set refreshed every
    `refresh` steps, at the same capacity, on the decode trace the CUDA path routes."""
    import torch
    from expert_cached_routed_router_b300.policy import RefreshedHotSet, StaticLayerSplit, miss_rate
    seed = SEED + rank
    pool = build_pool(wl, seed)
    L, E, k = wl["L"], wl["E"], wl["k"]
    n = wl["steps"] if args.steps == 200 else args.steps
    res = {}
    for b in wl["batches"]:
        x_all, bias_all, _ = decode_trace(wl, b, n, seed)
        st = make_stack(wl, pool, seed, max_tokens=16)
        out = torch.empty((b, wl["d"]), dtype=torch.int16, device="cuda")
        static = StaticLayerSplit(L, E, wl["n_slots"])
        hot = RefreshedHotSet(L, E, wl["n_slots"], wl["refresh"])
        for t in range(n):
            static.step_begin(t)
            hot.step_begin(t)
            st.set_router_bias(-1, bias_all[t])
            for l in range(L):
                st.forward(l, x_all[t], out)
                idx, _, _ = st.routing(b)
                static.access(l, idx.ravel())
                hot.access(l, idx.ravel())
        s = st.stats()
        st.close()
        # the same trace through the device cache with frequency admission (every miss,
        # cached or staged, crosses the host link)
        sta = make_stack(dict(wl, admission=1), pool, seed, max_tokens=16)
        for t in range(n):
            sta.set_router_bias(-1, bias_all[t])
            for l in range(L):
                sta.forward(l, x_all[t], out)
        sa = sta.stats()
        sta.close()
        res[str(b)] = {"lru_miss_rate": round(s["misses"] / max(1, s["hits"] + s["misses"]), 4),
                       "lru_admission_miss_rate": round(sa["misses"] / max(1, sa["hits"] + sa["misses"]), 4),
                       "lru_admission_bypass_share": round(sa["bypasses"] / max(1, sa["misses"]), 4),
                       "static_layer_split_miss_rate": round(miss_rate(static), 4),
                       "refreshed_hot_set_miss_rate": round(miss_rate(hot), 4),
                       "accesses": s["hits"] + s["misses"]}
    return {"metric": "decode expert miss rate by placement policy (same capacity, same trace)",
            "value": res[str(wl["batches"][0])]["lru_miss_rate"], "unit": "fraction",
            "higher_is_better": False, "n_gpus": world, "steps": n, "warmup": 0,
            "data": "synthetic",
            "config": {"workload": "policy", "layers": L, "experts": E, "top_k": k,
                       "capacity": wl["n_slots"], "refresh_steps": wl["refresh"],
                       "by_batch": res}}


# ----------------------------------------------------------------------------------------
# elastic-cache stress
# ----------------------------------------------------------------------------------------
def run_elastic(args, wl, rank, world):
    """10,000 decode steps of the 24-layer shapes: b = 1 in the first half of every block of
    1,000 steps and b = 8 in the second, the popularity order switching between two disjoint
    Zipf orders every 1,000 steps, and ft_cache_resize at the safe points before steps 3,500
    (768 -> 307 slots) and 6,500 (307 -> 1,228).  Each batch size runs as its own CUDA graph."""
    import torch
    import ft_synth
    import ft_synth.gpu as sg
    seed = SEED + rank
    pool = build_pool(wl, seed)
    L, E, d = wl["L"], wl["E"], wl["d"]
    n = min(wl["steps"], args.steps) if args.steps != 200 else wl["steps"]
    gen = ft_synth.DriftingZipfBias(seed, L, E, s=wl["zipf"], phase_len=wl["phase"])
    bias = np.empty((n, L, E), np.float32)
    for t in range(n):
        gen.advance()
        for l in range(L):
            bias[t, l] = gen.bias(l)
    bias_d = torch.from_numpy(bias).cuda()
    batch = [1 if (t % 1000) < 500 else 8 for t in range(n)]
    x = {b: torch.empty((n, b, d), dtype=torch.int16, device="cuda") for b in (1, 8)}
    for b in (1, 8):
        sg.activations_device(x[b].data_ptr(), seed, [1_000_000 * b + t for t in range(n)], b, d,
                              torch.cuda.current_stream().cuda_stream)
    st = make_stack(wl, pool, seed, max_tokens=16)
    xs = {b: torch.empty((b, d), dtype=torch.int16, device="cuda") for b in (1, 8)}
    bs = torch.empty((L, E), dtype=torch.float32, device="cuda")
    out = {b: torch.empty((L, b, d), dtype=torch.int16, device="cuda") for b in (1, 8)}
    graphs = {}
    for b in (1, 8):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            st.set_router_bias(-1, bs)
            for l in range(L):
                st.forward(l, xs[b], out[b][l])
        graphs[b] = g
    resizes = dict(wl["resizes"])
    phase_stats = []
    resize_ms = []
    tokens = 0
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    s_prev = st.stats()
    for t in range(n):
        if t in resizes:
            r0 = time.perf_counter()
            st.resize(resizes[t])
            resize_ms.append((t, resizes[t], (time.perf_counter() - r0) * 1e3))
            # the captured decode graphs stay valid: their kernels find the new slot storage
            # through the library's device-side cache descriptor
        b = batch[t]
        xs[b].copy_(x[b][t])
        bs.copy_(bias_d[t])
        graphs[b].replay()
        tokens += b
        if (t + 1) % 500 == 0:
            s = st.stats()
            dh, dm = s["hits"] - s_prev["hits"], s["misses"] - s_prev["misses"]
            phase_stats.append(dict(steps=f"{t - 499}-{t}", b=b, hit_rate=round(dh / max(1, dh + dm), 4),
                                    n_slots=s["n_slots"]))
            s_prev = s
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier(world)
    wall = max_over_ranks(wall, world)
    s = st.stats()
    assert s["status"] == 0, s
    st.close()
    return {
        "metric": "MoE-layer tokens/s (elastic-cache stress trace, b=1/8, resizes)",
        "value": round(world * tokens / wall, 2), "unit": "tokens/s", "n_gpus": world,
        "steps": n, "warmup": 0, "ms_per_step": round(wall * 1e3 / n, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "elastic", "layers": L, "d": d, "d_ff": wl["d_ff"], "experts": E,
                   "top_k": wl["k"], "slots": [768, 307, 1228], "resize_ms": resize_ms,
                   "hit_rate_by_500_steps": phase_stats, "hits": s["hits"],
                   "misses": s["misses"], "evictions": s["evictions"],
                   "timing": "host wall clock around the whole trace (includes the resizes)"},
    }


# ----------------------------------------------------------------------------------------
# reference arm: the CPU oracle on the same workload
# ----------------------------------------------------------------------------------------
def run_reference(args, wl, rank, world):
    import torch
    if rank != 0:
        return None
    b = wl["headline_b"]
    seed = SEED
    n = wl["L"] * wl["E"] * 3 * wl["d"] * wl["d_ff"]
    import ft_synth.gpu as sg
    sg.build()
    pool = torch.empty(n, dtype=torch.int16, pin_memory=True)
    sg.fill_pool(pool.data_ptr(), seed, wl["L"], wl["E"], wl["d"], wl["d_ff"])
    n_steps = (args.warmup + args.steps) // wl["L"] + 2
    import ft_synth
    gen = ft_synth.DriftingZipfBias(seed, wl["L"], wl["E"], s=wl["zipf"])
    bias = np.empty((n_steps, wl["L"], wl["E"]), np.float32)
    for t in range(n_steps):
        gen.advance()
        for l in range(wl["L"]):
            bias[t, l] = gen.bias(l)
    cpu_oracle_decode(wl, pool, b, bias, seed, max_calls=max(1, args.warmup))
    t0 = time.perf_counter()
    calls, el = cpu_oracle_decode(wl, pool, b, bias, seed, max_calls=args.steps)
    tok_s = b * calls / wl["L"] / el
    return {
        "impl": "reference", "metric": "MoE-layer tokens/s (decode trace, b=1)",
        "value": round(tok_s, 4), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(el * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "layers": wl["L"], "d": wl["d"],
                   "d_ff": wl["d_ff"], "experts": wl["E"], "top_k": wl["k"],
                   "n_slots": wl["n_slots"], "batch": b,
                   "step": "one layer call of the b=1 decode trace (oracle)"},
        "cpu_baseline": {"value": round(tok_s, 4), "unit": "tokens/s", "cores": 1,
                         "kind": "oracle",
                         "sample": f"{calls} layer calls of the b={b} trace, single thread"},
        "e2e": {"value": round(tok_s, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decode24")
    ap.add_argument("--profile-steps", type=int, default=100)
    ap.add_argument("--prefill-steps", type=int, default=2)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="leave the prefill block out of the decode line")
    ap.add_argument("--batches", default="", help="comma list of decode batch sizes")
    ap.add_argument("--slots", type=int, default=0, help="override the slot count")
    ap.add_argument("--fp4", action="store_true",
                    help="MXFP4 expert entries (decode workloads only)")
    ap.add_argument("--admission", action="store_true",
                    help="frequency admission: misses that would displace a more frequently "
                         "used entry are staged for one call instead of cached")
    ap.add_argument("--experts", type=int, default=0, help="override E (profiling cases)")
    ap.add_argument("--layers", type=int, default=0, help="override L (profiling cases)")
    ap.add_argument("--tokens", default="", help="prefill token counts, comma list")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    wl = dict(WORKLOADS[args.workload])
    if args.batches:
        wl["batches"] = tuple(int(v) for v in args.batches.split(","))
        if wl.get("headline_b") not in wl["batches"]:
            wl["headline_b"] = wl["batches"][0]
    if args.slots:
        wl["n_slots"] = args.slots
    if args.admission:
        wl["admission"] = 1
    if args.fp4:
        wl["fp4"] = 1
    if args.experts:
        wl["E"] = args.experts
    if args.layers:
        wl["L"] = args.layers
    if args.tokens:
        wl["tokens"] = tuple(int(v) for v in args.tokens.split(","))
    import torch
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        line = run_reference(args, wl, rank, int(os.environ.get("WORLD_SIZE", "1")))
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    rank, world, _ = dist_setup(args)
    import expert_cached_routed_router_b300 as ftm
    ftm.load_library()
    if args.workload in ("prefill8", "prefill8_topup"):
        line = run_prefill(args, wl, rank, world)
    elif args.workload == "elastic":
        line = run_elastic(args, wl, rank, world)
    elif args.workload == "policy":
        line = run_policy(args, wl, rank, world)
    else:
        line = run_decode(args, wl, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
