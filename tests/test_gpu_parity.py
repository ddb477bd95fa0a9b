"""Parity of the CUDA path with the oracle on small seeded configurations (GPU)."""
import numpy as np
import pytest

import ft_synth
from oracle import lru as olru
from oracle import moe as omoe

from helpers import (Config, assert_cache_equal, assert_out_close, assert_routing_equal,
                     gpu_host_pool, make_stack, oracle_layer, out_bits_to_f64, to_dev_bf16)

pytestmark = pytest.mark.gpu


def _run(st, l, x_bits):
    import torch
    x = to_dev_bf16(x_bits)
    out = torch.empty_like(x)
    st.forward(l, x, out)
    torch.cuda.synchronize()
    return out


def test_tiny_layer_all_resident():
    """d=256, d_ff=128, E=16 top-2, 64 tokens, 16 slots prewarmed: no misses, all bit-exact."""
    cfg = Config(L=1, E=16, k=2, d=256, d_ff=128, n_slots=16)
    st = make_stack(cfg, max_tokens=64)
    x = ft_synth.activations(0, 0, 64, 256)
    out = _run(st, 0, x)
    ref = oracle_layer(cfg, 0, x)
    np.testing.assert_array_equal(st.logits(64).view(np.uint32), ref["logits"].view(np.uint32))
    assert_routing_equal(st, ref, 64)
    assert_out_close(out_bits_to_f64(out), ref["out"])
    s = st.stats()
    assert s["misses"] == 0 and s["hits"] == len(set(ref["idx"].ravel())) and s["status"] == 0
    assert len(st.fills()) == 0
    st.close()


@pytest.mark.parametrize("T", [1, 3, 4, 5, 16, 17, 40, 300])
def test_layer_token_counts(T):
    """GEMV path (T <= 16) and grouped-GEMM path (T > 16), ragged expert groups."""
    cfg = Config(L=2, E=32, k=4, d=512, d_ff=384, n_slots=64, seed=1)
    st = make_stack(cfg, max_tokens=512)
    for l in range(2):
        x = ft_synth.activations(1, 100 * T + l, T, cfg.d)
        out = _run(st, l, x)
        ref = oracle_layer(cfg, l, x)
        np.testing.assert_array_equal(st.logits(T).view(np.uint32),
                                      ref["logits"].view(np.uint32))
        assert_routing_equal(st, ref, T)
        assert_out_close(out_bits_to_f64(out), ref["out"])
    assert st.status() == 0
    st.close()


@pytest.mark.parametrize("E,k,T,n_slots", [
    (512, 8, 16, 200),    # T*E > 4096: the fused decode kernel falls back to warp top-k
    (1024, 32, 1, 300),   # largest E and k, in-CTA top-k
    (1024, 32, 4, 300),   # T*E = 4096, the in-CTA limit
    (1024, 32, 5, 300),   # just past it
])
def test_decode_edge_shapes(E, k, T, n_slots):
    """Decode calls at the limits of the in-CTA top-k and of E and k, with evictions: routing,
    grouping, fills and the whole cache state bit-exact; outputs within tolerance."""
    cfg = Config(L=2, E=E, k=k, d=128, d_ff=128, n_slots=n_slots, seed=12)
    st = make_stack(cfg, max_tokens=16, pool=gpu_host_pool(cfg))
    sim = olru.SlotCacheSim(cfg.L, cfg.E, cfg.n_slots, cfg.entry_bytes, prewarm=True)
    for step in range(3):
        for l in (1, 0):
            x = ft_synth.activations(12, 1000 * T + 10 * step + l, T, cfg.d)
            out = _run(st, l, x)
            ref = oracle_layer(cfg, l, x, tokens=np.arange(min(T, 3)))
            assert_routing_equal(st, ref, T)
            code, hits, fills = sim.access(l, ref["idx"].ravel())
            assert code == olru.OK
            np.testing.assert_array_equal(st.fills(), np.array([f[:3] for f in fills],
                                                                dtype=np.int32).reshape(-1, 3))
            assert_cache_equal(st, sim)
            assert_out_close(out_bits_to_f64(out)[ref["tokens"]], ref["out"])
    assert sim.evictions > 0 and st.status() == 0
    st.close()


@pytest.mark.parametrize("T,d_ff,shared", [(16, 2048, 1), (4, 512, 1), (1, 2048, 0)])
def test_decode_misses_with_shared_expert_every_row(T, d_ff, shared):
    """Decode calls with misses (and a shared expert) at 16, 4 and 1 tokens with d_ff = 2048
    and 512: routing, fills and cache state bit-exact, every output row within tolerance."""
    cfg = Config(L=2, E=24, k=4, d=256, d_ff=d_ff, n_slots=24, n_shared=shared, seed=14)
    st = make_stack(cfg, max_tokens=16, pool=gpu_host_pool(cfg))
    sim = olru.SlotCacheSim(cfg.L, cfg.E, cfg.n_slots, cfg.entry_bytes, prewarm=True)
    for step in range(4):
        for l in (0, 1):
            x = ft_synth.activations(14, 100 * T + 10 * step + l, T, cfg.d)
            out = _run(st, l, x)
            ref = oracle_layer(cfg, l, x)
            assert_routing_equal(st, ref, T)
            code, hits, fills = sim.access(l, ref["idx"].ravel())
            assert code == olru.OK
            np.testing.assert_array_equal(st.fills(), np.array([f[:3] for f in fills],
                                                                dtype=np.int32).reshape(-1, 3))
            assert_cache_equal(st, sim)
            assert_out_close(out_bits_to_f64(out), ref["out"])
    assert sim.misses > 0 and st.status() == 0
    st.close()


def test_victims_beyond_shared_memory_staging():
    """More than 2,048 slots: the control reads the eviction keys from global memory."""
    cfg = Config(L=40, E=64, k=4, d=128, d_ff=128, n_slots=2100, seed=13)
    st = make_stack(cfg, max_tokens=16, pool=gpu_host_pool(cfg))
    sim = olru.SlotCacheSim(cfg.L, cfg.E, cfg.n_slots, cfg.entry_bytes, prewarm=True)
    for step in range(6):
        for l in (39, 35, 3):
            x = ft_synth.activations(13, 10 * step + l, 4, cfg.d)
            out = _run(st, l, x)
            want = step % 3 == 0
            ref = oracle_layer(cfg, l, x, tokens=None if want else [])
            assert_routing_equal(st, ref, 4)
            code, hits, fills = sim.access(l, ref["idx"].ravel())
            assert code == olru.OK
            np.testing.assert_array_equal(st.fills(), np.array([f[:3] for f in fills],
                                                                dtype=np.int32).reshape(-1, 3))
            assert_cache_equal(st, sim)
            if want:
                assert_out_close(out_bits_to_f64(out), ref["out"])
    assert sim.evictions > 0 and st.status() == 0
    st.close()


def test_large_P_multi_cta_permutation():
    """P = T*k > 1024 takes the multi-CTA grouping kernels."""
    cfg = Config(L=1, E=64, k=6, d=256, d_ff=128, n_slots=64, seed=2)
    T = 700
    st = make_stack(cfg, max_tokens=T)
    x = ft_synth.activations(2, 0, T, cfg.d)
    out = _run(st, 0, x)
    ref = oracle_layer(cfg, 0, x, tokens=np.arange(0, T, 7))
    assert_routing_equal(st, ref, T)
    assert_out_close(out_bits_to_f64(out)[ref["tokens"]], ref["out"])
    st.close()


@pytest.mark.parametrize("T", [1, 4, 6])
def test_decode_trace_lru_bit_exact(T):
    """A drifting-Zipf decode trace with evictions: routing, fills and the whole cache state
    match the oracle simulator after every call; outputs within tolerance on every call."""
    cfg = Config(L=3, E=16, k=2, d=256, d_ff=128, n_slots=12, seed=3)
    st = make_stack(cfg, max_tokens=16)
    sim = olru.SlotCacheSim(cfg.L, cfg.E, cfg.n_slots, cfg.entry_bytes, prewarm=True)
    assert_cache_equal(st, sim)
    gen = ft_synth.DriftingZipfBias(3, cfg.L, cfg.E, s=0.8, sigma_walk=0.3)
    import torch
    n_fills = 0
    for step in range(25):
        gen.advance()
        x = ft_synth.activations(3, step, T, cfg.d)
        for l in range(cfg.L):
            b = gen.bias(l)
            st.set_router_bias(l, torch.from_numpy(b).cuda())
            out = _run(st, l, x)
            ref = oracle_layer(cfg, l, x, bias=b)
            assert_routing_equal(st, ref, T)
            st_code, hits, fills = sim.access(l, ref["idx"].ravel())
            assert st_code == olru.OK
            got = st.fills()
            np.testing.assert_array_equal(got, np.array([f[:3] for f in fills],
                                                        dtype=np.int32).reshape(-1, 3))
            n_fills += len(fills)
            assert_cache_equal(st, sim)
            assert_out_close(out_bits_to_f64(out), ref["out"])
    s = st.stats()
    assert s["misses"] == sim.misses == n_fills and s["hits"] == sim.hits
    assert s["evictions"] == sim.evictions and s["status"] == 0
    assert sim.evictions > 0
    st.close()


@pytest.mark.parametrize("T", [1, 4, 40])
def test_admission_trace_bit_exact(T):
    """Frequency admission on a skewed, drifting trace: every call's routing, fill list
    (bypassed misses staged in entries n_slots + b) and the whole cache state match the
    oracle simulator; outputs (bypassed experts read from staging) within tolerance."""
    import torch
    cfg = Config(L=3, E=16, k=2, d=256, d_ff=128, n_slots=10, seed=4)
    st = make_stack(cfg, max_tokens=64, admission=1)
    sim = olru.SlotCacheSim(cfg.L, cfg.E, cfg.n_slots, cfg.entry_bytes, prewarm=True,
                            admission=True)
    gen = ft_synth.DriftingZipfBias(4, cfg.L, cfg.E, s=1.2, sigma_walk=0.3)
    for step in range(40):
        gen.advance()
        x = ft_synth.activations(4, 500 + step, T, cfg.d)
        for l in range(cfg.L):
            b = gen.bias(l)
            st.set_router_bias(l, torch.from_numpy(b).cuda())
            out = _run(st, l, x)
            ref = oracle_layer(cfg, l, x, bias=b, tokens=np.arange(min(T, 6)))
            assert_routing_equal(st, ref, T)
            code, hits, fills = sim.access(l, ref["idx"].ravel())
            assert code == olru.OK
            np.testing.assert_array_equal(st.fills(), np.array([f[:3] for f in fills],
                                                                dtype=np.int32).reshape(-1, 3))
            assert_cache_equal(st, sim)
            assert_out_close(out_bits_to_f64(out)[ref["tokens"]], ref["out"])
    s = st.stats()
    assert s["bypasses"] == sim.bypasses > 0 and s["misses"] == sim.misses
    assert s["evictions"] == sim.evictions and s["hits"] == sim.hits and s["status"] == 0
    st.close()


@pytest.mark.parametrize("T,admission", [(1, 0), (4, 0), (16, 0), (4, 1)])
def test_mxfp4_decode_trace(T, admission):
    """MXFP4 entries: a drifting decode trace with evictions (fills move the 4-bit entries);
    routing, fills and cache state bit-exact; outputs against the oracle's expert network on
    the dequantized weights, within tolerance."""
    import torch
    cfg = Config(L=3, E=16, k=2, d=256, d_ff=384, n_slots=10, seed=14, fp4=True)
    st = make_stack(cfg, max_tokens=16, admission=admission)
    sim = olru.SlotCacheSim(cfg.L, cfg.E, cfg.n_slots, cfg.entry_bytes, prewarm=True,
                            admission=bool(admission))
    gen = ft_synth.DriftingZipfBias(14, cfg.L, cfg.E, s=1.0, sigma_walk=0.3)
    for step in range(8):
        gen.advance()
        x = ft_synth.activations(14, 300 + step, T, cfg.d)
        for l in range(cfg.L):
            b = gen.bias(l)
            st.set_router_bias(l, torch.from_numpy(b).cuda())
            out = _run(st, l, x)
            ref = oracle_layer(cfg, l, x, bias=b, tokens=np.arange(min(T, 4)))
            assert_routing_equal(st, ref, T)
            code, hits, fills = sim.access(l, ref["idx"].ravel())
            assert code == olru.OK
            np.testing.assert_array_equal(st.fills(), np.array([f[:3] for f in fills],
                                                                dtype=np.int32).reshape(-1, 3))
            assert_cache_equal(st, sim)
            assert_out_close(out_bits_to_f64(out)[ref["tokens"]], ref["out"])
    s = st.stats()
    assert s["misses"] == sim.misses > 0 and s["status"] == 0
    assert s["fill_bytes"] == sim.misses * cfg.entry_bytes
    st.close()


@pytest.mark.parametrize("fp4", [False, True])
def test_admission_across_resizes(fp4):
    """Admission counts survive resizes (shrink, then grow past the start), with bf16 and
    MXFP4 entries: fills, cache state and counters bit-exact against the oracle simulator."""
    import torch
    cfg = Config(L=3, E=16, k=2, d=256, d_ff=256, n_slots=12, seed=16, fp4=fp4)
    st = make_stack(cfg, max_tokens=16, admission=1)
    sim = olru.SlotCacheSim(cfg.L, cfg.E, cfg.n_slots, cfg.entry_bytes, prewarm=True,
                            admission=True)
    gen = ft_synth.DriftingZipfBias(16, cfg.L, cfg.E, s=1.1, sigma_walk=0.3)
    resizes = {10: 5, 20: 30}
    for step in range(30):
        if step in resizes:
            st.resize(resizes[step])
            sim.resize(resizes[step])
            assert_cache_equal(st, sim)
        gen.advance()
        x = ft_synth.activations(16, 700 + step, 4, cfg.d)
        for l in range(cfg.L):
            b = gen.bias(l)
            st.set_router_bias(l, torch.from_numpy(b).cuda())
            out = _run(st, l, x)
            want = step % 10 == 9
            ref = oracle_layer(cfg, l, x, bias=b, tokens=None if want else [])
            code, hits, fills = sim.access(l, ref["idx"].ravel())
            assert code == olru.OK
            np.testing.assert_array_equal(st.fills(), np.array([f[:3] for f in fills],
                                                                dtype=np.int32).reshape(-1, 3))
            assert_cache_equal(st, sim)
            if want:
                assert_out_close(out_bits_to_f64(out), ref["out"])
    s = st.stats()
    assert s["bypasses"] == sim.bypasses > 0 and s["evictions"] == sim.evictions
    assert s["status"] == 0 and s["resizes"] == 2
    st.close()


@pytest.mark.parametrize("T", [17, 40, 300, 700])
def test_mxfp4_grouped_gemm(T):
    """MXFP4 entries in calls with more tokens than the decode path takes: the touched entries
    (after their fills) are expanded to bf16 and run through the tcgen05 grouped GEMMs.
    Routing, fills and cache state bit-exact; every output row within tolerance of the oracle's
    expert network on the dequantized weights (T = 700 gives 3+ M-tiles per group)."""
    cfg = Config(L=2, E=8, k=2, d=256, d_ff=384, n_slots=10, seed=15, fp4=True)
    st = make_stack(cfg, max_tokens=1024)
    sim = olru.SlotCacheSim(cfg.L, cfg.E, cfg.n_slots, cfg.entry_bytes, prewarm=True)
    for l in (1, 0, 1):
        x = ft_synth.activations(15, 10 * T + l, T, cfg.d)
        out = _run(st, l, x)
        ref = oracle_layer(cfg, l, x)
        assert_routing_equal(st, ref, T)
        code, hits, fills = sim.access(l, ref["idx"].ravel())
        assert code == olru.OK
        np.testing.assert_array_equal(st.fills(), np.array([f[:3] for f in fills],
                                                            dtype=np.int32).reshape(-1, 3))
        assert_cache_equal(st, sim)
        assert_out_close(out_bits_to_f64(out), ref["out"])
    assert sim.misses > 0 and st.status() == 0
    st.close()


def test_mxfp4_prefill():
    """MXFP4 prefill: the double buffer carries the 4-bit entries over the host link (17/32 of
    the bf16 bytes), each layer is expanded to bf16 for the grouped GEMMs; residual stream and
    teacher-forced oracle as for bf16 entries."""
    import torch
    cfg = Config(L=3, E=8, k=2, d=256, d_ff=256, n_slots=4, seed=19, fp4=True)
    T = 300
    st = make_stack(cfg, max_tokens=T)
    x = ft_synth.activations(19, 0, T, cfg.d)
    out = torch.empty((cfg.L, T, cfg.d), dtype=torch.int16, device="cuda")
    st.prefill(0, cfg.L, to_dev_bf16(x), out)
    torch.cuda.synchronize()
    xin = x
    for l in range(cfg.L):
        ref = oracle_layer(cfg, l, xin)
        assert_out_close(out_bits_to_f64(out[l]), ref["out"])
        xin = omoe.residual_next(xin, out[l].cpu().numpy().view(np.uint16))
    assert_routing_equal(st, ref, T)
    assert st.prefill_bytes() == (cfg.L * cfg.E * cfg.entry_bytes, 0)
    assert st.status() == 0
    st.close()


def test_capacity_error_leaves_cache_unchanged():
    cfg = Config(L=1, E=16, k=4, d=256, d_ff=128, n_slots=3, seed=4)
    st = make_stack(cfg, max_tokens=16)
    before = st.cache_state()
    x = ft_synth.activations(4, 0, 4, cfg.d)   # 4 tokens x top-4 touch > 3 experts
    _run(st, 0, x)
    after = st.cache_state()
    for a, b in zip(before[:3], after[:3]):
        np.testing.assert_array_equal(a, b)
    assert before[3] == after[3]
    assert st.status() == 5
    st.stats_reset()
    assert st.status() == 0
    st.close()


def test_resize_matches_simulator():
    cfg = Config(L=2, E=16, k=2, d=256, d_ff=128, n_slots=8, seed=5)
    st = make_stack(cfg, max_tokens=16)
    sim = olru.SlotCacheSim(cfg.L, cfg.E, cfg.n_slots, cfg.entry_bytes, prewarm=True)
    gen = ft_synth.DriftingZipfBias(5, cfg.L, cfg.E, s=0.5, sigma_walk=0.5)
    import torch
    step = 0

    def run_steps(n):
        nonlocal step
        for _ in range(n):
            gen.advance()
            x = ft_synth.activations(5, step, 2, cfg.d)
            step += 1
            for l in range(cfg.L):
                b = gen.bias(l)
                st.set_router_bias(l, torch.from_numpy(b).cuda())
                out = _run(st, l, x)
                ref = oracle_layer(cfg, l, x, bias=b)
                sim.access(l, ref["idx"].ravel())
                assert_cache_equal(st, sim)
                assert_out_close(out_bits_to_f64(out), ref["out"])

    run_steps(6)
    for n_new in (4, 12, 5):
        st.resize(n_new)
        sim.resize(n_new)
        assert_cache_equal(st, sim)
        run_steps(4)
    assert st.stats()["resizes"] == 3
    st.close()


def test_shared_expert():
    cfg = Config(L=2, E=16, k=3, d=256, d_ff=256, n_slots=20, n_shared=1, seed=6)
    st = make_stack(cfg, max_tokens=64)
    for T in (1, 7, 33):
        x = ft_synth.activations(6, T, T, cfg.d)
        out = _run(st, 1, x)
        ref = oracle_layer(cfg, 1, x)
        assert_routing_equal(st, ref, T)
        assert_out_close(out_bits_to_f64(out), ref["out"])
    st.close()


def test_prefill_double_buffer_matches_oracle():
    """Prefill reads the double buffer only, and chains the layers through the residual
    stream: layer l+1 reads x_{l+1} = bf16(x_l + out_l).  Every layer matches the oracle on the
    GPU's own input (teacher forcing, the input rebuilt from the outputs by the oracle's
    residual step); the last layer's logits are bit-exact, so the GPU's chained input is too;
    the cache is untouched."""
    import torch
    cfg = Config(L=3, E=16, k=2, d=256, d_ff=128, n_slots=4, seed=7)
    T = 600
    st = make_stack(cfg, max_tokens=T)
    before = st.cache_state()
    x = ft_synth.activations(7, 0, T, cfg.d)
    xd = to_dev_bf16(x)
    out = torch.empty((3, T, cfg.d), dtype=torch.int16, device="cuda")
    st.prefill(0, 3, xd, out)
    torch.cuda.synchronize()
    rows = np.arange(0, T, 5)
    xin = x
    for l in range(3):
        ref = oracle_layer(cfg, l, xin, tokens=rows)
        assert_out_close(out_bits_to_f64(out[l])[rows], ref["out"])
        if l == 2:
            np.testing.assert_array_equal(st.logits(T).view(np.uint32),
                                          ref["logits"].view(np.uint32))
            assert_routing_equal(st, ref, T)  # last layer's routing
        xin = omoe.residual_next(xin, out[l].cpu().numpy().view(np.uint16))
    after = st.cache_state()
    for a, b in zip(before[:3], after[:3]):
        np.testing.assert_array_equal(a, b)
    c, k, w = st.prefill_timing()
    assert c > 0 and k > 0 and w > 0
    assert st.prefill_bytes() == (3 * cfg.E * cfg.entry_bytes, 0)
    st.close()


@pytest.mark.parametrize("T", [1, 16])
def test_prefill_short_prompts(T):
    """Prompts as short as decode batches still take the grouped-GEMM path in prefill (one
    M-tile, mostly empty rows) and chain through the residual stream."""
    import torch
    cfg = Config(L=2, E=16, k=2, d=256, d_ff=128, n_slots=4, seed=8)
    st = make_stack(cfg, max_tokens=64)
    x = ft_synth.activations(8, T, T, cfg.d)
    out = torch.empty((2, T, cfg.d), dtype=torch.int16, device="cuda")
    st.prefill(0, 2, to_dev_bf16(x), out)
    torch.cuda.synchronize()
    xin = x
    for l in range(2):
        ref = oracle_layer(cfg, l, xin)
        assert_out_close(out_bits_to_f64(out[l]), ref["out"])
        xin = omoe.residual_next(xin, out[l].cpu().numpy().view(np.uint16))
    assert_routing_equal(st, ref, T)
    assert st.status() == 0
    st.close()


def test_prefill_topup_from_cache_slots():
    """Prefill top-up: entries the decode cache holds are copied slot -> buffer, the rest from
    the host.  Decode calls first scatter layers 2-3 over arbitrary slots (state followed by
    the oracle simulator); the prefill's outputs then match the oracle on every layer, the
    cache is unchanged, and the bytes split exactly as the simulator's table says."""
    import torch
    cfg = Config(L=4, E=16, k=2, d=256, d_ff=128, n_slots=20, seed=9)
    T = 300
    st = make_stack(cfg, max_tokens=T, prefill_topup=1)
    sim = olru.SlotCacheSim(cfg.L, cfg.E, cfg.n_slots, cfg.entry_bytes, prewarm=True)
    for step in range(4):
        x = ft_synth.activations(9, 100 + step, 4, cfg.d)
        for l in (3, 2):
            _run(st, l, x)
            ref = oracle_layer(cfg, l, x, tokens=[])
            assert sim.access(l, ref["idx"].ravel())[0] == olru.OK
    assert_cache_equal(st, sim)
    before = st.cache_state()
    resident = (sim.table >= 0).sum(axis=1)
    assert resident.min() < cfg.E and resident[2:].sum() > 0   # a mix of both kinds of copy
    x = ft_synth.activations(9, 0, T, cfg.d)
    out = torch.empty((cfg.L, T, cfg.d), dtype=torch.int16, device="cuda")
    st.prefill(0, cfg.L, to_dev_bf16(x), out)
    torch.cuda.synchronize()
    rows = np.arange(1, T, 7)
    xin = x
    for l in range(cfg.L):
        ref = oracle_layer(cfg, l, xin, tokens=rows)
        assert_out_close(out_bits_to_f64(out[l])[rows], ref["out"])
        xin = omoe.residual_next(xin, out[l].cpu().numpy().view(np.uint16))
    after = st.cache_state()
    for a, b in zip(before, after):
        np.testing.assert_array_equal(a, b)
    n_res = int(resident.sum())
    assert st.prefill_bytes() == ((cfg.L * cfg.E - n_res) * cfg.entry_bytes,
                                  n_res * cfg.entry_bytes)
    st.close()


@pytest.mark.parametrize("T", [1, 4, 40])
def test_chained_layers_read_previous_output(T):
    """Layer l+1 takes layer l's output as its input, enqueued back to back with no host
    synchronisation, so each call's first kernels may start while the previous call's last
    kernel is still running.  Every layer matches the oracle applied to the GPU's own input
    (teacher forcing); the cache state after the chain matches the simulator."""
    import torch
    # 40 tokens touch nearly all 16 experts of a layer: give them room for one layer and more
    cfg = Config(L=5, E=16, k=2, d=256, d_ff=128, n_slots=10 if T <= 4 else 24, seed=11)
    st = make_stack(cfg, max_tokens=64)
    sim = olru.SlotCacheSim(cfg.L, cfg.E, cfg.n_slots, cfg.entry_bytes, prewarm=True)
    x0 = to_dev_bf16(ft_synth.activations(11, T, T, cfg.d))
    outs = [torch.empty_like(x0) for _ in range(cfg.L)]
    for rep in range(3):
        xin = x0
        for l in range(cfg.L):
            st.forward(l, xin, outs[l])
            xin = outs[l]
        torch.cuda.synchronize()
        xin_bits = x0.cpu().numpy().view(np.uint16)
        for l in range(cfg.L):
            ref = oracle_layer(cfg, l, xin_bits)
            assert sim.access(l, ref["idx"].ravel())[0] == olru.OK
            got = outs[l].cpu().numpy().view(np.uint16)
            assert_out_close(out_bits_to_f64(outs[l]), ref["out"])
            xin_bits = got
        assert_routing_equal(st, ref, T)   # the last call's routing
        assert_cache_equal(st, sim)
    assert st.stats()["status"] == 0 and sim.misses > 0
    st.close()


@pytest.mark.parametrize("E,k,T", [(32, 4, 1), (32, 4, 3), (128, 8, 4), (128, 8, 16),
                                   (512, 8, 1), (64, 6, 40)])
@pytest.mark.parametrize("pattern", ["ties_inside", "ties_across_k"])
def test_topk_exact_ties_minus_inf_and_nan_logits(E, k, T, pattern):
    """Router biases that force exact logit ties (1e30 absorbs the dot product), -inf logits
    and a NaN logit: the order (logit descending, expert id ascending), the (k+1)-th logit of
    the near-tie flag and NaN never being selected match the oracle for the ranking top-k
    (small T*E^2), the warp-argmax top-k (T = 16 at E = 128, E = 512) and the grouped path
    (T = 40)."""
    import torch
    cfg = Config(L=1, E=E, k=k, d=128, d_ff=128, n_slots=min(E, 256), seed=19)
    st = make_stack(cfg, max_tokens=64)
    bias = np.zeros(E, np.float32)
    top = [5, 9, 17, 30]                                 # 4 tied experts, all selected
    if pattern == "ties_across_k":
        top = [10 + 3 * i for i in range(k + 2)]         # k + 2 tied: the tie spans rank k
    bias[top] = 1e30
    bias[[1, 2, E - 1]] = -np.inf
    bias[7] = np.nan
    st.set_router_bias(0, torch.from_numpy(bias).cuda())
    x = ft_synth.activations(19, T, T, cfg.d)
    out = _run(st, 0, x)
    ref = oracle_layer(cfg, 0, x, bias=bias, tokens=np.arange(min(T, 3)))
    lg, rl = st.logits(T), ref["logits"]
    fin = ~np.isnan(rl)                                  # a NaN's payload is not compared
    np.testing.assert_array_equal(np.isnan(lg), ~fin)
    np.testing.assert_array_equal(lg[fin].view(np.uint32), rl[fin].view(np.uint32))
    assert_routing_equal(st, ref, T)
    assert not np.isin(7, ref["idx"]) and ref["tie"].all()
    assert_out_close(out_bits_to_f64(out)[ref["tokens"]], ref["out"])
    assert st.status() == 0
    st.close()


@pytest.mark.parametrize("E,k,T", [(32, 4, 1), (512, 8, 16), (32, 4, 40), (32, 4, 300)])
def test_non_finite_input_refuses_call(E, k, T):
    """All-NaN activations leave every logit NaN, so no expert can be ranked: the call is
    refused with FT_ERR_INVALID (in-CTA top-k, warp top-k, single- and multi-CTA grouping),
    out is not written, the cache does not change, and the next valid call is exact."""
    import torch
    from expert_cached_routed_router_b300 import FT_ERR_INVALID
    # room for the T*k distinct experts of the valid call that follows (128 at T = 16, k = 8)
    cfg = Config(L=1, E=E, k=k, d=128, d_ff=128, n_slots=160, seed=17)
    st = make_stack(cfg, max_tokens=512, pool=gpu_host_pool(cfg))
    before = st.cache_state()
    x = torch.full((T, cfg.d), 0x7FC0, dtype=torch.int16, device="cuda")   # bf16 NaN
    out = torch.zeros_like(x)
    st.forward(0, x, out)
    torch.cuda.synchronize()
    assert st.status() == FT_ERR_INVALID
    assert int(out.abs().sum()) == 0
    for a_, b_ in zip(before, st.cache_state()):
        np.testing.assert_array_equal(a_, b_)
    st.stats_reset()
    xv = ft_synth.activations(17, T, T, cfg.d)
    out = _run(st, 0, xv)
    ref = oracle_layer(cfg, 0, xv, tokens=np.arange(min(T, 4)))
    assert_routing_equal(st, ref, T)
    assert_out_close(out_bits_to_f64(out)[ref["tokens"]], ref["out"])
    assert st.status() == 0
    st.close()


def test_forward_is_deterministic():
    cfg = Config(L=1, E=32, k=4, d=512, d_ff=384, n_slots=32, seed=8)
    st = make_stack(cfg, max_tokens=16)
    x = ft_synth.activations(8, 0, 16, cfg.d)
    a = _run(st, 0, x).cpu().numpy()
    b = _run(st, 0, x).cpu().numpy()
    np.testing.assert_array_equal(a, b)
    st.close()


def test_resize_allocation_failure_leaves_cache_intact(monkeypatch):
    """An injected allocation failure during resize returns FT_ERR_OOM and changes nothing."""
    import expert_cached_routed_router_b300 as ftm
    cfg = Config(L=2, E=16, k=2, d=256, d_ff=128, n_slots=8, seed=9)
    st = make_stack(cfg, max_tokens=16)
    x = ft_synth.activations(9, 0, 3, cfg.d)
    _run(st, 0, x)
    before = st.cache_state()
    monkeypatch.setenv("FT_FAULT_INJECT", "resize_alloc")
    with pytest.raises(ftm.FtError) as ei:
        st.resize(4)
    assert ei.value.code == ftm.FT_ERR_OOM
    monkeypatch.delenv("FT_FAULT_INJECT")
    after = st.cache_state()
    for a, b in zip(before, after):
        np.testing.assert_array_equal(np.asarray(a), np.asarray(b))
    st.resize(4)          # a real resize still works afterwards
    assert st.stats()["n_slots"] == 4
    st.close()


def test_decode_step_graph_capture_matches_eager():
    """One decode step (several layers, shared cache) captured into a CUDA graph and replayed
    gives the same outputs and the same cache state as the same calls run eagerly, also across
    an elastic resize between two replays (the graph is not captured again)."""
    import torch
    cfg = Config(L=3, E=16, k=2, d=256, d_ff=128, n_slots=10, seed=10)
    gen = ft_synth.DriftingZipfBias(10, cfg.L, cfg.E, s=0.8, sigma_walk=0.3)
    steps = []
    for t in range(6):
        gen.advance()
        steps.append((ft_synth.activations(10, t, 4, cfg.d),
                      np.stack([gen.bias(l) for l in range(cfg.L)])))
    pool = None

    def run(use_graph):
        nonlocal pool
        st = make_stack(cfg, max_tokens=16, pool=pool)
        pool = st._pool
        xs = torch.empty((4, cfg.d), dtype=torch.int16, device="cuda")
        bs = torch.empty((cfg.L, cfg.E), dtype=torch.float32, device="cuda")
        out = torch.empty((cfg.L, 4, cfg.d), dtype=torch.int16, device="cuda")

        def body():
            st.set_router_bias(-1, bs)
            for l in range(cfg.L):
                st.forward(l, xs, out[l])

        g = None
        if use_graph:
            xs.copy_(to_dev_bf16(steps[0][0]))
            bs.copy_(torch.from_numpy(steps[0][1]).cuda())
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                body()
        outs = []
        for i, (x, b) in enumerate(steps):
            if i == 3:
                st.resize(7)            # safe point between steps
            xs.copy_(to_dev_bf16(x))
            bs.copy_(torch.from_numpy(b).cuda())
            if use_graph:
                g.replay()
            else:
                body()
            torch.cuda.synchronize()
            outs.append(out.cpu().numpy().copy())
        state = st.cache_state()
        stats = st.stats()
        st.close()
        return outs, state, stats

    eager, st_e, s_e = run(False)
    graph, st_g, s_g = run(True)
    for a, b in zip(eager, graph):
        np.testing.assert_array_equal(a, b)
    for a, b in zip(st_e, st_g):
        np.testing.assert_array_equal(np.asarray(a), np.asarray(b))
    assert s_e["misses"] == s_g["misses"] > 0 and s_e["hits"] == s_g["hits"]


def test_decode_wait_times_out_and_context_recovers():
    """Every cross-CTA wait of the decode expert kernel is bounded.  With a host-set flag the
    kernel copies its fills but never reports them done, so the work waiting for them runs out
    of its (shortened) wait limit: the call records FT_ERR_TIMEOUT and returns, the GPU context
    stays usable, and the next calls (flag cleared) match the oracle and its simulator."""
    import time
    import torch
    import expert_cached_routed_router_b300 as ftm
    cfg = Config(L=2, E=16, k=2, d=256, d_ff=128, n_slots=8, seed=12)
    st = make_stack(cfg, max_tokens=16)   # prewarm: layer 0's experts 0..7 in slots 0..7
    sim = olru.SlotCacheSim(cfg.L, cfg.E, cfg.n_slots, cfg.entry_bytes, prewarm=True)
    st.debug_set(ftm.FT_DEBUG_WAIT_NS, 20_000_000)
    st.debug_set(ftm.FT_DEBUG_HOLD_FILLS, 1)
    x = ft_synth.activations(12, 0, 3, cfg.d)
    t0 = time.perf_counter()
    _run(st, 1, x)                         # layer 1: every touched expert misses
    elapsed = time.perf_counter() - t0
    assert st.status() == ftm.FT_ERR_TIMEOUT
    assert elapsed < 10.0
    ref = oracle_layer(cfg, 1, x)
    assert sim.access(1, ref["idx"].ravel())[0] == olru.OK
    assert_cache_equal(st, sim)            # the control ran; only the expert work timed out
    st.debug_set(ftm.FT_DEBUG_HOLD_FILLS, 0)
    st.debug_set(ftm.FT_DEBUG_WAIT_NS, 4_000_000_000)
    st.stats_reset()
    for l, t in ((1, 3), (0, 5), (1, 4)):  # hits on the (copied) entries, then new misses
        xv = ft_synth.activations(12, 10 + t, t, cfg.d)
        out = _run(st, l, xv)
        ref = oracle_layer(cfg, l, xv)
        assert sim.access(l, ref["idx"].ravel())[0] == olru.OK
        assert_routing_equal(st, ref, t)
        assert_out_close(out_bits_to_f64(out), ref["out"])
        assert_cache_equal(st, sim)
    assert st.status() == 0
    st.close()
