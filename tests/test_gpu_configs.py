"""Parity at the full sizes of the decode, large-expert, prefill and elastic configurations (GPU).

The CUDA path runs in the launch configuration bench.py times (same pools, same graph-free
per-layer calls); routing, the grouping by expert and the whole LRU cache state are compared
bit-exactly with the oracle on every call; outputs are compared within
max|gpu-ref| <= 1e-2 max|ref| + 1e-3 on sampled calls and tokens (the oracle computes them
one by one in fp64).  Step counts are cut from the configurations' 2,000 / 10,000 steps to
keep the suite within minutes; bench.py runs the long traces.
"""
import numpy as np
import pytest

import ft_synth
from oracle import lru as olru
from oracle import moe as omoe

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _gpu_pool(seed, L, E, d, d_ff):
    import torch
    import ft_synth.gpu as sg
    sg.build()
    n = L * E * 3 * d * d_ff
    pool = torch.empty(n, dtype=torch.int16, pin_memory=True)
    sg.fill_pool(pool.data_ptr(), seed, L, E, d, d_ff)
    return pool


def _stack(pool, seed, L, E, k, d, d_ff, n_slots, max_tokens, shared=0, admission=0):
    import torch
    from expert_cached_routed_router_b300 import MoELayerStack
    st = MoELayerStack(L, E, k, d, d_ff, n_slots, n_shared=shared, max_tokens=max_tokens,
                       admission=admission)
    for l in range(L):
        st.load_router(l, torch.from_numpy(ft_synth.router_weight(seed, l, E, d).view(np.int16)).cuda())
        if shared:
            st.load_shared(l, torch.from_numpy(ft_synth.shared_entry(seed, l, d, d_ff).view(np.int16)).cuda())
    st.load_pool(pool, pool.numel() * 2)
    torch.cuda.synchronize()
    return st


def _entry_view(pool, L, E, d, d_ff):
    pv = pool.numpy().view(np.uint16)
    ent = 3 * d * d_ff
    return lambda l, e: pv[(l * E + e) * ent:(l * E + e + 1) * ent]


def _decode_trace_parity(seed, L, E, k, d, d_ff, n_slots, zipf, b, n_steps, out_every, shared=0,
                         phase_len=0, resizes=(), pool=None, batch_of=None, out_tokens=4,
                         admission=0):
    """Run a decode trace; compare every call bit-exactly, sampled outputs within tolerance."""
    import torch
    pool = _gpu_pool(seed, L, E, d, d_ff) if pool is None else pool
    st = _stack(pool, seed, L, E, k, d, d_ff, n_slots, max_tokens=16, shared=shared,
                admission=admission)
    entry = _entry_view(pool, L, E, d, d_ff)
    sim = olru.SlotCacheSim(L, E, n_slots, 6 * d * d_ff, prewarm=True,
                            admission=bool(admission))
    gen = ft_synth.DriftingZipfBias(seed, L, E, s=zipf, phase_len=phase_len)
    routers = [ft_synth.router_weight(seed, l, E, d) for l in range(L)]
    w_stack = np.concatenate(routers, axis=0)     # every layer's experts, one oracle call
    shared_e = [ft_synth.shared_entry(seed, l, d, d_ff) for l in range(L)] if shared else None
    resizes = dict(resizes)
    checked_out = 0
    for step in range(n_steps):
        if step in resizes:
            st.resize(resizes[step])
            sim.resize(resizes[step])
            tb, ow, stp, tk = st.cache_state()
            np.testing.assert_array_equal(tb, sim.table)
            np.testing.assert_array_equal(ow, sim.owner)
            np.testing.assert_array_equal(stp.astype(np.int64), sim.stamp)
        gen.advance()
        bb = batch_of(step) if batch_of else b
        x = ft_synth.activations(seed, 1_000_000 * bb + step, bb, d)
        xd = torch.from_numpy(x.view(np.int16)).cuda()
        bias = torch.from_numpy(np.stack([gen.bias(l) for l in range(L)])).cuda()
        st.set_router_bias(-1, bias)
        # the oracle's logits of all layers at once (each logit is its own fixed-order sum)
        logits_all = omoe.router_logits(x, w_stack)
        for l in range(L):
            out = torch.empty_like(xd)
            st.forward(l, xd, out)
            torch.cuda.synchronize()
            want_out = (step % out_every == 0) and l in (0, L - 1)
            if want_out:
                ref = omoe.moe_layer(x, routers[l], k, lambda e: entry(l, e), d, d_ff,
                                     bias=gen.bias(l),
                                     shared_entry=shared_e[l] if shared else None,
                                     tokens=np.arange(min(bb, out_tokens)))
            else:
                lg = (logits_all[:, l * E:(l + 1) * E] + gen.bias(l)[None, :]).astype(np.float32)
                ridx, rtie = omoe.topk(lg, k)
                rw = omoe.gates(lg, ridx)
                _, roff, rperm, _ = omoe.permutation(ridx, E)
                ref = dict(idx=ridx, w=rw, offsets=roff, perm=rperm)
            idx, w, tie = st.routing(bb)
            np.testing.assert_array_equal(idx, ref["idx"])
            np.testing.assert_allclose(w, ref["w"], rtol=2e-6, atol=1e-7)
            counts, offsets, perm = st.perm(bb)
            np.testing.assert_array_equal(perm, ref["perm"])
            np.testing.assert_array_equal(offsets, ref["offsets"])
            code, hits, fills = sim.access(l, ref["idx"].ravel())
            assert code == olru.OK
            np.testing.assert_array_equal(st.fills(), np.array([f[:3] for f in fills],
                                                              np.int32).reshape(-1, 3))
            tb, ow, stp, tk = st.cache_state()
            np.testing.assert_array_equal(tb, sim.table)
            np.testing.assert_array_equal(ow, sim.owner)
            np.testing.assert_array_equal(stp.astype(np.int64), sim.stamp)
            assert tk == sim.tick
            if want_out:
                got = omoe.bf16_to_f64(out.cpu().numpy().view(np.uint16))[ref["tokens"]]
                ok, err, bound = omoe.within_tolerance(got, ref["out"])
                assert ok, (step, l, err, bound)
                checked_out += 1
    s = st.stats()
    assert s["hits"] == sim.hits and s["misses"] == sim.misses and s["status"] == 0
    assert s["evictions"] == sim.evictions and s["bypasses"] == sim.bypasses
    st.close()
    return sim, checked_out


def test_decode_trace_24_layers():
    """24 layers, d=2048, d_ff=768, E=128 top-8, Zipf(1.1) + drift, 768 slots (25%), b=4."""
    sim, n_out = _decode_trace_parity(0, 24, 128, 8, 2048, 768, 768, 1.1, b=4, n_steps=60,
                                      out_every=20)
    assert sim.misses > 0 and sim.evictions > 0 and n_out == 6


def test_decode_trace_24_layers_admission():
    """The same 24-layer trace with frequency admission: bypassed misses are staged past the
    768 slots; fills, cache state and counters bit-exact, outputs within tolerance."""
    sim, n_out = _decode_trace_parity(0, 24, 128, 8, 2048, 768, 768, 1.1, b=4, n_steps=60,
                                      out_every=20, admission=1)
    assert sim.bypasses > 0 and n_out == 6


def test_elastic_resize_trace():
    """24-layer shapes; b alternating 1 and 8; popularity switching between two disjoint Zipf
    orders every 100 steps; resizes 768 -> 307 -> 1228 at fixed safe points."""
    _decode_trace_parity(0, 24, 128, 8, 2048, 768, 768, 1.1, b=1, n_steps=400, out_every=100,
                         phase_len=100, resizes={120: 307, 260: 1228},
                         batch_of=lambda s: 1 if (s // 50) % 2 == 0 else 8)


@pytest.fixture(scope="module")
def large_pool():
    pool = _gpu_pool(0, 8, 256, 4096, 2048)
    yield pool
    del pool


def test_large_expert_decode(large_pool):
    """8 layers, d=4096, d_ff=2048, E=256 top-6 + shared expert, 640 slots (30 GiB)."""
    for b in (1, 16):
        _decode_trace_parity(0, 8, 256, 6, 4096, 2048, 640, 1.0, b=b, n_steps=12, out_every=6,
                             shared=1, pool=large_pool, out_tokens=2)


@pytest.mark.parametrize("T", [4096, 16384])
def test_prefill_streaming(large_pool, T):
    """8 layers streamed through the double buffer; routing bit-exact on sampled tokens of
    every layer (one layer per call), outputs within tolerance on sampled tokens."""
    import torch
    import ft_synth.gpu as sg
    L, E, k, d, d_ff = 8, 256, 6, 4096, 2048
    st = _stack(large_pool, 0, L, E, k, d, d_ff, n_slots=16, max_tokens=T)
    x = torch.empty((T, d), dtype=torch.int16, device="cuda")
    sg.activations_device(x.data_ptr(), 0, [7_000_000 + T], T, d,
                          torch.cuda.current_stream().cuda_stream)
    x_np = x.cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(x_np, ft_synth.activations(0, 7_000_000 + T, T, d))
    out = torch.empty((L, T, d), dtype=torch.int16, device="cuda")
    st.prefill(0, L, x, out)                      # all layers, double-buffered
    torch.cuda.synchronize()
    entry = _entry_view(large_pool, L, E, d, d_ff)
    rng = np.random.default_rng(T)
    sample = np.sort(rng.choice(T, size=256, replace=False))
    for l in range(L):
        wr = ft_synth.router_weight(0, l, E, d)
        one = torch.empty((1, T, d), dtype=torch.int16, device="cuda")
        st.prefill(l, 1, x, one)                  # routing of layer l stays readable
        torch.cuda.synchronize()
        # the prefill combine adds fp32 partial sums atomically, so runs agree to rounding only
        a1 = omoe.bf16_to_f64(one[0].cpu().numpy().view(np.uint16))
        a8 = omoe.bf16_to_f64(out[l].cpu().numpy().view(np.uint16))
        assert omoe.within_tolerance(a1, a8)[0]
        idx, w, tie = st.routing(T)
        lg = omoe.router_logits(x_np[sample], wr)
        ridx, rtie = omoe.topk(lg, k)
        np.testing.assert_array_equal(idx[sample], ridx)
        if l in (0, L - 1):
            toks = sample[:3]
            ref = omoe.moe_layer(x_np[toks], wr, k, lambda e: entry(l, e), d, d_ff)
            got = omoe.bf16_to_f64(out[l].cpu().numpy().view(np.uint16))[toks]
            ok, err, bound = omoe.within_tolerance(got, ref["out"])
            assert ok, (l, err, bound)
    c, kk, wall = st.prefill_timing()
    assert c > 0 and kk > 0 and wall > 0
    st.close()
