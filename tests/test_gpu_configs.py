"""Parity at the full sizes and full lengths of the decode, large-expert, prefill and elastic
configurations (GPU).

The CUDA path runs in the launch configuration bench.py times (same pools, per-layer forward
calls).  Long traces run their stated lengths: the 24-layer decode trace 2,000 steps, the
large-expert trace 2,000 steps and the elastic trace 10,000 steps with its 1,000-step
popularity phases, b = 1 / 8 halves and resizes before steps 3,500 and 6,500.  On every call
the fill list and the whole cache state (slot table, owners, stamps, tick) are compared with
the oracle's simulator, fed with the routing the GPU reports; that routing is itself compared
bit-exactly with the oracle's (logits in the fixed fp32 order, top-k, gates, grouping) on
sampled steps, and outputs within max|gpu-ref| <= 1e-2 max|ref| + 1e-3 on sampled calls and
tokens (the oracle computes them one by one in fp64).
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


def _long_trace_parity(seed, L, E, k, d, d_ff, n_slots, zipf, n_steps, batch_of,
                       route_every, out_every, out_tokens=2, shared=0, phase_len=0,
                       resizes=(), pool=None):
    """A decode trace at its stated length.

    Every call: the GPU's routing feeds the oracle's simulator, whose fill list, slot table,
    owners, stamps and tick must equal the GPU's.  Every ``route_every`` steps: the routing of
    all layers equals the oracle's (fixed-order fp32 logits, top-k, gates, grouping).  Every
    ``out_every`` steps: the outputs of layers 0 and L-1 on the first tokens are within the
    output tolerance.  Returns the simulator and the per-phase hit counts."""
    import torch
    pool = _gpu_pool(seed, L, E, d, d_ff) if pool is None else pool
    st = _stack(pool, seed, L, E, k, d, d_ff, n_slots, max_tokens=16, shared=shared)
    entry = _entry_view(pool, L, E, d, d_ff)
    sim = olru.SlotCacheSim(L, E, n_slots, 6 * d * d_ff, prewarm=True)
    gen = ft_synth.DriftingZipfBias(seed, L, E, s=zipf, phase_len=phase_len)
    routers = [ft_synth.router_weight(seed, l, E, d) for l in range(L)]
    w_stack = np.concatenate(routers, axis=0)
    shared_e = [ft_synth.shared_entry(seed, l, d, d_ff) for l in range(L)] if shared else None
    resizes = dict(resizes)
    outs = {b: torch.empty((b, d), dtype=torch.int16, device="cuda") for b in set(
        batch_of(s) for s in range(n_steps))}
    n_route = n_out = 0
    for step in range(n_steps):
        if step in resizes:
            st.resize(resizes[step])
            sim.resize(resizes[step])
            tb, ow, stp, tk = st.cache_state()
            np.testing.assert_array_equal(tb, sim.table)
            np.testing.assert_array_equal(ow, sim.owner)
            np.testing.assert_array_equal(stp.astype(np.int64), sim.stamp)
            assert tk == sim.tick
        gen.advance()
        b = batch_of(step)
        x = ft_synth.activations(seed, 1_000_000 * b + step, b, d)
        xd = torch.from_numpy(x.view(np.int16)).cuda()
        biases = np.stack([gen.bias(l) for l in range(L)])
        st.set_router_bias(-1, torch.from_numpy(biases).cuda())
        check_route = step % route_every == route_every - 1
        check_out = step % out_every == out_every - 1
        if check_route:
            logits_all = omoe.router_logits(x, w_stack)
        for l in range(L):
            out = outs[b]
            st.forward(l, xd, out)
            torch.cuda.synchronize()
            idx, w, tie = st.routing(b)
            if check_route:
                lg = (logits_all[:, l * E:(l + 1) * E] + biases[l][None, :]).astype(np.float32)
                ridx, rtie = omoe.topk(lg, k)
                np.testing.assert_array_equal(idx, ridx, err_msg=f"step {step} layer {l}")
                np.testing.assert_allclose(w, omoe.gates(lg, ridx), rtol=2e-6, atol=1e-7)
                np.testing.assert_array_equal(tie.astype(bool), rtie)
                _, roff, rperm, _ = omoe.permutation(ridx, E)
                _, offsets, perm = st.perm(b)
                np.testing.assert_array_equal(offsets, roff)
                np.testing.assert_array_equal(perm, rperm)
                n_route += 1
            code, hits, fills = sim.access(l, idx.ravel())
            assert code == olru.OK
            np.testing.assert_array_equal(
                st.fills(), np.array([f[:3] for f in fills], np.int32).reshape(-1, 3),
                err_msg=f"fills, step {step} layer {l}")
            tb, ow, stp, tk = st.cache_state()
            np.testing.assert_array_equal(tb, sim.table, err_msg=f"table, step {step} layer {l}")
            np.testing.assert_array_equal(ow, sim.owner)
            np.testing.assert_array_equal(stp.astype(np.int64), sim.stamp)
            assert tk == sim.tick
            if check_out and l in (0, L - 1):
                toks = np.arange(min(b, out_tokens))
                ref = omoe.moe_layer(x, routers[l], k, lambda e: entry(l, e), d, d_ff,
                                     bias=biases[l], tokens=toks,
                                     shared_entry=shared_e[l] if shared else None)
                np.testing.assert_array_equal(idx, ref["idx"])
                got = omoe.bf16_to_f64(out.cpu().numpy().view(np.uint16))[toks]
                ok, err, bound = omoe.within_tolerance(got, ref["out"])
                assert ok, (step, l, err, bound)
                n_out += 1
    s = st.stats()
    assert s["hits"] == sim.hits and s["misses"] == sim.misses and s["status"] == 0
    assert s["evictions"] == sim.evictions and s["tick"] == sim.tick
    st.close()
    return sim, n_route, n_out


def test_decode_trace_24_layers_2000_steps():
    """24 layers, d=2048, d_ff=768, E=128 top-8, Zipf(1.1) + drift, 768 slots (25%), b=4, the
    configuration's 2,000 steps (48,000 calls): LRU state bit-exact after every call."""
    sim, n_route, n_out = _long_trace_parity(0, 24, 128, 8, 2048, 768, 768, 1.1, n_steps=2000,
                                             batch_of=lambda s: 4, route_every=20,
                                             out_every=250)
    assert sim.misses > 0 and sim.evictions > 0
    assert n_route == 100 * 24 and n_out == 16
    assert sim.tick > 100_000   # stamps far past the 768 slots' first wrap of the LRU order


def test_decode_trace_24_layers_admission():
    """The same 24-layer trace with frequency admission: bypassed misses are staged past the
    768 slots; fills, cache state and counters bit-exact, outputs within tolerance."""
    sim, n_out = _decode_trace_parity(0, 24, 128, 8, 2048, 768, 768, 1.1, b=4, n_steps=60,
                                      out_every=20, admission=1)
    assert sim.bypasses > 0 and n_out == 6


def test_elastic_resize_trace_10000_steps():
    """The elastic-cache stress configuration at its stated length: 24-layer shapes, 10,000
    steps, b = 1 in the first half and b = 8 in the second half of every block of 1,000
    steps, the popularity order switching between two disjoint Zipf orders every 1,000 steps,
    resizes 768 -> 307 before step 3,500 and 307 -> 1,228 before step 6,500.  The whole LRU
    state is compared with the simulator after both resizes and after every call."""
    sim, n_route, n_out = _long_trace_parity(
        0, 24, 128, 8, 2048, 768, 768, 1.1, n_steps=10_000,
        batch_of=lambda s: 1 if (s % 1000) < 500 else 8, route_every=50, out_every=1000,
        phase_len=1000, resizes={3500: 307, 6500: 1228})
    assert sim.resizes == 2 and sim.n_slots == 1228
    assert n_route == 200 * 24 and n_out == 20


@pytest.fixture(scope="module")
def large_pool():
    pool = _gpu_pool(0, 8, 256, 4096, 2048)
    yield pool
    del pool


def test_large_expert_decode_2000_steps(large_pool):
    """8 layers, d=4096, d_ff=2048, E=256 top-6 + shared expert, 640 slots (30 GiB), b=4, the
    configuration's 2,000 steps (16,000 calls): LRU state bit-exact after every call."""
    sim, n_route, n_out = _long_trace_parity(0, 8, 256, 6, 4096, 2048, 640, 1.0, n_steps=2000,
                                             batch_of=lambda s: 4, route_every=50,
                                             out_every=500, shared=1, pool=large_pool)
    assert sim.misses > 0 and sim.evictions > 0
    assert n_route == 40 * 8 and n_out == 8


def test_large_expert_decode_b1_b16(large_pool):
    """The large-expert shapes at b = 1 and 16 (shorter traces)."""
    for b in (1, 16):
        _decode_trace_parity(0, 8, 256, 6, 4096, 2048, 640, 1.0, b=b, n_steps=12, out_every=6,
                             shared=1, pool=large_pool, out_tokens=2)


@pytest.mark.parametrize("T", [4096, 16384])
def test_prefill_streaming(large_pool, T):
    """8 layers streamed through the double buffer and chained by the residual stream; every
    layer is rerun alone on its input rebuilt from the outputs (teacher forcing): routing
    bit-exact on sampled tokens of every layer, outputs within tolerance on tokens spread
    over the prompt (the last ones sit in their groups' last M-tiles)."""
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
    xl_np = x_np
    for l in range(L):
        # layer l's input on the residual stream, rebuilt from the outputs (teacher forcing)
        if l > 0:
            xl_np = omoe.residual_next(xl_np, out[l - 1].cpu().numpy().view(np.uint16))
        xl = torch.from_numpy(xl_np.view(np.int16)).cuda()
        wr = ft_synth.router_weight(0, l, E, d)
        one = torch.empty((1, T, d), dtype=torch.int16, device="cuda")
        st.prefill(l, 1, xl, one)                 # routing of layer l stays readable
        torch.cuda.synchronize()
        # the prefill combine adds fp32 partial sums atomically, so runs agree to rounding only
        a1 = omoe.bf16_to_f64(one[0].cpu().numpy().view(np.uint16))
        a8 = omoe.bf16_to_f64(out[l].cpu().numpy().view(np.uint16))
        assert omoe.within_tolerance(a1, a8)[0]
        idx, w, tie = st.routing(T)
        lg = omoe.router_logits(xl_np[sample], wr)
        ridx, rtie = omoe.topk(lg, k)
        np.testing.assert_array_equal(idx[sample], ridx)
        if l in (0, L - 1):
            # tokens spread over the whole prompt: inside each expert's group rows are ordered
            # by token, so the largest ids sit in the groups' last (ragged) M-tiles
            toks = np.unique(np.concatenate([sample[:2], sample[len(sample) // 2:][:1],
                                             sample[-2:], [T - 1]]))
            ref = omoe.moe_layer(xl_np[toks], wr, k, lambda e: entry(l, e), d, d_ff)
            np.testing.assert_array_equal(idx[toks], ref["idx"])
            got = omoe.bf16_to_f64(out[l].cpu().numpy().view(np.uint16))[toks]
            ok, err, bound = omoe.within_tolerance(got, ref["out"])
            assert ok, (l, err, bound)
            # row rank of (T-1, its experts) inside their groups: past the first M-tile
            rank = [(idx[:T - 1] == e).sum() for e in idx[T - 1]]
            if T >= 16384:
                assert min(rank) >= 256      # the third M-tile of every one of its groups
    c, kk, wall = st.prefill_timing()
    assert c > 0 and kk > 0 and wall > 0
    st.close()
