"""Test helpers: seeded configurations, host pools, and oracle runs for the parity tests."""
from __future__ import annotations

import numpy as np

import ft_synth
from oracle import lru as olru
from oracle import moe as omoe


class Config:
    def __init__(self, L, E, k, d, d_ff, n_slots, n_shared=0, seed=0, fp4=False):
        self.L, self.E, self.k, self.d, self.d_ff = L, E, k, d, d_ff
        self.n_slots, self.n_shared, self.seed, self.fp4 = n_slots, n_shared, seed, fp4
        self.entry_elems = 3 * d * d_ff
        self.entry_bytes = (ft_synth.entry_bytes_fp4(d, d_ff) if fp4 else 2 * self.entry_elems)
        self._entries = {}

    def entry(self, l, e):
        """bf16 bits (uint16), or the packed 4-bit entry (uint8) with fp4."""
        key = (l, e)
        if key not in self._entries:
            gen = ft_synth.expert_entry_fp4 if self.fp4 else ft_synth.expert_entry
            self._entries[key] = gen(self.seed, l, e, self.d, self.d_ff)
        return self._entries[key]

    def shared(self, l):
        return ft_synth.shared_entry(self.seed, l, self.d, self.d_ff)

    def router(self, l):
        return ft_synth.router_weight(self.seed, l, self.E, self.d)


def host_pool(cfg: Config):
    """Pinned torch tensor [L*E*entry] built from the generator (int16 for bf16 entries,
    uint8 for 4-bit ones)."""
    import torch
    if cfg.fp4:
        pool = torch.empty(cfg.L * cfg.E * cfg.entry_bytes, dtype=torch.uint8, pin_memory=True)
        view, n = pool.numpy(), cfg.entry_bytes
    else:
        pool = torch.empty(cfg.L * cfg.E * cfg.entry_elems, dtype=torch.int16, pin_memory=True)
        view, n = pool.numpy().view(np.uint16), cfg.entry_elems
    for l in range(cfg.L):
        for e in range(cfg.E):
            o = (l * cfg.E + e) * n
            view[o:o + n] = cfg.entry(l, e)
    return pool


def gpu_host_pool(cfg: Config):
    """The same pool as host_pool, written by the GPU generator (for large L*E)."""
    import torch
    import ft_synth.gpu as sg
    sg.build()
    if cfg.fp4:
        pool = torch.empty(cfg.L * cfg.E * cfg.entry_bytes, dtype=torch.uint8, pin_memory=True)
        sg.fill_pool_fp4(pool.data_ptr(), cfg.seed, cfg.L, cfg.E, cfg.d, cfg.d_ff)
    else:
        pool = torch.empty(cfg.L * cfg.E * cfg.entry_elems, dtype=torch.int16, pin_memory=True)
        sg.fill_pool(pool.data_ptr(), cfg.seed, cfg.L, cfg.E, cfg.d, cfg.d_ff)
    return pool


def to_dev_bf16(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def make_stack(cfg: Config, max_tokens=512, prewarm=1, pool=None, **opts):
    """A MoELayerStack with routers, pool (and shared experts) loaded; `opts` go to create."""
    import torch
    from expert_cached_routed_router_b300 import MoELayerStack
    st = MoELayerStack(cfg.L, cfg.E, cfg.k, cfg.d, cfg.d_ff, cfg.n_slots, n_shared=cfg.n_shared,
                       prewarm=prewarm, max_tokens=max_tokens, weight_format=1 if cfg.fp4 else 0,
                       **opts)
    for l in range(cfg.L):
        st.load_router(l, to_dev_bf16(cfg.router(l)))
        if cfg.n_shared:
            st.load_shared(l, to_dev_bf16(cfg.shared(l)))
    pool = host_pool(cfg) if pool is None else pool
    st.load_pool(pool, pool.numel() * pool.element_size())
    torch.cuda.synchronize()
    st._pool = pool     # keep alive
    return st


def oracle_layer(cfg: Config, l, x_bits, bias=None, tokens=None):
    from oracle import fp4 as ofp4
    return omoe.moe_layer(x_bits, cfg.router(l), cfg.k, lambda e: cfg.entry(l, e), cfg.d,
                          cfg.d_ff, bias=bias,
                          shared_entry=cfg.shared(l) if cfg.n_shared else None, tokens=tokens,
                          ffn=ofp4.expert_ffn_fp4 if cfg.fp4 else None)


def out_bits_to_f64(t):
    """Device bf16 (int16) tensor -> float64 numpy."""
    return omoe.bf16_to_f64(t.cpu().numpy().view(np.uint16))


def assert_routing_equal(st, ref, T):
    idx, w, tie = st.routing(T)
    np.testing.assert_array_equal(idx, ref["idx"])
    np.testing.assert_allclose(w, ref["w"], rtol=2e-6, atol=1e-7)
    np.testing.assert_array_equal(tie.astype(bool), ref["tie"])
    counts, offsets, perm = st.perm(T)
    np.testing.assert_array_equal(counts, ref["counts"])
    np.testing.assert_array_equal(offsets, ref["offsets"])
    np.testing.assert_array_equal(perm, ref["perm"])


def assert_cache_equal(st, sim: olru.SlotCacheSim):
    table, owner, stamps, tick = st.cache_state()
    np.testing.assert_array_equal(table, sim.table)
    np.testing.assert_array_equal(owner, sim.owner)
    np.testing.assert_array_equal(stamps.astype(np.int64), sim.stamp)
    assert tick == sim.tick


def assert_out_close(got_f64, ref_f64):
    ok, err, bound = omoe.within_tolerance(got_f64, ref_f64)
    assert ok, f"max err {err:.3e} > bound {bound:.3e}"
    return err, bound
