"""bench.py's CPU oracle loop (its cpu_baseline and reference arm) on tiny pools of both entry
formats: it runs without a GPU, touches the layer calls in trace order, and sizes entries the
way the library does."""
import numpy as np
import torch

import bench
import ft_synth


def _pool(fp4, L, E, d, d_ff):
    if fp4:
        return torch.from_numpy(np.concatenate(
            [ft_synth.expert_entry_fp4(0, l, e, d, d_ff) for l in range(L) for e in range(E)]))
    return torch.from_numpy(np.concatenate(
        [ft_synth.expert_entry(0, l, e, d, d_ff) for l in range(L) for e in range(E)]).view(np.int16))


def test_oracle_decode_loop_both_formats():
    L, E, d, d_ff = 2, 8, 128, 128
    gen = ft_synth.DriftingZipfBias(0, L, E, s=1.1)
    bias = np.empty((4, L, E), np.float32)
    for t in range(4):
        gen.advance()
        for l in range(L):
            bias[t, l] = gen.bias(l)
    for fp4 in (False, True):
        wl = dict(L=L, E=E, k=2, d=d, d_ff=d_ff, n_slots=6, zipf=1.1, shared=0)
        if fp4:
            wl["fp4"] = 1
        pool = _pool(fp4, L, E, d, d_ff)
        assert pool.numel() * pool.element_size() == L * E * bench.entry_bytes(wl)
        calls, el = bench.cpu_oracle_decode(wl, pool, 1, bias, 0, max_calls=5)
        assert calls == 5 and el > 0
