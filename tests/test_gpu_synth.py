"""The GPU input generator reproduces the host generator bit for bit (GPU)."""
import numpy as np
import pytest

import ft_synth

pytestmark = pytest.mark.gpu


def test_gpu_pool_matches_host_generator():
    import torch
    import ft_synth.gpu as sg
    sg.build()
    L, E, d, d_ff = 2, 5, 256, 128
    n = L * E * 3 * d * d_ff
    pool = torch.empty(n, dtype=torch.int16, pin_memory=True)
    sg.fill_pool(pool.data_ptr(), 11, L, E, d, d_ff, stage_entries=3)
    pv = pool.numpy().view(np.uint16)
    ent = 3 * d * d_ff
    for l in range(L):
        for e in range(E):
            want = ft_synth.expert_entry(11, l, e, d, d_ff)
            np.testing.assert_array_equal(pv[(l * E + e) * ent:(l * E + e + 1) * ent], want)


def test_gpu_activations_match_host_generator():
    import torch
    import ft_synth.gpu as sg
    sg.build()
    T, d = 3, 512
    x = torch.empty((4, T, d), dtype=torch.int16, device="cuda")
    sg.activations_device(x.data_ptr(), 5, [10, 11, 12, 99], T, d,
                          torch.cuda.current_stream().cuda_stream)
    got = x.cpu().numpy().view(np.uint16)
    for i, s in enumerate([10, 11, 12, 99]):
        np.testing.assert_array_equal(got[i], ft_synth.activations(5, s, T, d))


def test_gpu_fp4_pool_matches_host_generator():
    import torch
    import ft_synth.gpu as sg
    sg.build()
    L, E, d, d_ff = 2, 5, 256, 128
    eb = ft_synth.entry_bytes_fp4(d, d_ff)
    pool = torch.empty(L * E * eb, dtype=torch.uint8, pin_memory=True)
    sg.fill_pool_fp4(pool.data_ptr(), 11, L, E, d, d_ff, stage_entries=3)
    pv = pool.numpy()
    for l in range(L):
        for e in range(E):
            want = ft_synth.expert_entry_fp4(11, l, e, d, d_ff)
            np.testing.assert_array_equal(pv[(l * E + e) * eb:(l * E + e + 1) * eb], want)
