"""The allocation-free routing entry point against the regular forward path (GPU).

ft_route_topk_noalloc serves callers that cannot allocate device memory (open global-mode
stream captures, allocation-free serving loops, hosts whose framework owns all device
memory): the caller passes inputs and outputs, and the logits scratch is a fixed device
array inside the library.  This file is collected last so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import ft_synth

from helpers import Config, make_stack, to_dev_bf16

pytestmark = pytest.mark.gpu


def _noalloc(x, wr, bias, T, E, d, k):
    import torch
    import expert_cached_routed_router_b300 as ftm
    idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    tie = torch.zeros(T, dtype=torch.uint8, device="cuda")
    ftm.ft_route_topk_noalloc(x, wr, bias, T, E, d, k, idx, w, tie)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy(), tie.cpu().numpy()


def test_noalloc_routing_matches_forward_twice_in_a_row():
    import torch
    cfg = Config(L=1, E=32, k=4, d=512, d_ff=384, n_slots=32, seed=21)
    st = make_stack(cfg, max_tokens=64)
    wr = to_dev_bf16(cfg.router(0))
    bias_np = (0.3 * ft_synth.normal_f32(ft_synth.stream_key(21, 99), cfg.E)).astype(np.float32)
    bias = torch.from_numpy(bias_np).cuda()
    st.set_router_bias(0, bias)
    for call, T in enumerate((16, 64)):      # two calls in a row, different sizes
        x = to_dev_bf16(ft_synth.activations(21, call, T, cfg.d))
        out = torch.empty_like(x)
        st.forward(0, x, out)
        torch.cuda.synchronize()
        ref_idx, ref_w, ref_tie = st.routing(T)
        idx, w, tie = _noalloc(x, wr, bias, T, cfg.E, cfg.d, cfg.k)
        np.testing.assert_array_equal(idx, ref_idx)
        np.testing.assert_allclose(w, ref_w, rtol=2e-6, atol=1e-7)
        np.testing.assert_array_equal(tie, ref_tie)
    st.close()


def test_noalloc_rejects_sizes_beyond_the_scratch():
    import torch
    import expert_cached_routed_router_b300 as ftm
    E, d, k = 1024, 64, 2
    T = (1 << 18) // E + 1
    x = torch.zeros((T, d), dtype=torch.int16, device="cuda")
    wr = torch.zeros((E, d), dtype=torch.int16, device="cuda")
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    tie = torch.zeros(T, dtype=torch.uint8, device="cuda")
    with pytest.raises(ftm.FtError) as ei:
        ftm.ft_route_topk_noalloc(x, wr, None, T, E, d, k, idx, w, tie)
    assert ei.value.code == ftm.FT_ERR_INVALID
    assert "262144" in str(ei.value)
