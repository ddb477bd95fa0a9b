"""The allocation-free routing entry point against the oracle (GPU).

ft_route_topk_noalloc serves callers that cannot allocate device memory (open global-mode
stream captures, allocation-free serving loops, hosts whose framework owns all device
memory): the caller passes inputs and outputs, and the logits scratch is a fixed device
array inside the library.  Its routing is compared with the oracle's (logits in the fixed
fp32 order, top-k by logit then expert id, gates, near-tie flags) and with the regular
forward path's.  This file is collected last so that a run stopping at the first failure
has already run every other test.
"""
import numpy as np
import pytest

import ft_synth
from oracle import moe as omoe

from helpers import Config, make_stack, to_dev_bf16

pytestmark = pytest.mark.gpu


def _outputs(T, k):
    import torch
    idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    tie = torch.full((T,), 7, dtype=torch.uint8, device="cuda")
    return idx, w, tie


def _noalloc(x, wr, bias, T, E, d, k):
    import torch
    import expert_cached_routed_router_b300 as ftm
    idx, w, tie = _outputs(T, k)
    ftm.ft_route_topk_noalloc(x, wr, bias, T, E, d, k, idx, w, tie)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy(), tie.cpu().numpy()


def _oracle(x_bits, wr_bits, bias, k):
    lg = omoe.router_logits(x_bits, wr_bits, bias)
    idx, tie = omoe.topk(lg, k)
    return idx, omoe.gates(lg, idx), tie


def _assert_matches(got, ref):
    np.testing.assert_array_equal(got[0], ref[0])
    np.testing.assert_allclose(got[1], ref[1], rtol=2e-6, atol=1e-7)
    np.testing.assert_array_equal(got[2].astype(bool), ref[2])


@pytest.mark.parametrize("E,k,T,d,with_bias", [
    (32, 4, 16, 512, True),
    (32, 4, 64, 512, False),      # no bias
    (200, 5, 3, 256, True),       # E not a multiple of 4 or 32
    (1024, 8, 256, 64, False),    # T * E = 262,144: exactly the scratch size
    (1024, 32, 2, 128, True),     # largest E and k
])
def test_noalloc_routing_matches_oracle(E, k, T, d, with_bias):
    import torch
    seed = 41 + E + T
    x = ft_synth.activations(seed, 0, T, d)
    wr = ft_synth.router_weight(seed, 0, E, d)
    bias = (0.3 * ft_synth.normal_f32(ft_synth.stream_key(seed, 99), E)).astype(np.float32) \
        if with_bias else None
    got = _noalloc(to_dev_bf16(x), to_dev_bf16(wr),
                   torch.from_numpy(bias).cuda() if with_bias else None, T, E, d, k)
    _assert_matches(got, _oracle(x, wr, bias, k))


def test_noalloc_routing_matches_forward_twice_in_a_row():
    """Two calls in a row (the scratch keeps the first call's logits) of different sizes,
    against the oracle and against the routing ft_moe_forward reports."""
    import torch
    cfg = Config(L=1, E=32, k=4, d=512, d_ff=384, n_slots=32, seed=21)
    st = make_stack(cfg, max_tokens=64)
    wr_np = cfg.router(0)
    wr = to_dev_bf16(wr_np)
    bias_np = (0.3 * ft_synth.normal_f32(ft_synth.stream_key(21, 99), cfg.E)).astype(np.float32)
    bias = torch.from_numpy(bias_np).cuda()
    st.set_router_bias(0, bias)
    for call, T in enumerate((64, 16)):
        x_np = ft_synth.activations(21, call, T, cfg.d)
        x = to_dev_bf16(x_np)
        out = torch.empty_like(x)
        st.forward(0, x, out)
        torch.cuda.synchronize()
        got = _noalloc(x, wr, bias, T, cfg.E, cfg.d, cfg.k)
        _assert_matches(got, _oracle(x_np, wr_np, bias_np, cfg.k))
        ref_idx, ref_w, ref_tie = st.routing(T)
        np.testing.assert_array_equal(got[0], ref_idx)
        np.testing.assert_array_equal(got[2], ref_tie)
    st.close()


def test_noalloc_inside_a_global_stream_capture():
    """The call that exists for open captures: after one eager call, capture it with the
    global capture mode (which refuses cudaMalloc), replay the graph on new inputs twice."""
    import torch
    E, k, T, d = 64, 6, 8, 256
    x_np = [ft_synth.activations(51, i, T, d) for i in range(3)]
    wr_np = ft_synth.router_weight(51, 0, E, d)
    x = to_dev_bf16(x_np[0])
    wr = to_dev_bf16(wr_np)
    idx, w, tie = _outputs(T, k)
    import expert_cached_routed_router_b300 as ftm
    ftm.ft_route_topk_noalloc(x, wr, None, T, E, d, k, idx, w, tie)   # eager, before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=s, capture_error_mode="global"):
        ftm.ft_route_topk_noalloc(x, wr, None, T, E, d, k, idx, w, tie, stream=s)
    for i in (1, 2):
        x.copy_(to_dev_bf16(x_np[i]))
        g.replay()
        torch.cuda.synchronize()
        got = (idx.cpu().numpy(), w.cpu().numpy(), tie.cpu().numpy())
        _assert_matches(got, _oracle(x_np[i], wr_np, None, k))


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
