"""Grouped-GEMM parity where expert groups span several 128-row M-tiles (GPU).

The tcgen05 grouped GEMM walks M-tiles of 128 (token, expert) pair rows inside each
expert's group; rows are ordered by token, so a group's later M-tiles hold its larger token
ids.  These cases give groups of 3 to 6 M-tiles with ragged last tiles, several N-blocks per
tile (d_ff / 128 for gate/up, d / 256 or d / 128 for down), and compare EVERY output row
with the oracle at max|gpu-ref| <= 1e-2 max|ref| + 1e-3, through ft_moe_forward (T > 16)
and through the prefill double buffer.
"""
import numpy as np
import pytest

import ft_synth
from oracle import moe as omoe

from helpers import (Config, assert_out_close, assert_routing_equal, make_stack, oracle_layer,
                     out_bits_to_f64, to_dev_bf16)

pytestmark = pytest.mark.gpu


def _forward(st, l, x_bits):
    import torch
    x = to_dev_bf16(x_bits)
    out = torch.empty_like(x)
    st.forward(l, x, out)
    torch.cuda.synchronize()
    return out


def _tiles_per_expert(counts):
    return (np.asarray(counts) + 127) // 128


@pytest.mark.parametrize("E,k,T,d,d_ff,skew", [
    (4, 2, 700, 512, 512, 0.0),    # ~350 rows per expert: 3 M-tiles, down N = 256
    (4, 2, 700, 512, 512, 8.0),    # expert 0 takes every token: 6 M-tiles (last one ragged)
    (4, 3, 520, 384, 640, 0.0),    # d % 256 != 0: down N = 128; 5 gate/up N-blocks
    (8, 2, 1000, 256, 384, 3.0),   # skewed over 8 experts: one large group, small ones
])
def test_forward_every_row_across_m_tiles(E, k, T, d, d_ff, skew):
    import torch
    cfg = Config(L=1, E=E, k=k, d=d, d_ff=d_ff, n_slots=E, seed=31)
    st = make_stack(cfg, max_tokens=T)
    bias = np.zeros(E, np.float32)
    bias[0] = skew
    if skew:
        st.set_router_bias(0, torch.from_numpy(bias).cuda())
    x = ft_synth.activations(31, T, T, d)
    out = _forward(st, 0, x)
    ref = oracle_layer(cfg, 0, x, bias=bias if skew else None)
    assert_routing_equal(st, ref, T)
    tiles = _tiles_per_expert(ref["counts"])
    assert tiles.max() >= 3
    if skew == 8.0:
        assert ref["counts"][0] == T and tiles[0] == 6
    assert_out_close(out_bits_to_f64(out), ref["out"])
    # the rows of the last M-tile of the largest group, on their own
    e = int(np.argmax(ref["counts"]))
    q0 = int(ref["offsets"][e]) + 128 * (int(tiles[e]) - 1)
    last = np.unique(ref["perm"][q0:int(ref["offsets"][e + 1])] // k)
    assert_out_close(out_bits_to_f64(out)[last], ref["out"][last])
    assert st.status() == 0
    st.close()


def test_shared_expert_across_m_tiles():
    """The shared expert is one work item of T rows: T = 300 spans 3 M-tiles."""
    cfg = Config(L=1, E=8, k=2, d=256, d_ff=256, n_slots=8, n_shared=1, seed=33)
    st = make_stack(cfg, max_tokens=512)
    x = ft_synth.activations(33, 300, 300, cfg.d)
    out = _forward(st, 0, x)
    ref = oracle_layer(cfg, 0, x)
    assert_routing_equal(st, ref, 300)
    assert_out_close(out_bits_to_f64(out), ref["out"])
    st.close()


def test_prefill_every_row_across_m_tiles():
    """Two layers through the prefill double buffer, groups of 3+ M-tiles, every row checked."""
    import torch
    cfg = Config(L=2, E=4, k=2, d=512, d_ff=512, n_slots=2, seed=35)
    T = 700
    st = make_stack(cfg, max_tokens=T)
    x = ft_synth.activations(35, 0, T, cfg.d)
    out = torch.empty((cfg.L, T, cfg.d), dtype=torch.int16, device="cuda")
    st.prefill(0, cfg.L, to_dev_bf16(x), out)
    torch.cuda.synchronize()
    xin = x
    for l in range(cfg.L):
        ref = oracle_layer(cfg, l, xin)   # the GPU's own input of layer l (residual stream)
        assert _tiles_per_expert(ref["counts"]).max() >= 3
        assert_out_close(out_bits_to_f64(out[l]), ref["out"])
        xin = omoe.residual_next(xin, out[l].cpu().numpy().view(np.uint16))
    np.testing.assert_array_equal(st.logits(T).view(np.uint32), ref["logits"].view(np.uint32))
    st.close()
