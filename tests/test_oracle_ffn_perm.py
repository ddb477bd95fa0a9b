"""Pins of the oracle's permutation, expert FFN and combine."""
import math

import numpy as np
import pytest
import torch

import ft_synth
from oracle import moe


def _route(T, E, k, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,k", [(1, 4, 1), (7, 16, 2), (64, 16, 2), (33, 128, 8), (50, 256, 6)])
def test_permutation_identity_and_order(T, E, k):
    idx = _route(T, E, k, T * E)
    counts, offsets, perm, inv = moe.permutation(idx, E)
    P = T * k
    assert offsets[0] == 0 and offsets[E] == P and counts.sum() == P
    assert np.array_equal(np.diff(offsets), counts)
    # brute force: pairs sorted by (expert, token, rank)
    want = sorted(range(P), key=lambda p: (idx[p // k, p % k], p // k, p % k))
    assert list(perm) == want
    # permute then un-permute random rows: identity
    X = np.random.default_rng(1).standard_normal((P, 5))
    Xp = X[perm]
    assert np.array_equal(Xp[inv], X)
    # every position inside expert e's range holds a pair routed to e
    flat = idx.reshape(-1)
    for e in range(E):
        assert np.all(flat[perm[offsets[e]:offsets[e + 1]]] == e)


def test_permutation_degenerate():
    idx = np.zeros((9, 1), np.int32) + 3          # all tokens on one expert, others empty
    counts, offsets, perm, inv = moe.permutation(idx, 5)
    assert list(counts) == [0, 0, 0, 9, 0]
    assert list(offsets) == [0, 0, 0, 0, 9, 9]
    assert list(perm) == list(range(9))
    counts, offsets, perm, inv = moe.permutation(np.zeros((0, 2), np.int32), 4)
    assert list(offsets) == [0] * 5 and perm.size == 0


def test_silu_closed_forms():
    assert moe.silu(np.float64(0.0)) == 0.0
    np.testing.assert_allclose(moe.silu(np.log(3.0)), 0.75 * np.log(3.0), rtol=1e-15)
    np.testing.assert_allclose(moe.silu(-np.log(3.0)), -0.25 * np.log(3.0), rtol=1e-15)
    g = np.linspace(-8, 8, 101)
    np.testing.assert_allclose(moe.silu(g), torch.nn.functional.silu(torch.tensor(g)).numpy(),
                               rtol=1e-14, atol=1e-300)


def _logical(entry, d, d_ff):
    """W_gate, W_up [d][d_ff] and W_down [d_ff][d] from the documented entry layout."""
    wg, wu, wd = ft_synth.split_entry(entry, d, d_ff)
    f = moe.bf16_to_f64
    return f(wg).T.copy(), f(wu).T.copy(), f(wd).T.copy()


def _torch_dense(x, w_gate, w_up, w_down):
    x = torch.tensor(x, dtype=torch.float64)
    return ((torch.nn.functional.silu(x @ torch.tensor(w_gate)) * (x @ torch.tensor(w_up)))
            @ torch.tensor(w_down)).numpy()


def test_single_expert_top1_is_dense_swiglu():
    """E = 1, k = 1: the layer is a dense SwiGLU FFN (gate 1); d != d_ff catches transposes."""
    d, d_ff, T = 24, 16, 5
    entry = ft_synth.expert_entry(0, 0, 0, d, d_ff)
    x = ft_synth.activations(0, 0, T, d)
    wr = ft_synth.router_weight(0, 0, 1, d)
    r = moe.moe_layer(x, wr, 1, lambda e: entry, d, d_ff)
    assert np.all(r["idx"] == 0) and np.all(r["w"] == 1.0)
    xf = moe.bf16_to_f64(x)
    wg, wu, wdn = _logical(entry, d, d_ff)
    np.testing.assert_allclose(r["out"], _torch_dense(xf, wg, wu, wdn), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(r["out"], moe.dense_swiglu(xf, wg, wu, wdn), rtol=1e-12, atol=1e-15)


def test_identical_experts_sum_to_dense():
    """All experts equal: out = dense(x) because the gates sum to 1."""
    d, d_ff, E, k, T = 16, 8, 6, 3, 7
    entry = ft_synth.expert_entry(1, 0, 0, d, d_ff)
    x = ft_synth.activations(1, 0, T, d)
    wr = ft_synth.router_weight(1, 0, E, d)
    r = moe.moe_layer(x, wr, k, lambda e: entry, d, d_ff)
    dense = _torch_dense(moe.bf16_to_f64(x), *_logical(entry, d, d_ff))
    np.testing.assert_allclose(r["out"], dense, rtol=1e-6, atol=1e-12)


def test_scaled_experts_weight_by_gates():
    """Expert e = base expert with W_down scaled by (e+1): out = (sum_j w_j (e_j+1)) dense(x).

    The scale is a power of two or small integer so the scaled bf16 weights stay exact;
    a gate applied to the wrong rank, or a missing gate, breaks the identity."""
    d, d_ff, E, k, T = 16, 8, 4, 2, 9
    base = ft_synth.expert_entry(2, 0, 0, d, d_ff)
    n = d * d_ff
    scales = [1.0, 2.0, 4.0, 8.0]

    def entry_of(e):
        f = moe.bf16_to_f64(base).astype(np.float32)
        f[2 * n:] *= scales[e]
        return ft_synth.f32_to_bf16_bits(f)

    x = ft_synth.activations(2, 0, T, d)
    wr = ft_synth.router_weight(2, 0, E, d)
    r = moe.moe_layer(x, wr, k, entry_of, d, d_ff)
    dense = _torch_dense(moe.bf16_to_f64(x), *_logical(base, d, d_ff))
    factor = np.array([sum(float(r["w"][t, j]) * scales[r["idx"][t, j]] for j in range(k))
                       for t in range(T)])
    np.testing.assert_allclose(r["out"], factor[:, None] * dense, rtol=1e-12, atol=1e-15)
    # the two experts of a token really differ, so the test is not vacuous
    assert np.all(r["idx"][:, 0] != r["idx"][:, 1])


def test_shared_expert_adds_with_weight_one():
    d, d_ff, E, k, T = 16, 8, 4, 2, 3
    entry = ft_synth.expert_entry(3, 0, 0, d, d_ff)
    x = ft_synth.activations(3, 0, T, d)
    wr = ft_synth.router_weight(3, 0, E, d)
    r = moe.moe_layer(x, wr, k, lambda e: entry, d, d_ff, shared_entry=entry)
    dense = _torch_dense(moe.bf16_to_f64(x), *_logical(entry, d, d_ff))
    np.testing.assert_allclose(r["out"], 2 * dense, rtol=1e-6, atol=1e-12)


def test_token_subset_matches_full():
    d, d_ff, E, k, T = 32, 16, 8, 2, 10
    x = ft_synth.activations(4, 0, T, d)
    wr = ft_synth.router_weight(4, 0, E, d)
    ent = {e: ft_synth.expert_entry(4, 0, e, d, d_ff) for e in range(E)}
    full = moe.moe_layer(x, wr, k, ent.__getitem__, d, d_ff)
    sub = moe.moe_layer(x, wr, k, ent.__getitem__, d, d_ff, tokens=[7, 2])
    np.testing.assert_array_equal(sub["out"], full["out"][[7, 2]])


def test_tolerance_rule():
    ok, err, bound = moe.within_tolerance([1.0, 2.0], [1.0, 2.0])
    assert ok and err == 0 and math.isclose(bound, 0.021)
    ok, _, _ = moe.within_tolerance([1.0, 2.03], [1.0, 2.0])
    assert not ok
