"""Pins of the oracle's router, top-k and gates against things other than itself."""
import itertools
import json
import os

import numpy as np
import pytest
from scipy.special import softmax

import ft_synth
from oracle import moe

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "router_order.json")


def _bits(vals):
    return ft_synth.f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_router_order_golden(case):
    d = case["d"]
    x = np.zeros(d, np.float32)
    w = np.zeros(d, np.float32)
    for f, xv, wv in case["features"]:
        x[f], w[f] = xv, wv
    # the golden values must be representable in bf16 (they are powers of two or 1)
    assert np.array_equal(ft_synth.bf16_bits_to_f32(_bits(x)), x)
    bias = None if case["bias"] is None else np.array([case["bias"]], np.float32)
    got = moe.router_logits(_bits(x)[None, :], _bits(w)[None, :], bias)
    assert got.dtype == np.float32
    assert float(got[0, 0]) == case["expected"]


@pytest.mark.parametrize("d", [8, 64, 256, 520, 2048])
def test_router_logits_within_fp32_error_bound(d):
    """|l - exact| <= gamma_n * sum|x_i w_i| with n = (terms per lane) + 5 butterfly levels + 1."""
    rng = np.random.default_rng(d)
    T, E = 5, 7
    x = _bits(rng.standard_normal((T, d)))
    w = _bits(0.02 * rng.standard_normal((E, d)))
    bias = rng.standard_normal(E).astype(np.float32)
    got = moe.router_logits(x, w, bias).astype(np.float64)
    xf = ft_synth.bf16_bits_to_f32(x).astype(np.float64)
    wf = ft_synth.bf16_bits_to_f32(w).astype(np.float64)
    exact = xf @ wf.T + bias[None, :]
    n = -(-d // 256) * 8 + 5 + 1
    u = 2.0 ** -24
    gamma = n * u / (1 - n * u)
    bound = gamma * (np.abs(xf) @ np.abs(wf).T + np.abs(bias)[None, :])
    assert np.all(np.abs(got - exact) <= bound)
    # and it is a real dot product, not a permuted one
    assert np.corrcoef(got.ravel(), exact.ravel())[0, 1] > 0.999999


def _brute_topk(row, k):
    """k rounds of a full scan: larger value wins, lower index on equal values."""
    chosen = []
    for _ in range(k):
        best = None
        for e, v in enumerate(row):
            if e in chosen:
                continue
            if best is None or v > row[best]:
                best = e
        chosen.append(best)
    return chosen


@pytest.mark.parametrize("E,k", [(4, 1), (6, 2), (16, 2), (33, 5), (128, 8), (256, 6)])
def test_topk_matches_brute_force(E, k):
    rng = np.random.default_rng(E * 100 + k)
    logits = rng.standard_normal((12, E)).astype(np.float32)
    # plant exact ties: copy values between experts, including across the k-th boundary
    logits[0, 1] = logits[0, 0]
    logits[1, :] = 0.5
    logits[2, E - 1] = logits[2].max()
    idx, _ = moe.topk(logits, k)
    for t in range(logits.shape[0]):
        assert list(idx[t]) == _brute_topk(list(logits[t]), k)


def test_topk_subset_is_the_argmax_subset():
    """For tiny E, the selected set maximises the sum over all k-subsets (distinct logits)."""
    rng = np.random.default_rng(7)
    for _ in range(50):
        E, k = 6, 3
        row = rng.permutation(E).astype(np.float32) + rng.random(E).astype(np.float32) * 0.1
        idx, _ = moe.topk(row[None, :], k)
        best = max(itertools.combinations(range(E), k), key=lambda s: sum(row[list(s)]))
        assert set(idx[0]) == set(best)


def test_near_tie_flags():
    E, k = 5, 2
    base = np.array([3.0, 2.0, 1.0, 0.0, -1.0], np.float32)
    cases = [
        (base, False),
        (np.array([3.0, 2.0, 2.0, 0.0, -1.0], np.float32), True),              # k-th == (k+1)-th
        (np.array([3.0, 2.0, np.float32(2.0) - np.float32(5e-7), 0, -1], np.float32), True),
        (np.array([3.0, 2.0, 1.999, 0.0, -1.0], np.float32), False),
        (np.array([3.0, 3.0, 1.0, 0.0, -1.0], np.float32), True),              # inside the top-k
    ]
    for row, want in cases:
        _, tie = moe.topk(row[None, :], k)
        assert bool(tie[0]) == want, row


@pytest.mark.parametrize("E,k", [(8, 1), (16, 2), (128, 8), (256, 6)])
def test_gates_are_renormalised_full_softmax(E, k):
    """Closed form: renormalising the full softmax over the top-k equals the top-k softmax."""
    rng = np.random.default_rng(E + k)
    logits = (3 * rng.standard_normal((20, E))).astype(np.float32)
    idx, _ = moe.topk(logits, k)
    w = moe.gates(logits, idx)
    full = softmax(logits.astype(np.float64), axis=1)
    for t in range(20):
        sel = full[t, idx[t]]
        np.testing.assert_allclose(w[t], sel / sel.sum(), rtol=2e-7, atol=1e-9)
        assert abs(float(w[t].astype(np.float64).sum()) - 1.0) <= 1e-6
        assert np.all(np.diff(w[t]) <= 0)       # rank order = gate order
    if k == 1:
        assert np.all(w == 1.0)


def test_gates_two_way_closed_form():
    """l = (a, a - ln 3) -> w = (3/4, 1/4) exactly up to one rounding."""
    a = np.float32(0.25)
    logits = np.array([[a, a - np.float32(np.log(3.0)), -5.0]], np.float32)
    idx, _ = moe.topk(logits, 2)
    w = moe.gates(logits, idx)
    assert list(idx[0]) == [0, 1]
    gap = float(logits[0, 0]) - float(logits[0, 1])     # the fp32 gap actually used
    np.testing.assert_allclose(w[0], [1 / (1 + np.exp(-gap)), 1 / (1 + np.exp(gap))], rtol=1e-7)
    np.testing.assert_allclose(w[0], [0.75, 0.25], rtol=1e-6)
