"""Oracle of one routed MoE layer forward (TEST INFRASTRUCTURE ONLY).

Definition implemented (the pages name the parts - top-k routed experts, expert networks,
a combine - but print no formula; the plain reading, stated once here):

1. Router logits  l[t, e] = sum_i x[t, i] * W_r[e, i]  (+ bias[e]), bf16 inputs, fp32
   arithmetic in ONE fixed order (``router_logits``), so that the choice of experts is a
   reproducible function of the inputs.
2. Top-k: the k experts with the largest logits, larger logit first, lower expert id first
   on equal logits (``topk``).  "6 of 256 routed experts per layer" is the pages' example
   (FreeToken RTX 4090, section "how the MoE memory hierarchy works").
3. Gates: softmax over all E logits, renormalised over the selected k; the full-softmax
   denominator cancels, so w_j = exp(l_j - l_max) / sum_{i<k} exp(l_i - l_max) (``gates``).
4. Permutation grouped by expert: pairs p = t*k + j ordered by (expert, t, j) (``permutation``).
5. Expert e: SwiGLU FFN  y = W_down^T (silu(W_gate^T x) * (W_up^T x)) in fp64 (``expert_ffn``).
6. Combine: out[t] = sum_j w[t, j] * y_{idx[t, j]}(x_t)  (+ the shared expert with weight 1).
7. Prefill residual stream (attention omitted): layer i+1 reads x_{i+1} = bf16(x_i + out_i)
   (``residual_next``); the layers are checked one by one on the GPU's own x_i.
"""
from __future__ import annotations

import math

import numpy as np

NEAR_TIE = 1e-6   # absolute fp32 logit gap below which a top-k decision is reported


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def bf16_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float32 values."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32)


def f32_to_bf16_bits(v) -> np.ndarray:
    """float32 values -> bf16 bit patterns (uint16), rounded to nearest, ties to even
    (finite values; the 16 dropped bits decide, with the kept last bit breaking ties)."""
    u = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return (u >> np.uint64(16)).astype(np.uint16)


def residual_next(x_bits, out_bits) -> np.ndarray:
    """Input of the next layer of a prefill's residual stream (attention omitted): the layer's
    bf16 input plus its bf16 output, added in fp32 and rounded to bf16 (nearest even)."""
    s = bf16_to_f32(x_bits) + bf16_to_f32(out_bits)      # one IEEE fp32 add
    return f32_to_bf16_bits(s)


def router_logits(x_bits, wr_bits, bias=None) -> np.ndarray:
    """Router logits in the canonical fp32 order.  x [T][d], W_r [E][d] bf16; bias [E] fp32.

    The order (a reading: the pages fix none; it is the natural one for a 32-lane warp
    reading 16-byte vectors):
      * d is cut into chunks of 8 consecutive features, c = 0 .. d/8 - 1;
      * lane lam in 0..31 owns the chunks c with c mod 32 == lam, visited in increasing c,
        and adds the products of each chunk's 8 features in increasing feature order,
        starting from +0.0:  acc_lam = acc_lam + x*w (fp32; the product of two bf16
        values is exact in fp32, so fused or separate multiply-add agree);
      * the 32 partial sums are combined by a butterfly: for off = 16, 8, 4, 2, 1,
        acc_lam = acc_lam + acc_{lam xor off};
      * the logit is acc_0 (+ bias[e], one fp32 add).
    Returns float32 [T][E].
    """
    xf = bf16_to_f32(x_bits)
    wf = bf16_to_f32(wr_bits)
    T, d = xf.shape
    E = wf.shape[0]
    assert d % 8 == 0 and wf.shape[1] == d
    acc = np.zeros((32, T, E), dtype=np.float32)
    for c in range(d // 8):
        lam = c % 32
        for i in range(8):
            f = 8 * c + i
            acc[lam] = acc[lam] + np.outer(xf[:, f], wf[:, f])
    lanes = np.arange(32)
    for off in (16, 8, 4, 2, 1):
        acc = acc + acc[lanes ^ off]
    logits = acc[0]
    if bias is not None:
        logits = logits + np.asarray(bias, dtype=np.float32)[None, :]
    return logits.astype(np.float32)


def topk(logits, k: int):
    """Top-k per token: (idx int32 [T][k], near_tie bool [T]).

    Order: logit descending, expert id ascending among equal logits.  A token is reported
    as a near-tie when the k-th and (k+1)-th logits, or any two selected logits, are within
    1e-6 of each other (the exact difference of the fp32 logits): there a different summation
    order could pick a different expert or rank.
    """
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), dtype=np.int32)
    tie = np.zeros(T, dtype=bool)
    for t in range(T):
        order = np.argsort(-logits[t], kind="stable")
        idx[t] = order[:k]
        sel = logits[t, order[:k]]
        if k < E and float(sel[-1]) - float(logits[t, order[k]]) <= NEAR_TIE:
            tie[t] = True
        if k > 1 and np.min(np.diff(-sel.astype(np.float64))) <= NEAR_TIE:
            tie[t] = True
    return idx, tie


def gates(logits, idx) -> np.ndarray:
    """Gate weights w [T][k] (fp32), softmax renormalised over the selected experts.

    Computed in double and rounded once: w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0),
    l_0 the largest selected logit.
    """
    logits = np.asarray(logits, dtype=np.float32)
    T, k = idx.shape
    w = np.empty((T, k), dtype=np.float32)
    for t in range(T):
        sel = logits[t, idx[t]].astype(np.float64)
        ex = np.exp(sel - sel.max())
        w[t] = (ex / ex.sum()).astype(np.float32)
    return w


def permutation(idx, E: int):
    """Group the (token, rank) pairs by expert.

    Pairs are numbered p = t*k + j.  Returns
      counts  int32 [E]    pairs routed to each expert,
      offsets int32 [E+1]  exclusive prefix sum of counts (offsets[E] = T*k),
      perm    int32 [P]    perm[q] = the pair at position q, pairs ordered by (expert, p),
      inv     int32 [P]    inv[p] = position of pair p.
    """
    flat = np.asarray(idx, dtype=np.int64).reshape(-1)
    P = flat.size
    counts = np.zeros(E, dtype=np.int64)
    for e in flat:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    perm = np.empty(P, dtype=np.int64)
    fill = offsets[:-1].copy()
    for p in range(P):          # increasing p: stable within each expert
        e = flat[p]
        perm[fill[e]] = p
        fill[e] += 1
    inv = np.empty(P, dtype=np.int64)
    inv[perm] = np.arange(P)
    return (counts.astype(np.int32), offsets.astype(np.int32),
            perm.astype(np.int32), inv.astype(np.int32))


def silu(g):
    """silu(g) = g * sigmoid(g) = g / (1 + exp(-g))."""
    return g / (1.0 + np.exp(-g))


def expert_ffn(x_f64, entry_bits, d: int, d_ff: int) -> np.ndarray:
    """SwiGLU expert on rows x [n][d] (float64) -> y [n][d] float64.

    ``entry_bits`` is one flat bf16 entry: Wg [d_ff][d] | Wu [d_ff][d] | Wd [d][d_ff],
    each row one output feature (so W_gate = Wg^T is the d x d_ff matrix).
      g = x W_gate,  u = x W_up,  h = silu(g) * u,  y = h W_down.
    """
    n = d * d_ff
    e = np.asarray(entry_bits, dtype=np.uint16)
    wg = bf16_to_f64(e[:n]).reshape(d_ff, d)
    wu = bf16_to_f64(e[n:2 * n]).reshape(d_ff, d)
    wd = bf16_to_f64(e[2 * n:3 * n]).reshape(d, d_ff)
    return swiglu_rows(x_f64, wg, wu, wd)


def swiglu_rows(x_f64, wg, wu, wd) -> np.ndarray:
    """g = x Wg^T, u = x Wu^T, h = silu(g) * u, y = h Wd^T on rows x [n][d], in float64."""
    x = np.atleast_2d(np.asarray(x_f64, dtype=np.float64))
    g = x @ wg.T
    u = x @ wu.T
    h = silu(g) * u
    return h @ wd.T


def moe_layer(x_bits, wr_bits, k: int, entry_of, d: int, d_ff: int, bias=None,
              shared_entry=None, tokens=None, ffn=None):
    """One routed MoE layer forward.

    x [T][d] bf16, W_r [E][d] bf16, ``entry_of(e)`` -> flat bf16 entry of expert e.
    ``tokens``: optional subset of token rows whose outputs are computed (routing is
    always computed for all T).  ``ffn(x, entry, d, d_ff)``: the expert network of an entry
    (default ``expert_ffn``, bf16 entries).  Returns a dict with logits, idx, tie, w, counts,
    offsets, perm, inv and ``out`` (float64 [len(tokens)][d]).
    """
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    T = x_bits.shape[0]
    E = np.asarray(wr_bits).shape[0]
    logits = router_logits(x_bits, wr_bits, bias)
    idx, tie = topk(logits, k)
    w = gates(logits, idx)
    counts, offsets, perm, inv = permutation(idx, E)
    rows = np.arange(T) if tokens is None else np.asarray(tokens)
    xf = bf16_to_f64(x_bits)
    out = np.zeros((len(rows), d), dtype=np.float64)
    ffn = expert_ffn if ffn is None else ffn
    cache = {}
    for r, t in enumerate(rows):
        for j in range(k):
            e = int(idx[t, j])
            if e not in cache:
                cache[e] = np.asarray(entry_of(e))
            out[r] += float(w[t, j]) * ffn(xf[t], cache[e], d, d_ff)[0]
        if shared_entry is not None:
            out[r] += ffn(xf[t], shared_entry, d, d_ff)[0]
    return dict(logits=logits, idx=idx, tie=tie, w=w, counts=counts, offsets=offsets,
                perm=perm, inv=inv, out=out, tokens=rows)


def dense_swiglu(x, w_gate, w_up, w_down) -> np.ndarray:
    """A dense SwiGLU FFN written out element by element (for the 1-expert special case).

    x [n][d]; W_gate, W_up [d][d_ff]; W_down [d_ff][d] (the column-vector-free
    convention y = (silu(x W_gate) * (x W_up)) W_down), all float64.
    """
    x = np.atleast_2d(x)
    n, d = x.shape
    d_ff = w_gate.shape[1]
    y = np.zeros((n, w_down.shape[1]))
    for r in range(n):
        h = np.empty(d_ff)
        for j in range(d_ff):
            g = math.fsum(x[r, i] * w_gate[i, j] for i in range(d))
            u = math.fsum(x[r, i] * w_up[i, j] for i in range(d))
            h[j] = g / (1.0 + math.exp(-g)) * u
        for o in range(w_down.shape[1]):
            y[r, o] = math.fsum(h[j] * w_down[j, o] for j in range(d_ff))
    return y


def within_tolerance(gpu, ref):
    """Output bar: max|gpu - ref| <= 1e-2 * max|ref| + 1e-3 (bf16 weights).

    Returns (ok, max_err, bound)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = float(np.max(np.abs(gpu - ref))) if ref.size else 0.0
    bound = 1e-2 * (float(np.max(np.abs(ref))) if ref.size else 0.0) + 1e-3
    return err <= bound, err, bound
