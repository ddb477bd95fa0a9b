"""Seeded synthetic inputs for the routed MoE layer, shared by the CUDA path and the oracle.

This module draws random numbers and lays them out; it holds none of the layer's
arithmetic (no router, no top-k, no FFN, no cache policy).

Generator definition (the same on the host here and in ``synth.cu`` on the GPU, bit for bit):

* ``mix64`` is the splitmix64 output function (Steele, Lea and Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014; the finaliser constants are
  Stafford's "Mix13").
* A stream is a 64-bit key.  Output ``i`` of stream ``key`` is ``mix64(key + (i+1)*G)``
  with ``G = 0x9E3779B97F4A7C15`` (the splitmix64 increment), i.e. the i-th draw of a
  splitmix64 generator seeded with ``key``: counter based, so any element is
  computable on its own.
* Normal variates use the Irwin-Hall sum of 12 uniforms (the classical "sum of twelve
  uniforms minus six" approximation): variate ``i`` takes draws 3i, 3i+1, 3i+2, splits
  each into four 16-bit fields u_j, and returns ``z = (sum_j u_j - 393210) / 65536``, i.e.
  ``sum_j (u_j + 1/2)/65536 - 6``.  Mean 0, variance 1 - 2^-32, excess kurtosis -0.1,
  support [-6, 6].  Integer sums make it exact (z is an fp32 value), so the host and the
  GPU produce identical bits without any transcendental function.
* A value ``sigma * z`` is one fp32 multiply (sigma rounded to fp32 first), then bf16
  (round to nearest even).  For sigma = 1 the value is bf16(z).

bf16 tensors are returned as ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import numpy as np

G = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Stream tags: which tensor a key belongs to.
TAG_X = 1          # activations
TAG_ROUTER = 2     # router weight W_r[l] [E][d]
TAG_POOL = 3       # routed expert entry (l, e)
TAG_SHARED = 4     # shared expert entry of layer l
TAG_DRIFT = 5      # random-walk increments of the router bias
TAG_PERM = 6       # per-layer popularity order
TAG_POOL_FP4 = 7   # routed expert entry (l, e), 4-bit codes and block scales

ENTRY_SIGMA = 0.02
ROUTER_SIGMA = 0.02


def mix64(z):
    """splitmix64 output function on uint64 (scalars or arrays); wraps mod 2^64."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tag: int, a: int = 0, b: int = 0, c: int = 0) -> int:
    """Key of the stream (seed, tag, a, b, c): a chain of mix64 over the fields."""
    with np.errstate(over="ignore"):
        k = mix64(np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + G)
        for f in (tag, a, b, c):
            k = mix64(k ^ (np.uint64(f & 0xFFFFFFFFFFFFFFFF) * G + np.uint64(1)))
    return int(k)


def draws(key: int, start: int, n: int) -> np.ndarray:
    """Outputs start .. start+n-1 of stream ``key`` as uint64."""
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(np.uint64(key) + i * G)


def normal_f32(key: int, n: int, start: int = 0) -> np.ndarray:
    """Irwin-Hall normals z[start .. start+n-1] of stream ``key`` (exact fp32 values)."""
    s = draws(key, 3 * start, 3 * n).reshape(n, 3)
    tot = np.zeros(n, dtype=np.int64)
    for j in range(3):
        for f in range(4):
            tot += ((s[:, j] >> np.uint64(16 * f)) & np.uint64(0xFFFF)).astype(np.int64)
    return ((tot - 393210).astype(np.float32) / np.float32(65536.0)).astype(np.float32)


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to fp32 exactly."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(key: int, n: int, sigma: float, start: int = 0) -> np.ndarray:
    """bf16(fp32(sigma) * z) as uint16 bits (one fp32 multiply, then round to nearest even)."""
    z = normal_f32(key, n, start)
    if sigma != 1.0:
        z = np.float32(sigma) * z
    return f32_to_bf16_bits(z)


# ---------------------------------------------------------------------------
# Tensors of the layer
# ---------------------------------------------------------------------------

def entry_elems(d: int, d_ff: int) -> int:
    """Elements of one complete (layer, expert) entry: W_gate, W_up and W_down."""
    return 3 * d * d_ff


def expert_entry(seed: int, layer: int, expert: int, d: int, d_ff: int,
                 start: int = 0, n: int | None = None) -> np.ndarray:
    """Flat bf16 entry of routed expert (layer, expert), elements [start, start+n).

    Layout of one entry (row-major, every row contiguous over its input features):
    ``Wg[d_ff][d]`` (row j holds W_gate[:, j]), ``Wu[d_ff][d]``, ``Wd[d][d_ff]``
    (row i holds W_down[:, i]).  Element values are i.i.d. approximately N(0, 0.02^2), so
    the orientation changes no statistic.
    """
    n = entry_elems(d, d_ff) - start if n is None else n
    return normal_bf16(stream_key(seed, TAG_POOL, layer, expert), n, ENTRY_SIGMA, start)


def entry_bytes_fp4(d: int, d_ff: int) -> int:
    """Bytes of one 4-bit entry: 3*d*d_ff codes of 4 bits plus one scale byte per 32."""
    return 3 * d * d_ff * 17 // 32


def expert_entry_fp4(seed: int, layer: int, expert: int, d: int, d_ff: int) -> np.ndarray:
    """Packed 4-bit entry of routed expert (layer, expert) as uint8 [entry_bytes_fp4].

    The first 3*d*d_ff/2 bytes (the codes) are the little-endian bytes of draws
    0 .. 3*d*d_ff/16 - 1 of the stream, so every 4-bit code is uniform over its 16 values;
    the remaining 3*d*d_ff/32 bytes (the block scales) are 118 + (draw mod 3) of the draws
    that follow, one draw per byte.  The layout of the regions is the 4-bit entry layout
    (codes of W_gate, W_up, W_down, then their scales); interpreting it is the oracle's and
    the kernels' business.
    """
    key = stream_key(seed, TAG_POOL_FP4, layer, expert)
    nc = 3 * d * d_ff // 2
    ns = 3 * d * d_ff // 32
    codes = draws(key, 0, nc // 8).astype("<u8").view(np.uint8)
    scales = (np.uint64(118) + draws(key, nc // 8, ns) % np.uint64(3)).astype(np.uint8)
    return np.concatenate([codes, scales])


def shared_entry(seed: int, layer: int, d: int, d_ff: int) -> np.ndarray:
    """Flat bf16 entry of the always-active shared expert of ``layer`` (same layout)."""
    return normal_bf16(stream_key(seed, TAG_SHARED, layer), entry_elems(d, d_ff), ENTRY_SIGMA)


def split_entry(entry: np.ndarray, d: int, d_ff: int):
    """Views (Wg [d_ff][d], Wu [d_ff][d], Wd [d][d_ff]) of a flat entry."""
    n = d * d_ff
    return (entry[:n].reshape(d_ff, d), entry[n:2 * n].reshape(d_ff, d),
            entry[2 * n:3 * n].reshape(d, d_ff))


def router_weight(seed: int, layer: int, E: int, d: int) -> np.ndarray:
    """Router weight W_r of ``layer``: bf16 [E][d] ~ N(0, 0.02^2)."""
    return normal_bf16(stream_key(seed, TAG_ROUTER, layer), E * d, ROUTER_SIGMA).reshape(E, d)


def activations(seed: int, stream: int, T: int, d: int, sigma: float = 1.0) -> np.ndarray:
    """Activations x: bf16 [T][d] ~ N(0, sigma^2); ``stream`` selects the batch (e.g. step)."""
    return normal_bf16(stream_key(seed, TAG_X, stream), T * d, sigma).reshape(T, d)


def popularity_order(seed: int, layer: int, E: int) -> np.ndarray:
    """A seeded permutation pi of the experts; rank(e) = 1 + position of e in pi."""
    u = draws(stream_key(seed, TAG_PERM, layer), 0, E)
    return np.argsort(u, kind="stable").astype(np.int64)


def zipf_rank(seed: int, layer: int, E: int, rotate: int = 0) -> np.ndarray:
    """rank[e] in 1..E for the popularity order of ``layer``, optionally rotated.

    ``rotate = E // 2`` gives the disjoint-hot-half order used by the phase-switching trace.
    """
    pi = popularity_order(seed, layer, E)
    pi = np.roll(pi, -rotate) if rotate else pi
    rank = np.empty(E, dtype=np.int64)
    rank[pi] = np.arange(1, E + 1)
    return rank


class DriftingZipfBias:
    """Router bias of a decode trace: ``-s * ln(rank_l(e)) + r_{t,l,e}`` (fp32).

    ``r`` is a random walk, ``r_{t} = r_{t-1} + sigma_walk * N(0,1)`` per (layer, expert),
    ``r_0 = 0``, kept in double.  ``phase_len`` > 0 switches the popularity order to the
    half-rotated one on every odd block of ``phase_len`` steps.
    """

    def __init__(self, seed: int, L: int, E: int, s: float, sigma_walk: float = 0.02,
                 phase_len: int = 0):
        self.seed, self.L, self.E, self.s = seed, L, E, s
        self.sigma_walk, self.phase_len = sigma_walk, phase_len
        self.logr = [[-s * np.log(zipf_rank(seed, l, E, rot).astype(np.float64))
                      for rot in (0, E // 2)] for l in range(L)]
        self.r = np.zeros((L, E), dtype=np.float64)
        self.t = 0

    def advance(self):
        """Advance the walk to the next step."""
        self.t += 1
        for l in range(self.L):
            self.r[l] += self.sigma_walk * normal_f32(
                stream_key(self.seed, TAG_DRIFT, l, self.t), self.E).astype(np.float64)

    def bias(self, layer: int) -> np.ndarray:
        """fp32 [E] bias of ``layer`` at the current step."""
        phase = 0
        if self.phase_len > 0 and ((self.t - 1) // self.phase_len) % 2 == 1:
            phase = 1
        return (self.logr[layer][phase] + self.r[layer]).astype(np.float32)
