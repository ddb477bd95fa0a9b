"""The seeded input generator: published splitmix64 vectors, Irwin-Hall normal moments, bf16 rounding."""
import numpy as np

import ft_synth


def test_splitmix64_published_vectors():
    # splitmix64 seeded with 0: first outputs of the reference generator
    got = ft_synth.draws(0, 0, 3)
    assert [int(v) for v in got] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_access_is_random_access():
    k = ft_synth.stream_key(0, ft_synth.TAG_POOL, 3, 5)
    full = ft_synth.normal_f32(k, 101)
    for s, n in [(0, 1), (1, 1), (1, 6), (37, 20), (100, 1)]:
        assert np.array_equal(ft_synth.normal_f32(k, n, start=s), full[s:s + n])


def test_irwin_hall_by_hand():
    """Variate 0 of a stream from its three draws, field by field."""
    key = ft_synth.stream_key(0, ft_synth.TAG_X, 9)
    d = [int(v) for v in ft_synth.draws(key, 0, 3)]
    tot = sum((v >> (16 * f)) & 0xFFFF for v in d for f in range(4))
    assert float(ft_synth.normal_f32(key, 1)[0]) == (tot - 393210) / 65536.0


def test_normal_moments():
    """Irwin-Hall(12): mean 0, variance 1 - 2^-32, kurtosis 3 - 6/60 = 2.9, |z| <= 6."""
    z = ft_synth.normal_f32(ft_synth.stream_key(0, ft_synth.TAG_X, 0), 400_000).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    assert abs(np.mean(z ** 4) - 2.9) < 0.05
    assert np.abs(z).max() <= 6.0


def test_bf16_round_to_nearest_even():
    f = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 65504.0], np.float32)
    b = ft_synth.bf16_bits_to_f32(ft_synth.f32_to_bf16_bits(f))
    # 1+2^-8 is a tie between 1 and 1+2^-7 -> even (1.0); 1+3*2^-8 -> 1+2^-6 (even)
    assert list(b) == [1.0, 1.0, 1.0 + 2 ** -6, 1.0, -2.5, 65536.0]


def test_streams_are_distinct():
    a = ft_synth.expert_entry(0, 0, 0, 8, 8)
    b = ft_synth.expert_entry(0, 0, 1, 8, 8)
    c = ft_synth.expert_entry(0, 1, 0, 8, 8)
    assert not np.array_equal(a, b) and not np.array_equal(a, c)


def test_drifting_bias_phase_switch():
    gen = ft_synth.DriftingZipfBias(0, 2, 16, 1.1, phase_len=3)
    tops = []
    for _ in range(6):
        gen.advance()
        tops.append(int(np.argmax(gen.bias(0))))
    r0 = ft_synth.zipf_rank(0, 0, 16)
    r1 = ft_synth.zipf_rank(0, 0, 16, rotate=8)
    assert tops[0] == int(np.argmin(r0)) and tops[3] == int(np.argmin(r1))
    assert set(np.nonzero(r0 <= 8)[0]).isdisjoint(set(np.nonzero(r1 <= 8)[0]))
