"""Pins of the 4-bit (MXFP4) entry oracle: element and scale values against the OCP MX
tables, nibble order and block scales on hand-built rows, and the full expert network against
the independently pinned bf16 oracle on entries whose values bf16 holds exactly."""
import numpy as np

import ft_synth
from oracle import fp4, moe


def test_e2m1_table():
    # OCP MX v1.0, FP4 E2M1: the eight magnitudes and their negatives
    assert [fp4.e2m1_value(c) for c in range(8)] == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert [fp4.e2m1_value(c) for c in range(8, 16)] == [-0.0, -0.5, -1.0, -1.5, -2.0, -3.0,
                                                         -4.0, -6.0]


def test_e8m0_scale():
    assert fp4.e8m0_value(127) == 1.0 and fp4.e8m0_value(128) == 2.0
    assert fp4.e8m0_value(120) == 2.0 ** -7 and fp4.e8m0_value(0) == 2.0 ** -127
    assert np.isnan(fp4.e8m0_value(255))


def test_nibble_order_and_block_scale():
    """Row of 64 inputs: byte i holds element 2i (low nibble) and 2i+1 (high nibble);
    block 0 scaled by 2, block 1 by 1/4."""
    codes = np.zeros(32, np.uint8)
    codes[0] = 0x21          # element 0 -> code 1 (0.5), element 1 -> code 2 (1.0)
    codes[15] = 0xF7         # element 30 -> code 7 (6.0), element 31 -> code 15 (-6.0)
    codes[16] = 0x0B         # element 32 -> code 11 (-1.5), element 33 -> 0
    scales = np.array([128, 125], np.uint8)
    w = fp4.dequantize(codes, scales, 1, 64)[0]
    want = np.zeros(64)
    want[0], want[1], want[30], want[31] = 1.0, 2.0, 12.0, -12.0
    want[32] = -1.5 / 4
    assert np.array_equal(w, want)


def _bf16_entry_of(wg, wu, wd):
    """The bf16 entry holding the same values (E2M1 times a power of two fits bf16 exactly)."""
    flat = np.concatenate([wg.ravel(), wu.ravel(), wd.ravel()]).astype(np.float32)
    bits = ft_synth.f32_to_bf16_bits(flat)
    assert np.array_equal(moe.bf16_to_f64(bits), flat.astype(np.float64))
    return bits


def test_expert_network_matches_bf16_oracle():
    d, d_ff = 128, 256
    entry = ft_synth.expert_entry_fp4(3, 1, 2, d, d_ff)
    assert entry.size == fp4.entry_bytes(d, d_ff)
    wg, wu, wd = fp4.split_entry(entry, d, d_ff)
    x = moe.bf16_to_f64(ft_synth.activations(3, 0, 3, d))
    y4 = fp4.expert_ffn_fp4(x, entry, d, d_ff)
    y16 = moe.expert_ffn(x, _bf16_entry_of(wg, wu, wd), d, d_ff)
    assert np.array_equal(y4, y16)


def test_entry_regions_are_independent():
    """Changing one code byte of W_down changes only W_down, in the two elements it holds."""
    d, d_ff = 128, 128
    entry = ft_synth.expert_entry_fp4(4, 0, 0, d, d_ff).copy()
    a = fp4.split_entry(entry, d, d_ff)
    off = 2 * d * d_ff // 2 + 5 * (d_ff // 2) + 3     # W_down row 5, byte 3
    entry[off] ^= 0x77
    b = fp4.split_entry(entry, d, d_ff)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    diff = np.argwhere(a[2] != b[2])
    assert {tuple(v) for v in diff} <= {(5, 6), (5, 7)} and len(diff) >= 1


def test_generator_values():
    """The synthetic 4-bit entries: codes of every value, scales 2^-9 .. 2^-7."""
    d, d_ff = 256, 128
    e = ft_synth.expert_entry_fp4(0, 0, 0, d, d_ff)
    n2 = 3 * d * d_ff // 2
    sc = e[n2:]
    assert set(np.unique(sc).tolist()) == {118, 119, 120}
    nib = np.concatenate([e[:n2] & 15, e[:n2] >> 4])
    assert set(np.unique(nib).tolist()) == set(range(16))
    wg, wu, wd = fp4.split_entry(e, d, d_ff)
    rms = np.sqrt(np.mean(np.concatenate([wg.ravel(), wu.ravel(), wd.ravel()]) ** 2))
    assert 0.005 < rms < 0.03
