"""Oracle of 4-bit (MXFP4) routed-expert entries (TEST INFRASTRUCTURE ONLY).

The pages deploy routed experts in MXFP4 (FreeToken benchmark, "benchmark results", model
table: the DeepSeek-V4-Flash routed experts) without defining the format.  Reading: the OCP
Microscaling (MX) v1.0 MXFP4 format -

* element: FP4 E2M1 - 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit, no infinities
  or NaN; exponent field 0 is subnormal (0 or 0.5), otherwise 2^(e-1) * (1 + m/2);
* block: 32 consecutive elements share one E8M0 scale, the power of two 2^(s - 127)
  (s = 255 is NaN);
* value = element * scale.

Packing and entry layout (readings; the pages give none).  A row of K inputs holds K/2 code
bytes, element 2i in the low nibble and 2i+1 in the high nibble of byte i, and K/32 scale
bytes, block b covering elements 32b .. 32b+31.  One entry is

    codes  Wg [d_ff][d/2] | codes Wu [d_ff][d/2] | codes Wd [d][d_ff/2]
  | scales Wg [d_ff][d/32] | scales Wu [d_ff][d/32] | scales Wd [d][d_ff/32]

with the same row orientation as the bf16 entry (row j of Wg holds W_gate[:, j]), i.e.
3*d*d_ff*17/32 bytes.  The expert network applied to the dequantized weights is the bf16
oracle's SwiGLU in fp64.
"""
from __future__ import annotations

import numpy as np

from . import moe as _moe


def e2m1_value(code: int) -> float:
    """Value of a 4-bit E2M1 code (0..15), from its sign, exponent and mantissa fields."""
    code = int(code)
    sign = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        mag = 0.5 * m                         # subnormal: 2^(1 - bias) * (m / 2)
    else:
        mag = 2.0 ** (e - 1) * (1.0 + 0.5 * m)
    return sign * mag


def e8m0_value(s: int) -> float:
    """Value of an E8M0 block scale byte."""
    s = int(s)
    return float("nan") if s == 255 else 2.0 ** (s - 127)


_E2M1 = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
_E8M0 = np.array([e8m0_value(s) for s in range(256)], dtype=np.float64)


def entry_bytes(d: int, d_ff: int) -> int:
    return 3 * d * d_ff * 17 // 32


def dequantize(codes, scales, rows: int, K: int) -> np.ndarray:
    """codes uint8 [rows * K/2], scales uint8 [rows * K/32] -> float64 [rows][K]."""
    c = np.asarray(codes, dtype=np.uint8).reshape(rows, K // 2)
    s = np.asarray(scales, dtype=np.uint8).reshape(rows, K // 32)
    el = np.empty((rows, K), dtype=np.uint8)
    el[:, 0::2] = c & 0x0F
    el[:, 1::2] = c >> 4
    vals = _E2M1[el]
    return vals * np.repeat(_E8M0[s], 32, axis=1)


def split_entry(entry, d: int, d_ff: int):
    """Dequantized (Wg [d_ff][d], Wu [d_ff][d], Wd [d][d_ff]) of a packed entry (float64)."""
    e = np.asarray(entry, dtype=np.uint8)
    assert e.size == entry_bytes(d, d_ff)
    n2, n32 = d * d_ff // 2, d * d_ff // 32
    cg, cu, cd = e[:n2], e[n2:2 * n2], e[2 * n2:3 * n2]
    s0 = 3 * n2
    sg, su, sd = e[s0:s0 + n32], e[s0 + n32:s0 + 2 * n32], e[s0 + 2 * n32:s0 + 3 * n32]
    return (dequantize(cg, sg, d_ff, d), dequantize(cu, su, d_ff, d),
            dequantize(cd, sd, d, d_ff))


def expert_ffn_fp4(x_f64, entry, d: int, d_ff: int) -> np.ndarray:
    """SwiGLU expert with 4-bit weights on rows x [n][d] (float64) -> y [n][d] float64."""
    wg, wu, wd = split_entry(entry, d, d_ff)
    return _moe.swiglu_rows(x_f64, wg, wu, wd)
