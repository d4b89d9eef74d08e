"""Rounding of fp64 oracle values to the library's storage types (test infrastructure only).

A bf16 output is graded against RNE_bf16(o), o the fp64 oracle value rounded once,
directly to bf16 (8 significant bits, ties to even) with no stop in fp32, and
against that value's two bf16 neighbours.
"""
from __future__ import annotations

import numpy as np

_BF16_MIN_EXP = -133          # spacing of bf16 subnormals: 2^-133
_BF16_MAX = float.fromhex("0x1.fep127")


def round_bf16(x) -> np.ndarray:
    """fp64 -> nearest bf16 value (returned as float64), ties to even, overflow to +-inf."""
    x = np.asarray(x, np.float64)
    out = np.array(x, copy=True)
    fin = np.isfinite(x) & (x != 0)
    xf = x[fin]
    m, e = np.frexp(xf)                      # xf = m * 2^e, 0.5 <= |m| < 1
    # 8 significant bits -> quantum 2^(e-8); bf16 subnormals have a fixed quantum 2^-133
    q = np.maximum(e - 8, _BF16_MIN_EXP)
    r = np.rint(np.ldexp(xf, -q))            # exact scaling by a power of two; rint = ties-to-even
    v = np.ldexp(r, q)
    v = np.where(np.abs(v) > _BF16_MAX, np.copysign(np.inf, v), v)
    out[fin] = v
    return out


def bf16_bits(v) -> np.ndarray:
    """uint16 storage bits of values that are exactly representable in bf16."""
    f = np.asarray(v, np.float64).astype(np.float32)
    assert np.array_equal(f.astype(np.float64), np.asarray(v, np.float64), equal_nan=True)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_value(bits) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def bf16_order(bits) -> np.ndarray:
    """Map bf16 bits to integers that are monotone in the value (+0 and -0 both map to 0)."""
    b = np.asarray(bits, np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_ulp_distance(got_bits, want_value) -> np.ndarray:
    """|order(got) - order(RNE_bf16(want))|: 0 exact, 1 a neighbour, ..."""
    want_bits = bf16_bits(round_bf16(want_value))
    return np.abs(bf16_order(got_bits) - bf16_order(want_bits))
