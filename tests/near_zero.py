"""Blocks at the bottom of the binary32 / bf16 range, where the method's
Adaptive Scale matters most (the near-zero "zero collapse" region of the TACO
paper, Section 4.2.1 and Fig. 5): alpha = tau / sqrt(m + eps) is about 1e15
there, so the oracle's scaled block alpha * G is an ordinary float, while the
unscaled rotation H G of a kernel can sit near or inside the subnormal range.

Each builder returns bf16 bit patterns of shape [blocks, B]; the values are
exact in bf16 (and in float64), so the float64 helpers can check them.
"""
from __future__ import annotations

import numpy as np

from helpers import hadamard

FLT_MAX = float(np.finfo(np.float32).max)
CODE_QMAX = {0: 448.0, 1: 57344.0}
BF16_MIN_SUBNORMAL = 2.0 ** -133


def bf16_bits(values) -> np.ndarray:
    """bf16 bit patterns of float64 values that are exact in bf16 (checked)."""
    v = np.asarray(values, dtype=np.float64)
    f = v.astype(np.float32)
    assert np.array_equal(f.astype(np.float64), v), "value not exact in float32"
    bits = f.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0), "value not exact in bf16"
    return (bits >> 16).astype(np.uint16)


def largest_bf16_below(x: float) -> float:
    """The largest positive bf16 value strictly below x (x a normal float)."""
    e = np.floor(np.log2(x))
    step = 2.0 ** (e - 7)
    v = np.floor(x / step) * step
    return float(v - step if v >= x else v)


def near_zero_blocks(B: int, code: int = 0, seed: int = 7) -> np.ndarray:
    """The tiny blocks of the near-zero tests, as bf16 bits [blocks, B]:

    - c (e_0 + e_1) for c = 2^-120 and 2^-125;
    - one bf16 subnormal 2^-133 (the smallest) and one 2^-127;
    - c h_i (a Hadamard row) with c = 2^-130: every input subnormal, the
      rotation c B e_i normal;
    - random bf16 subnormals k 2^-133, |k| < 128, some zeros;
    - random subnormals next to one normal value 2^-126;
    - a single element x e_j and x h_i / sqrt-free variants whose max|H G|
      is the largest bf16 value below Q_max / FLT_MAX, and one step above it
      (where Q_max / max|H G| first overflows binary32);
    - random values of magnitude about 2^-118 to 2^-122 (normal bf16).
    """
    rng = np.random.default_rng(seed + 1000 * code + B)
    H = hadamard(B)
    rows = []

    def unit(j):
        e = np.zeros(B)
        e[j] = 1.0
        return e

    for c in (2.0 ** -120, 2.0 ** -125):
        rows.append(c * (unit(0) + unit(1)))
    rows.append(BF16_MIN_SUBNORMAL * unit(5))
    rows.append(-(2.0 ** -127) * unit(B - 1))
    rows.append(2.0 ** -130 * H[3 % B])
    k = rng.integers(-127, 128, size=B).astype(np.float64)
    k[rng.random(B) < 0.2] = 0.0
    k[0] = 127.0
    rows.append(k * BF16_MIN_SUBNORMAL)
    k2 = rng.integers(-127, 128, size=B).astype(np.float64)
    k2 = k2 * BF16_MIN_SUBNORMAL
    k2[B // 3] = 2.0 ** -126
    rows.append(k2)
    thr = CODE_QMAX[code] / FLT_MAX
    below = largest_bf16_below(thr)
    above = below + 2.0 ** (np.floor(np.log2(below)) - 7)
    rows.append(below * unit(B // 2))
    rows.append(-above * unit(1))
    # A block with several nonzeros whose rotation's maximum is `below`:
    # x = below * (e_0 + e_1) / 2 has H x = below on the even columns.
    rows.append(below / 2 * (unit(0) + unit(1)))
    # Random normal-but-tiny values, rounded to bf16 in float64.
    mag = 2.0 ** rng.uniform(-122, -118, size=(2, B))
    sign = np.where(rng.random((2, B)) < 0.5, -1.0, 1.0)
    v = (sign * mag).astype(np.float32)
    v = (v.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)
    rows.extend(list(v))
    return np.stack([bf16_bits(r) for r in rows])
