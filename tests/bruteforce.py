"""Brute-force references used only to pin the C oracle on tiny inputs.

Nothing here shares code with ``oracle/oracle.c``; the methods differ on purpose:

* number formats: every finite bf16 / e4m3 code is decoded to an exact
  ``Fraction`` from its bit fields, and rounding is an exhaustive nearest-code
  search (ties to the code with an even last bit) instead of the oracle's
  frexp/nearbyint grid rounding;
* fp32 arithmetic: numpy ``float32`` scalar adds and divides (IEEE library
  arithmetic) instead of C floats;
* the norm: ``decimal`` at 60 significant digits instead of fp64.
"""
from __future__ import annotations

import bisect
from decimal import Decimal, localcontext
from fractions import Fraction

import numpy as np


def _bf16_fraction(code: int):
    s, e, m = (code >> 15) & 1, (code >> 7) & 0xFF, code & 0x7F
    if e == 0xFF:
        return None
    v = Fraction(m, 128) * Fraction(2) ** -126 if e == 0 else (1 + Fraction(m, 128)) * Fraction(2) ** (e - 127)
    return -v if s else v


def _e4m3_fraction(code: int):
    s, e, m = (code >> 7) & 1, (code >> 3) & 0xF, code & 0x7
    if e == 0xF and m == 0x7:
        return None
    v = Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return -v if s else v


def _e2m1_fraction(code: int) -> Fraction:
    s, e, m = (code >> 3) & 1, (code >> 1) & 0x3, code & 0x1
    v = Fraction(m, 2) if e == 0 else (1 + Fraction(m, 2)) * Fraction(2) ** (e - 1)
    return -v if s else v


# Non-negative finite codes in increasing value order.
_BF16_POS = [(_bf16_fraction(c), c) for c in range(0x0000, 0x7F80)]
_BF16_VALS = [v for v, _ in _BF16_POS]
_E4M3_POS = [(_e4m3_fraction(c), c) for c in range(0x00, 0x7F)]
_E4M3_VALS = [v for v, _ in _E4M3_POS]
_E2M1_POS = [(_e2m1_fraction(c), c) for c in range(0x0, 0x8)]
_E2M1_VALS = [v for v, _ in _E2M1_POS]


def e2m1_value(code: int) -> Fraction:
    return _e2m1_fraction(int(code))


def nearest_e2m1_satfinite(x) -> int:
    """Exact RNE of a real to E2M1 with saturation to +-6, by exhaustive search."""
    x = Fraction(x)
    sign = 0x8 if x < 0 else 0
    return sign | _nearest(_E2M1_VALS, _E2M1_POS, abs(x), allow_overflow_code=None)


def bf16_value(code: int) -> Fraction:
    v = _bf16_fraction(int(code))
    if v is None:
        raise ValueError("not finite")
    return v


def e4m3_value(code: int) -> Fraction:
    v = _e4m3_fraction(int(code))
    if v is None:
        raise ValueError("NaN code")
    return v


def _nearest(vals, table, a: Fraction, allow_overflow_code: int | None):
    """Index search for the nearest of ``vals`` to a >= 0, ties to the even code."""
    i = bisect.bisect_left(vals, a)
    if i < len(vals) and vals[i] == a:
        return table[i][1]
    cands = []
    if i > 0:
        cands.append(table[i - 1])
    if i < len(vals):
        cands.append(table[i])
    if len(cands) == 1 and i == len(vals):
        # above the largest finite value
        top_v, top_c = table[-1]
        if allow_overflow_code is None:
            return top_c                       # saturate
        # bf16: the next grid point above max is 2^128; RNE goes there (-> inf)
        # once a reaches the midpoint max + ulp/2 (max has an odd last bit).
        ulp = top_v - table[-2][0]
        return allow_overflow_code if a >= top_v + ulp / 2 else top_c
    (v0, c0), (v1, c1) = cands
    d0, d1 = a - v0, v1 - a
    if d0 < d1:
        return c0
    if d1 < d0:
        return c1
    return c0 if (c0 & 1) == 0 else c1


def nearest_bf16(x) -> int:
    """Exact RNE of a real (Fraction/int/float) to bf16 by exhaustive search."""
    x = Fraction(x)
    sign = 0x8000 if x < 0 else 0
    return sign | _nearest(_BF16_VALS, _BF16_POS, abs(x), allow_overflow_code=0x7F80)


def nearest_e4m3_satfinite(x) -> int:
    """Exact RNE of a real to e4m3fn with saturation to +-448, by exhaustive search."""
    x = Fraction(x)
    sign = 0x80 if x < 0 else 0
    return sign | _nearest(_E4M3_VALS, _E4M3_POS, abs(x), allow_overflow_code=None)


def reduce_rmsnorm(partials: np.ndarray, residual: np.ndarray | None, gamma: np.ndarray, eps: float):
    """Brute-force residual_out and y for tiny inputs (uint16 bf16 bit arrays)."""
    R, T, H = partials.shape
    ro = np.zeros((T, H), dtype=np.uint16)
    y = np.zeros((T, H), dtype=np.uint16)
    eps32 = Fraction(float(np.float32(eps)))
    for t in range(T):
        for h in range(H):
            acc = np.float32(float(bf16_value(partials[0, t, h])))
            for r in range(1, R):
                acc = np.float32(acc + np.float32(float(bf16_value(partials[r, t, h]))))
            res = np.float32(float(bf16_value(residual[t, h]))) if residual is not None else np.float32(0.0)
            acc = np.float32(acc + res)
            ro[t, h] = nearest_bf16(Fraction(float(acc)))
        xs = [bf16_value(ro[t, h]) for h in range(H)]
        mean = sum(x * x for x in xs) / H + eps32
        with localcontext() as ctx:
            ctx.prec = 60
            rstd = 1 / (Decimal(mean.numerator) / Decimal(mean.denominator)).sqrt()
            for h in range(H):
                g = bf16_value(gamma[h])
                prod = Decimal((xs[h] * g).numerator) / Decimal((xs[h] * g).denominator) * rstd
                y[t, h] = nearest_bf16(Fraction(prod))
    return ro, y


def quant_per_group(y: np.ndarray, group: int = 128):
    """Brute-force per-group e4m3 quant: scales in numpy fp32, codes by exhaustive search."""
    T, H = y.shape
    q = np.zeros((T, H), dtype=np.uint8)
    s_out = np.zeros((T, H // group), dtype=np.float32)
    for t in range(T):
        for g in range(H // group):
            vals = [np.float32(float(bf16_value(y[t, g * group + i]))) for i in range(group)]
            a = max(abs(v) for v in vals)
            s = np.float32(np.float32(a) / np.float32(448.0))
            s_out[t, g] = s
            for i, v in enumerate(vals):
                if s == 0:
                    q[t, g * group + i] = 0
                else:
                    q[t, g * group + i] = nearest_e4m3_satfinite(Fraction(float(np.float32(v / s))))
    return q, s_out


def mxfp4(y: np.ndarray):
    """Brute-force MXFP4 of bf16 bits [T, H]: the shared exponent from the exact
    binary logarithm of the block's absmax (no library log), codes by exhaustive
    search; element 2i in the low nibble."""
    T, H = y.shape
    q = np.zeros((T, H // 2), dtype=np.uint8)
    sc = np.zeros((T, H // 32), dtype=np.uint8)
    for t in range(T):
        for b in range(H // 32):
            vals = [bf16_value(y[t, b * 32 + i]) for i in range(32)]
            amax = max(abs(v) for v in vals)
            if amax == 0:
                e = -127
            else:
                e = 0
                while Fraction(2) ** (e + 1) <= amax:
                    e += 1
                while Fraction(2) ** e > amax:
                    e -= 1
                e = max(-127, min(127, e - 2))
            sc[t, b] = e + 127
            for i in range(16):
                lo = nearest_e2m1_satfinite(vals[2 * i] / Fraction(2) ** e) if amax else 0
                hi = nearest_e2m1_satfinite(vals[2 * i + 1] / Fraction(2) ** e) if amax else 0
                q[t, b * 16 + i] = lo | (hi << 4)
    return q, sc
