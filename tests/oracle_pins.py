"""Pins for the CPU oracle: each function checks the oracle against something
other than itself -- a format definition, a closed form, a library routine, an
exhaustive search or exact rational brute force -- and raises AssertionError on
a mismatch.

Every pin takes an ``oracle.Oracle`` so that the mutation tests can run the same
pins against deliberately broken copies of the oracle and show that each
plausible mistake (a dropped term, a wrong order, a wrong constant, a wrong
index) trips at least one of them.
"""
from __future__ import annotations

import math
import os
from decimal import Decimal, localcontext
from fractions import Fraction

import numpy as np
import torch

import bruteforce as bf
from reduce_residual_rmsnorm_fp32_gb300.synthetic import f32_to_bf16_bits, bf16_bits_to_f32, make_inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_golden(name: str):
    sections: dict[str, list[tuple[str, str]]] = {}
    cur = None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("["):
                cur = line.strip("[]")
                sections[cur] = []
                continue
            a, b = line.split()
            sections[cur].append((a, b))
    return sections


def _eval(expr: str) -> float:
    return float(eval(expr, {"__builtins__": {}}, {"inf": math.inf}))


def _bits(vals) -> np.ndarray:
    return f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


def _ordered(b: np.ndarray) -> np.ndarray:
    """bf16 bits -> integers whose difference counts representable steps."""
    b = b.astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


# ---------------------------------------------------------------- formats --

def pin_golden_bf16(o):
    g = _read_golden("bf16_points.txt")
    for code, expr in g["decode"]:
        v = _eval(expr)
        got = o.bf16_to_double(int(code, 16))
        assert got == v and math.copysign(1, got) == math.copysign(1, v), (code, expr, got)
        assert o.bf16_from_double(v) == int(code, 16), (code, expr)
    for expr, code in g["round"]:
        got = o.bf16_from_double(_eval(expr))
        assert got == int(code, 16), (expr, hex(got), code)


def pin_golden_e4m3(o):
    g = _read_golden("e4m3_ocp_points.txt")
    for code, expr in g["decode"]:
        v = _eval(expr)
        got = o.e4m3_to_double(int(code, 16))
        assert got == v and math.copysign(1, got) == math.copysign(1, v), (code, expr, got)
        assert o.e4m3_from_double(v) == int(code, 16), (code, expr)
    for expr, code in g["round"]:
        got = o.e4m3_from_double(_eval(expr))
        assert got == int(code, 16), (expr, hex(got), code)


def pin_e4m3_exhaustive(o):
    """All 254 finite codes decode to the bit-field value and encode back."""
    for c in range(256):
        if c & 0x7F == 0x7F:
            assert math.isnan(o.e4m3_to_double(c))
            continue
        v = bf.e4m3_value(c)
        assert Fraction(o.e4m3_to_double(c)) == v, hex(c)
        if c & 0x7F:
            assert o.e4m3_from_double(float(v)) == c, hex(c)


def pin_e4m3_rounding_bruteforce(o):
    """Random magnitudes (subnormal..beyond max) and every exact midpoint between
    adjacent codes, against the exhaustive nearest-code search."""
    rng = np.random.default_rng(11)
    xs = list(np.exp2(rng.uniform(-12, 10, 3000)) * rng.choice([-1.0, 1.0], 3000))
    pos = [bf.e4m3_value(c) for c in range(0x00, 0x7F)]
    for a, b in zip(pos[:-1], pos[1:]):
        m = (a + b) / 2
        xs += [float(m), float(-m), float(m + Fraction(1, 2 ** 40)), float(m - Fraction(1, 2 ** 40))]
    for x in xs:
        want = bf.nearest_e4m3_satfinite(Fraction(float(x)))
        got = o.e4m3_from_double(float(x))
        assert got == want, (x, hex(got), hex(want))


def pin_e4m3_vs_torch(o):
    """torch's float8_e4m3fn cast (round to nearest even) agrees inside +-448."""
    rng = np.random.default_rng(12)
    v = (np.exp2(rng.uniform(-11, 8.8, 4000)) * rng.choice([-1.0, 1.0], 4000)).astype(np.float32)
    v = np.clip(v, -448, 448)
    codes = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for x, c in zip(v, codes):
        assert o.e4m3_from_double(float(x)) == int(c), (float(x), int(c))


def pin_bf16_vs_torch(o):
    """torch's bf16 cast of float32 (RNE) agrees, normals and subnormals."""
    rng = np.random.default_rng(13)
    v = (np.exp2(rng.uniform(-140, 127, 5000)) * rng.choice([-1.0, 1.0], 5000)).astype(np.float32)
    v = np.concatenate([v, rng.standard_normal(2000).astype(np.float32)])
    codes = _bits(v)
    for x, c in zip(v, codes):
        assert o.bf16_from_double(float(x)) == int(c), (float(x), hex(int(c)))


def pin_bf16_rounding_bruteforce(o):
    """Doubles at and around midpoints of adjacent bf16 codes vs exhaustive search."""
    rng = np.random.default_rng(14)
    codes = rng.integers(0x0001, 0x7F7F, 400)
    for c in codes:
        a, b = bf.bf16_value(int(c)), bf.bf16_value(int(c) + 1)
        m = (a + b) / 2
        for x in (m, m + (b - a) / 1024, m - (b - a) / 1024, -m):
            assert o.bf16_from_double(float(x)) == bf.nearest_bf16(Fraction(float(x))), (hex(int(c)), float(x))


# ----------------------------------------------------------- residual_out --

def pin_residual_integer_sums(o):
    """Small-integer bf16 inputs: every fp32 partial sum is exact, so residual_out is
    the integer sum, and any permutation of the partials gives the same bits."""
    rng = np.random.default_rng(21)
    R, T, H = 5, 3, 64
    p = rng.integers(-20, 21, (R, T, H)).astype(np.float32)
    res = rng.integers(-20, 21, (T, H)).astype(np.float32)
    gamma = _bits(np.ones(H))
    ro, _ = o.reduce_rmsnorm(_bits(p), _bits(res), gamma, 1e-6, want_y=False)
    assert np.array_equal(ro, _bits(p.sum(0) + res))
    ro2, _ = o.reduce_rmsnorm(_bits(p[::-1].copy()), _bits(res), gamma, 1e-6, want_y=False)
    assert np.array_equal(ro, ro2)


def pin_residual_rank_order(o):
    """fp32 sum in rank order 0..R-1: [1, 2^-8, 2^-24, 2^-24] gives 1 + 2^-8 (each
    2^-24 is a tie that rounds back to even), which rounds to bf16 1.0; the reverse
    order builds 1 + 2^-8 + 2^-23 exactly, which rounds up to 1 + 2^-7.  A double
    accumulator would also give 1 + 2^-7."""
    H = 8
    vals = [1.0, 2.0 ** -8, 2.0 ** -24, 2.0 ** -24]
    p = np.stack([np.full((1, H), v, np.float32) for v in vals])
    gamma = _bits(np.ones(H))
    ro, _ = o.reduce_rmsnorm(_bits(p), None, gamma, 1e-6, want_y=False)
    assert np.all(ro == 0x3F80), hex(int(ro[0, 0]))
    ro, _ = o.reduce_rmsnorm(_bits(p[::-1].copy()), None, gamma, 1e-6, want_y=False)
    assert np.all(ro == 0x3F81), hex(int(ro[0, 0]))


def pin_residual_added_last(o):
    """Partials [2^-8, 2^-24, 2^-24] then residual 1: the partials sum exactly to
    2^-8 + 2^-23, so the result is 1 + 2^-8 + 2^-23 -> bf16 1 + 2^-7.  Adding the
    residual first would lose both 2^-24 terms and round to 1.0."""
    H = 8
    vals = [2.0 ** -8, 2.0 ** -24, 2.0 ** -24]
    p = np.stack([np.full((1, H), v, np.float32) for v in vals])
    ro, _ = o.reduce_rmsnorm(_bits(p), _bits(np.ones((1, H))), _bits(np.ones(H)), 1e-6, want_y=False)
    assert np.all(ro == 0x3F81), hex(int(ro[0, 0]))


def pin_residual_special_cases(o):
    """NULL residual is a zero residual; R=1 with a zero partial returns the residual."""
    inp = make_inputs(3, 4, 96, seed=22)
    zero = np.zeros_like(inp.residual)
    a, ya = o.reduce_rmsnorm(inp.partials, None, inp.gamma, inp.eps)
    b, yb = o.reduce_rmsnorm(inp.partials, zero, inp.gamma, inp.eps)
    assert np.array_equal(a, b) and np.array_equal(ya, yb)
    p0 = np.zeros((1, 4, 96), np.uint16)
    c, _ = o.reduce_rmsnorm(p0, inp.residual, inp.gamma, inp.eps)
    assert np.array_equal(c, inp.residual)


# ---------------------------------------------------------------------- y --

def _exact_rms_y(x: Fraction, xs_sq_mean: Fraction, g: Fraction) -> int:
    with localcontext() as ctx:
        ctx.prec = 60
        m = Decimal(xs_sq_mean.numerator) / Decimal(xs_sq_mean.denominator)
        prod = x * g
        v = Decimal(prod.numerator) / Decimal(prod.denominator) / m.sqrt()
    return bf.nearest_bf16(Fraction(v))


def pin_y_constant_row(o):
    """A constant row c: y[h] = bf16(gamma[h] * c / sqrt(c^2 + eps)).  Includes rows
    small enough that eps is comparable to c^2, and negative rows."""
    H = 256
    rng = np.random.default_rng(31)
    gamma = _bits(rng.uniform(0.5, 1.5, H))
    eps = 1e-6
    eps32 = Fraction(float(np.float32(eps)))
    for c in (1.0, -3.5, 2.0 ** -10, 0.0009765625 * 1.5, 100.0, -2.0 ** -12):
        res = _bits(np.full((1, H), c, np.float32))
        p = np.zeros((1, 1, H), np.uint16)
        ro, y = o.reduce_rmsnorm(p, res, gamma, eps)
        cf = bf.bf16_value(int(ro[0, 0]))
        for h in range(H):
            want = _exact_rms_y(cf, cf * cf + eps32, bf.bf16_value(int(gamma[h])))
            assert int(y[0, h]) == want, (c, h, hex(int(y[0, h])), hex(want))


def pin_y_scale_invariance(o):
    """eps = 0: scaling every input by 2^k scales every fp32 sum and residual_out
    exactly by 2^k, and y is bit-identical."""
    inp = make_inputs(2, 3, 512, seed=32)
    _, y0 = o.reduce_rmsnorm(inp.partials, inp.residual, inp.gamma, 0.0)
    for k in (-6, 3, 9):
        p = _bits(bf16_bits_to_f32(inp.partials) * np.float32(2.0 ** k))
        r = _bits(bf16_bits_to_f32(inp.residual) * np.float32(2.0 ** k))
        _, yk = o.reduce_rmsnorm(p, r, inp.gamma, 0.0)
        assert np.array_equal(y0, yk), k


def pin_y_unit_rms(o):
    """gamma = 1, eps = 0: mean(y^2) = 1 up to the bf16 rounding of y."""
    inp = make_inputs(4, 6, 1024, seed=33)
    _, y = o.reduce_rmsnorm(inp.partials, inp.residual, _bits(np.ones(1024)), 0.0)
    yf = bf16_bits_to_f32(y).astype(np.float64)
    ms = (yf ** 2).mean(1)
    assert np.all(np.abs(ms - 1.0) < 2.0 ** -8), ms


def pin_y_vs_torch_rms_norm(o):
    """torch.nn.functional.rms_norm in fp64 over f32(residual_out): within 1 bf16 ulp
    (torch's fp64 -> bf16 cast goes through fp32, so ties may differ by one)."""
    inp = make_inputs(3, 5, 768, seed=34, partial_std=0.5)
    ro, y = o.reduce_rmsnorm(inp.partials, inp.residual, inp.gamma, inp.eps)
    x = torch.from_numpy(bf16_bits_to_f32(ro).astype(np.float64))
    g = torch.from_numpy(bf16_bits_to_f32(inp.gamma).astype(np.float64))
    eps32 = float(np.float32(inp.eps))
    ref = torch.nn.functional.rms_norm(x, (768,), weight=g, eps=eps32)
    ref_bits = ref.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    d = np.abs(_ordered(ref_bits) - _ordered(y))
    assert d.max() <= 1, int(d.max())
    assert (d > 0).mean() < 1e-3


def pin_bruteforce_tiny(o):
    """Exact rational brute force (numpy fp32 adds, decimal norm, exhaustive bf16
    search) on tiny shapes: residual_out and y bit-identical."""
    for seed, (R, T, H) in enumerate([(1, 1, 8), (2, 3, 16), (3, 2, 16), (2, 2, 24), (3, 3, 8)]):
        inp = make_inputs(R, T, H, seed=100 + seed)
        res = inp.residual if seed % 2 == 0 else None
        ro, y = o.reduce_rmsnorm(inp.partials, res, inp.gamma, inp.eps)
        bro, by = bf.reduce_rmsnorm(inp.partials, res, inp.gamma, inp.eps)
        assert np.array_equal(ro, bro), (R, T, H)
        assert np.array_equal(y, by), (R, T, H)


# ------------------------------------------------------------------ quant --

def _random_y(T, H, seed):
    rng = np.random.default_rng(seed)
    y = rng.standard_normal((T, H)).astype(np.float32) * np.exp2(rng.uniform(-3, 3, (T, 1))).astype(np.float32)
    return _bits(y)


def pin_quant_max_448(o):
    """Every group with a nonzero absmax decodes to max |q| = 448 exactly."""
    y = _random_y(8, 1024, 41)
    q, s = o.quant_per_group(y, 128)
    dec = np.vectorize(o.e4m3_to_double)(q).reshape(8, 8, 128)
    assert np.all(np.abs(dec).max(-1) == 448.0)
    assert np.all(s > 0)


def pin_quant_error_bound(o):
    """|decode(q) - fl32(y/s)| <= half an e4m3 ulp at that magnitude (RNE), with the
    subnormal spacing 2^-9 below 2^-6."""
    y = _random_y(4, 512, 42)
    q, s = o.quant_per_group(y, 128)
    yf = bf16_bits_to_f32(y).reshape(4, 4, 128)
    v = (yf / s[:, :, None]).astype(np.float32).astype(np.float64)
    dec = np.vectorize(o.e4m3_to_double)(q).reshape(4, 4, 128)
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -6)))
    half_ulp = np.exp2(e - 3) / 2
    assert np.all(np.abs(dec - v) <= half_ulp)


def pin_quant_bruteforce(o):
    """Scales by numpy fp32 division and codes by exhaustive nearest-code search."""
    y = _random_y(2, 256, 43)
    q, s = o.quant_per_group(y, 128)
    bq, bs = bf.quant_per_group(y, 128)
    assert np.array_equal(s.view(np.uint32), bs.view(np.uint32))
    assert np.array_equal(q, bq)


def pin_quant_vs_torch(o):
    """torch: fp32 y / s then the float8_e4m3fn cast of the clamped quotient."""
    y = _random_y(6, 768, 44)
    q, s = o.quant_per_group(y, 128)
    yt = torch.from_numpy(bf16_bits_to_f32(y)).view(6, 6, 128)
    st = torch.from_numpy(s).view(6, 6, 1)
    qt = (yt / st).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).view(6, 768).numpy()
    assert np.array_equal(q, qt)


def pin_quant_degenerate_groups(o):
    """An all-zero group gives s = 0 and q = 0; a group with one nonzero element
    gives that element +-448 and zeros elsewhere."""
    y = np.zeros((2, 256), np.float32)
    y[1, 130] = -0.75
    yb = _bits(y)
    q, s = o.quant_per_group(yb, 128)
    assert s[0, 0] == 0 and s[0, 1] == 0 and s[1, 0] == 0
    assert np.float32(s[1, 1]) == np.float32(np.float32(0.75) / np.float32(448))
    assert np.all(q[0] == 0) and np.all(q[1, :128] == 0)
    assert q[1, 130] == 0xFE
    assert np.all(np.delete(q[1, 128:], 2) == 0)


def pin_quant_outlier_groups(o):
    """A x50 outlier in one group lifts that group's scale about 50x and leaves the
    other groups of the row untouched (scales are per group, not per row)."""
    inp = make_inputs(2, 2, 512, seed=45)
    _, y, q0, s0 = o.reduce_rmsnorm_quant(inp.partials, inp.residual, inp.gamma, inp.eps)
    y2 = bf16_bits_to_f32(y).copy()
    y2[:, 200] = 50.0 * np.abs(y2[:, 128:256]).max(1)
    q, s = o.quant_per_group(_bits(y2), 128)
    assert np.array_equal(s[:, [0, 2, 3]], s0[:, [0, 2, 3]])
    assert np.all(s[:, 1] > 40 * s0[:, 1])


def pin_omp_matches_serial(o):
    """The row-parallel build computes each row exactly as the serial loop."""
    inp = make_inputs(3, 37, 384, seed=46)
    a = o.reduce_rmsnorm_quant(inp.partials, inp.residual, inp.gamma, inp.eps, 128, threads=1)
    b = o.reduce_rmsnorm_quant(inp.partials, inp.residual, inp.gamma, inp.eps, 128, threads=4)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


# ------------------------------------------------------------------ MXFP4 --

def pin_golden_e2m1_e8m0(o):
    g = _read_golden("e2m1_e8m0_ocp_mx_points.txt")
    for code, expr in g["e2m1"]:
        v = _eval(expr)
        got = o.e2m1_to_double(int(code, 16))
        assert got == v and math.copysign(1, got) == math.copysign(1, v), (code, expr, got)
        assert o.e2m1_from_double(v) == int(code, 16), (code, expr)
    for expr, code in g["round"]:
        assert o.e2m1_from_double(_eval(expr)) == int(code, 16), (expr, code)
    for code, expr in g["e8m0"]:
        assert o.e8m0_to_double(int(code, 16)) == _eval(expr), (code, expr)


def pin_e2m1_rounding_bruteforce(o):
    """Random values and every midpoint of adjacent E2M1 codes vs exhaustive search."""
    rng = np.random.default_rng(51)
    xs = list(rng.uniform(-9, 9, 2000)) + list(np.exp2(rng.uniform(-6, 3.5, 1000)))
    pos = [bf.e2m1_value(c) for c in range(8)]
    for a, b in zip(pos[:-1], pos[1:]):
        m = (a + b) / 2
        xs += [float(m), float(-m), float(m) + 2 ** -30, float(m) - 2 ** -30]
    for x in xs:
        assert o.e2m1_from_double(float(x)) == bf.nearest_e2m1_satfinite(Fraction(float(x))), x


def _mx_block_y(amax_sig: float, e: int, n: int, seed: int):
    rng = np.random.default_rng(seed)
    y = (rng.uniform(-1, 1, (1, n)) * amax_sig * 2.0 ** e).astype(np.float32)
    y[0, 3] = amax_sig * 2.0 ** e
    return _bits(y)


def pin_mxfp4_shared_exponent_closed_form(o):
    """A block whose absmax is m * 2^e (1 <= m < 2) has scale code e - 2 + 127; its
    absmax element becomes 4 (m < 1.25 by RNE, ...) up to 6, and the dequantised
    absmax m * 2^e is met to within half an E2M1 step."""
    for m, code_max in ((1.0, 0x6), (1.25, 0x6), (1.5, 0x7), (1.75, 0x7), (1.2, 0x6), (1.3, 0x7)):
        for e in (-20, -3, 0, 5, 60):
            y = _mx_block_y(m, e, 32, seed=e + 100)
            q, sc = o.mxfp4(y)
            assert sc[0, 0] == e - 2 + 127, (m, e, sc[0, 0])
            c = (q[0, 1] >> 4) & 0xF        # element 3 is the high nibble of byte 1
            assert c == code_max, (m, e, hex(c))


def pin_mxfp4_all_zero_block(o):
    y = np.zeros((1, 64), np.uint16)
    y[0, 40] = _bits(np.array([0.75]))[0]
    q, sc = o.mxfp4(y)
    assert sc[0, 0] == 0 and np.all(q[0, :16] == 0)
    assert sc[0, 1] == -1 - 2 + 127 and ((q[0, 20] & 0xF) == 0x7)   # 0.75 / 2^-3 = 6


def pin_mxfp4_clamped_exponent(o):
    """A block of bf16 subnormals: floor(log2(absmax)) - 2 falls below E8M0's
    -127, so the scale code is 0 (2^-127) and the elements are y * 2^127:
    2^-130 becomes 0.125 -> 0 (nearest), 2^-129 becomes 0.25 -> 0 (the tie
    between 0 and 0.5 goes to the even code), 3 * 2^-130 becomes 0.375 -> 0.5."""
    y = np.zeros((1, 32), np.uint16)
    y[0, 0] = 0x0008          # 2^-130 (bf16 subnormal: 8 * 2^-133)
    y[0, 1] = 0x0010          # 2^-129
    y[0, 2] = 0x0018          # 3 * 2^-130
    y[0, 5] = 0x8018          # -3 * 2^-130
    q, sc = o.mxfp4(y)
    bq, bsc = bf.mxfp4(y)
    assert sc[0, 0] == 0 and bsc[0, 0] == 0
    assert np.array_equal(q, bq)
    assert (q[0, 0] & 0xF) == 0x0 and (q[0, 0] >> 4) == 0x0 and (q[0, 1] & 0xF) == 0x1 and (q[0, 2] >> 4) == 0x9


def pin_mxfp4_bruteforce(o):
    """Exact shared exponent and exhaustive-search codes on random blocks."""
    rng = np.random.default_rng(52)
    y = (rng.standard_normal((2, 128)) * np.exp2(rng.uniform(-8, 8, (2, 1)))).astype(np.float32)
    yb = _bits(y)
    q, sc = o.mxfp4(yb)
    bq, bsc = bf.mxfp4(yb)
    assert np.array_equal(sc, bsc) and np.array_equal(q, bq)


def pin_mxfp4_error_bound(o):
    """|dequant - y| <= half an E2M1 step at that magnitude, times the scale."""
    y = _random_y(3, 256, 53)
    q, sc = o.mxfp4(y)
    yf = bf16_bits_to_f32(y).astype(np.float64).reshape(3, 8, 32)
    X = np.exp2(sc.astype(np.float64) - 127)[:, :, None]
    codes = np.stack([q & 0xF, q >> 4], axis=-1).reshape(3, 256)
    dq = np.vectorize(o.e2m1_to_double)(codes).reshape(3, 8, 32) * X
    v = np.abs(yf / X)
    step = np.where(v < 1, 0.5, np.where(v < 2, 0.5, np.where(v < 4, 1.0, 2.0)))
    assert np.all(np.abs(dq - yf) <= np.maximum(step / 2 * X, np.where(v > 6, (v - 6) * X, 0)) + 1e-300)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
