"""The quant epilogue computes the group scale absmax / 448 as RN(absmax *
RN(1/448)) plus one FMA correction, and divides y by the group scale with one correctly rounded
reciprocal per group and one FMA correction step (Markstein's theorem) instead
of an IEEE divide per element.  This CPU test replays that sequence in exact
rational arithmetic for every bf16 significand of y against every significand
the scale s = RN(absmax / 448) can take (absmax is a bf16), and checks that it
always equals the correctly rounded quotient RN(y / s).  Powers of two scale
the operands exactly (the kernel takes this path only for s >= 2^-64, where no
intermediate underflows or overflows), so these pairs cover every case."""
import math
from fractions import Fraction as F


def rn32(x: F) -> F:
    """Round a rational to the nearest fp32 value, ties to even (normal range)."""
    if x == 0:
        return F(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    while F(2) ** e > a:
        e -= 1
    while F(2) ** (e + 1) <= a:
        e += 1
    ulp = F(2) ** (e - 23)
    n = a / ulp
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > F(1, 2) or (rem == F(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * ulp


def test_fma_corrected_quotient_is_correctly_rounded():
    y_sigs = [F(128 + m, 128) for m in range(128)]          # bf16 significands in [1, 2)
    s_sigs = set()
    for m in y_sigs:
        s = rn32(m / 448)
        while s >= 2:
            s /= 2
        while s < 1:
            s *= 2
        s_sigs.add(s)
    assert len(s_sigs) == 128
    for s in s_sigs:
        rs = rn32(1 / s)                                   # __frcp_rn
        for y in y_sigs:
            q0 = rn32(y * rs)                              # __fmul_rn
            rem = rn32(y - s * q0)                         # __fmaf_rn(-s, q0, y)
            q1 = rn32(q0 + rem * rs)                       # __fmaf_rn(rem, rs, q0)
            assert q1 == rn32(y / s), (y, s)


def test_fma_corrected_scale_is_correctly_rounded():
    """absmax / 448 for every bf16 significand of absmax (the binade of absmax
    relative to 448 only shifts the exponent)."""
    c = rn32(F(1, 448))                                     # the constant 1.0f / 448.0f
    for m in range(128):
        a = F(128 + m, 128)
        for shift in range(0, 10):
            aa = a * 2 ** shift
            q0 = rn32(aa * c)
            rem = rn32(aa - 448 * q0)
            assert rn32(q0 + rem * c) == rn32(aa / 448), (m, shift)


def test_group_absmax_from_x_gamma():
    """The row kernel takes an FP8 group's absmax of y from x*gamma before rstd
    is known: y = bf16(fl32(x*gamma * rstd)) with rstd > 0, so
    max |y| == bf16(fl32(max |x*gamma| * rstd)).  Checked on random groups,
    including ties, zeros, subnormal-scale and overflow-scale values."""
    import numpy as np
    import torch
    rng = np.random.default_rng(17)
    for trial in range(400):
        scale = float(2.0 ** rng.integers(-140, 120))
        xg = (rng.standard_normal(128) * scale).astype(np.float32)
        if trial % 7 == 0:
            xg[rng.integers(0, 128, 5)] = 0.0
        if trial % 11 == 0:
            xg[3] = -xg[9]                                  # a tie in magnitude
        rstd = np.float32(2.0 ** rng.uniform(-20, 20))
        y = torch.from_numpy(xg * rstd).to(torch.bfloat16).float().numpy()
        lhs = np.max(np.abs(y))
        rhs = torch.from_numpy(np.array([np.max(np.abs(xg)) * rstd], dtype=np.float32)).to(torch.bfloat16).float()
        assert lhs == rhs.item() or (np.isinf(lhs) and np.isinf(rhs.item())), (trial, lhs, rhs)
