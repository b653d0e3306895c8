"""The quantisers' fast code rounding, checked in exact arithmetic on the CPU.

The kernels take a code as clamp(rint(u - 1.5 * 2^23), 0, 2^b - 1) read from the bit pattern of
u = fl(a * rs + 1.5 * 2^23), where a = fl(x - z) and rs = fl(1 / s), and flag the value for the
exact division when d = fl(a * rs - rint) lies within 1e-5 of +-1/2. The format defines the code as
clamp(rint_half_even(fl(a / s)), 0, 2^b - 1). Here each float32 step is evaluated on exact
rationals and rounded once to float32 (ties to even), and every value the fast path does not flag
must get the defined code, with the quotient from numpy's IEEE float32 division.
"""
from fractions import Fraction as F

import numpy as np
import pytest

MAGIC = F(12582912)            # 1.5 * 2^23
MAGIC_BITS = 0x4B400000
GUARD = F(float(np.float32(0.5 - 1e-5)))


def rn32(x: F) -> F:
    """x rounded to the nearest float32, ties to even (no overflow in these cases)."""
    if x == 0:
        return F(0)
    sign = -1 if x < 0 else 1
    x = abs(x)
    e = x.numerator.bit_length() - x.denominator.bit_length()
    while F(2) ** e > x:
        e -= 1
    while F(2) ** (e + 1) <= x:
        e += 1
    e = max(e, -126)
    q = x / F(2) ** (e - 23)
    n = q.numerator // q.denominator
    r = q - n
    if r > F(1, 2) or (r == F(1, 2) and n % 2 == 1):
        n += 1
    return sign * F(n) * F(2) ** (e - 23)


def f32_bits(v: F) -> int:
    return int(np.array([float(v)], dtype=np.float32).view(np.int32)[0])


def fast_code(x: F, z: F, rs: F, bits: int):
    qmax = (1 << bits) - 1
    a = rn32(x - z)
    u = rn32(a * rs + MAGIC)
    tn = rn32(MAGIC - u)
    d = rn32(a * rs + tn)
    code = min(max(f32_bits(u), MAGIC_BITS), MAGIC_BITS + qmax) - MAGIC_BITS
    return code, abs(d) > GUARD


def defined_code(x: np.float32, z: np.float32, s: np.float32, bits: int) -> int:
    q = np.float32(np.float32(x - z) / s)
    return int(np.clip(np.rint(q), 0, (1 << bits) - 1))


def groups(bits, rng):
    """bf16-valued groups: normal, wide-range, offset and tie-heavy (exact half-integer quotients)."""
    qmax = (1 << bits) - 1
    out = []
    for kind in range(4):
        for _ in range(10):
            if kind == 0:
                x = rng.standard_normal(32)
            elif kind == 1:
                x = rng.standard_normal(32) * 10.0 ** rng.integers(-6, 4)
            elif kind == 2:
                x = 1000 + rng.standard_normal(32)
            else:
                x = rng.integers(0, 2 * qmax + 1, 32) / 2 * 2.0 ** int(rng.integers(-8, 8))
            x = np.asarray(x, dtype=np.float32)
            # round to bf16 (keep the top 16 bits, nearest even)
            u = x.view(np.uint32).astype(np.uint64)
            u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
            out.append(u.astype(np.uint32).view(np.float32))
    return out


@pytest.mark.parametrize("bits", [2, 4])
def test_fast_rounding_matches_the_defined_code(bits):
    rng = np.random.default_rng(7 + bits)
    qmax = np.float32((1 << bits) - 1)
    checked = flagged = 0
    for x in groups(bits, rng):
        mn, mx = x.min(), x.max()
        s = np.float32(np.float16(np.float32(mx - mn) / qmax))
        z = np.float32(np.float16(mn))
        if s == 0:
            continue
        rs = rn32(1 / F(float(s)))
        for xi in x:
            code, near = fast_code(F(float(xi)), F(float(z)), rs, bits)
            if near:
                flagged += 1
                continue
            assert code == defined_code(xi, z, s, bits), (float(xi), float(z), float(s))
            checked += 1
    assert checked > 1000 and flagged > 0  # the tie-heavy groups reach the exact path


def test_exact_tie_is_flagged_and_clamped_region_agrees():
    # (x - z) / s = 1.5 exactly: the product lands on the tie and must go to the exact division
    code, near = fast_code(F(3, 4), F(0), rn32(1 / F(1, 2)), 2)
    assert near
    # far outside the code range on either side the clamp decides, whatever the rounding
    for v, want in ((F(1000), 3), (F(-1000), 0), (F(4), 3), (F(-2), 0)):
        code, near = fast_code(v, F(0), F(1), 2)
        assert code == want and not near
