"""Exact rational-arithmetic restatement of the quantizer and the GEMM, for pins.

Independent of the oracle: Python integers and fractions only, pure-Python loops,
so it is used on small cases. Rounding to binary32 and to E4M3FN is written out
from the definitions (round to nearest, ties to even).
"""
import math
from fractions import Fraction


def round_to_f32(v: Fraction) -> Fraction:
    """Round an exact rational to the nearest binary32 value, ties to even."""
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    # exponent E with 2^E <= a < 2^(E+1)
    E = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** E > a:
        E -= 1
    E = max(E, -126)                     # binary32 subnormals share exponent -126
    scaled = a * Fraction(2) ** (23 - E)  # significand in units of the last place
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * Fraction(n) * Fraction(2) ** (E - 23)


def e4m3_values():
    """The 127 non-negative finite E4M3FN values, index = code, from the field definition."""
    vals = []
    for code in range(0x7F):
        e, m = code >> 3, code & 7
        vals.append(Fraction(m, 512) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7))
    return vals


_TABLE = e4m3_values()


def round_to_e4m3_code(y: Fraction, negative_zero: bool = False) -> int:
    """Nearest E4M3FN code of an exact rational, ties to the even code, saturating."""
    neg = y < 0 or (y == 0 and negative_zero)
    a = abs(y)
    if a >= _TABLE[-1]:
        code = 0x7E
    else:
        hi = next(i for i, t in enumerate(_TABLE) if t >= a)
        if _TABLE[hi] == a:
            code = hi
        else:
            lo = hi - 1
            dl, dh = a - _TABLE[lo], _TABLE[hi] - a
            code = hi if (dh < dl or (dh == dl and hi % 2 == 0)) else lo
    return code | (0x80 if neg else 0)


def quantize_group(xs):
    """Exact restatement of one group: s = f32(amax/448), q = E4M3(f32(x/s))."""
    fx = [Fraction(float(x)) for x in xs]
    amax = max(abs(v) for v in fx)
    s = round_to_f32(amax / 448)
    if s == 0:
        return [0] * len(fx), 0.0
    codes = []
    for x, v in zip(xs, fx):
        y = round_to_f32(v / s)
        codes.append(round_to_e4m3_code(y, negative_zero=(y == 0 and math.copysign(1.0, float(x)) < 0)))
    return codes, float(s)


def decode(code: int) -> Fraction:
    v = _TABLE[code & 0x7F]
    return -v if code & 0x80 else v


def exact_gemm_entry(qa_row, sa_row, qb_row, sb_of_kblock):
    """sum_k dec(qa[k]) sa[k/128] dec(qb[k]) sb(k/128), exactly."""
    total = Fraction(0)
    for k, (ca, cb) in enumerate(zip(qa_row, qb_row)):
        kb = k // 128
        total += decode(int(ca)) * Fraction(float(sa_row[kb])) * decode(int(cb)) * Fraction(float(sb_of_kblock(kb)))
    return total
