"""The arithmetic claims the CUDA kernels rest on, checked exhaustively or exactly on the CPU.

These tests model the kernels' integer and FP32 steps in exact Python arithmetic. They
use no GPU and share no code with the kernels.

* Split, common case: a' < 2^52 is cut into four signed 13-bit limbs. For an odd modulus
  128 < m < 256, y = x0 + x1 (2^13 mod m) + x2 (2^26 mod m) + x3 (2^39 mod m) is formed in
  FP32. q = round(y * fl32(1/m)) then r = y - q m is the symmetric residue, for EVERY
  reachable y. For m = 256, q = round((y + 1/4) / 256) maps r into [-128, 127].
* Split, limb extraction: the bit operations that take an FP64 value and its row's shift
  base to the four limbs give trunc(|a| 2^(k_A - E)).
* CRT quotient estimate: z = Z/M - 2^-8 is taken in FP32 from the top words of Z, and
  Q = round(z). Q is round(Z/M) or one less, never more. Every element where Q is one less
  is flagged by |z - Q| > 63/128.
* Split, integer path: umulhi(ys, ceil(2^39 / m)) >> 7 is floor(ys / m) for every
  0 <= ys < 2^31 (both ends of every run of equal quotients are checked).
* GEMM epilogue: q = RN(v fl32(1/m)) keeps every remainder v - q m of an exact chunk sum
  below m in magnitude, and the 16-bit running lanes cannot overflow between reductions.
* CRT rounding: a 64-bit window is cut from the leading word down, with the words below
  kept only as a sticky bit, then rounded to nearest-even and assembled with the exponent.
  For normal results this equals the correctly rounded X 2^-D, at ties, near-ties, carries
  into the next binade and overflow.
"""
import math
import random
import struct
from fractions import Fraction as Fr

import numpy as np

from oracle import ozaki2 as O

MODULI = O.greedy_moduli(20)  # every list of <= 20 moduli is a prefix of this one


def test_greedy_moduli_have_the_shape_the_split_assumes():
    assert MODULI[0] == 256
    assert all(m % 2 == 1 and 128 < m < 256 for m in MODULI[1:])


def _f32_as_ratio(x: float):
    """x (an FP32 value) as n / 2^e with an integer n."""
    mant, ex = math.frexp(float(np.float32(x)))
    n, e = int(mant * (1 << 24)), 24 - ex
    assert Fr(n, 1 << e) == Fr(float(np.float32(x)))
    return n, e


def _round_half_even(num: np.ndarray, e: int) -> np.ndarray:
    fl = num >> e
    rem = num - (fl << e)
    half = 1 << (e - 1)
    return fl + (rem > half) + ((rem == half) & ((fl & 1) == 1))


def test_split_fp32_quotient_is_exact_for_every_reachable_value():
    ymax = 8191 * (1 + 3 * 254)  # |x_l| <= 8191, the constants 2^(13 l) mod m <= 254
    assert ymax < 1 << 23        # every partial sum is an exact FP32 integer
    chunk = np.arange(-(1 << 20), 1 << 20, dtype=np.int64)
    for m in MODULI[1:]:
        n, e = _f32_as_ratio(np.float32(1.0) / np.float32(m))  # the kernel's fl32(1/m)
        for base in range(-ymax - 1, ymax + 1, chunk.size):
            y = chunk + base
            y = y[(y >= -ymax) & (y <= ymax)]
            prod = y * n  # y fl(1/m) = prod / 2^e exactly
            rem = prod - ((prod >> e) << e)
            assert not np.any(rem == (1 << (e - 1))), m  # never a tie
            r = y - _round_half_even(prod, e) * m
            assert np.array_equal(r, ((y + m // 2) % m) - m // 2), m
    # m = 256: y = sign * x0, q = round((y + 1/4) / 256), i.e. (4y + 1) / 2^10
    y = np.arange(-8191, 8192, dtype=np.int64)
    num = 4 * y + 1
    assert not np.any(num - ((num >> 10) << 10) == 512)
    r = y - 256 * _round_half_even(num, 10)
    assert np.array_equal(r, ((y + 128) % 256) - 128)


def _bits(x: float) -> int:
    return struct.unpack("<Q", struct.pack("<d", x))[0]


def _limbs13(x: float, rb: int):
    """The kernel's limb extraction (None where it hands the value to the integer path)."""
    raw = _bits(x)
    lo, hi = raw & 0xFFFFFFFF, raw >> 32
    ex = (hi >> 20) & 0x7FF
    rs = rb - max(ex, 1)
    if rs < 1:
        return None
    hm = (hi & 0xFFFFF) | (0x100000 if ex else 0)
    sh = min(rs, 63)
    if sh < 32:
        ul, uh = (((hm << 32) | lo) >> sh) & 0xFFFFFFFF, hm >> sh
    else:
        ul, uh = hm >> (sh & 31), 0
    limbs = [ul & 0x1FFF, (ul >> 13) & 0x1FFF, (((uh << 32) | ul) >> 26) & 0x1FFF, uh >> 7]
    sign = -1 if hi >> 31 else 1
    return [sign * v for v in limbs]


def _ceil_log2(x: float) -> int:
    mant, e = math.frexp(abs(x))
    return e - 1 if mant == 0.5 else e


def test_split_limb_extraction_gives_the_scaled_truncation():
    rng = random.Random(7)
    fast = 0
    for _ in range(20000):
        pick = rng.random()
        if pick < 0.6:
            x = rng.uniform(-1, 1) * 2.0 ** rng.randint(-60, 60)
        elif pick < 0.7:
            x = rng.choice([0.0, -0.0])
        elif pick < 0.8:
            x = rng.uniform(-1, 1) * 2.0 ** rng.randint(-1074, -1000)  # subnormal range
        else:
            x = rng.choice([1.0, -1.0]) * 2.0 ** rng.randint(-1074, 1023)  # exact powers of two
        rowmax = abs(x) * 2.0 ** rng.randint(0, 70) if rng.random() < 0.7 else abs(x)
        if rowmax == 0 or math.isinf(rowmax):
            continue
        E, kA = _ceil_log2(rowmax), rng.randint(20, 51)
        limbs = _limbs13(x, 1075 + E - kA)
        if limbs is None:
            continue
        fast += 1
        assert all(abs(v) < 8192 for v in limbs)
        u = abs(Fr(x)) * Fr(2) ** (kA - E)
        expect = (u.numerator // u.denominator) * (-1 if x < 0 else 1)
        assert limbs[0] + limbs[1] * 2**13 + limbs[2] * 2**26 + limbs[3] * 2**39 == expect
    assert fast > 15000


def _rn32(q: Fr) -> Fr:
    """q rounded to the nearest FP32 value (ties to even), exactly."""
    if q == 0:
        return Fr(0)
    sign, a = (-1 if q < 0 else 1), abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fr(2) ** e > a:
        e -= 1
    ulp = Fr(2) ** (e - 23)
    n = a / ulp
    fl = n.numerator // n.denominator
    if n - fl > Fr(1, 2) or (n - fl == Fr(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * ulp


def test_crt_quotient_estimate_is_never_too_large_and_flags_every_shortfall():
    rng = random.Random(11)
    for s in range(2, 21):
        M = math.prod(MODULI[:s])
        NL = max(3, (M.bit_length() + 13 + 31) // 32)  # words of Z < 255 s M
        inv = _rn32(Fr(float(Fr(2 ** (32 * (NL - 1))) / Fr(float(M)))))
        zmax = 255 * s * M
        cases = [0, 1, M // 2, M // 2 + 1, zmax - 1]
        for _ in range(150):
            n = rng.randint(0, 255 * s - 1)
            off = rng.choice([0, 1, -1, 2, -2]) + rng.randint(-3, 3) * rng.choice([1, 2**20, 2**40, M // 1000, M // 256])
            cases += [n * M + M // 2 + off, rng.randint(0, zmax - 1)]
        for Z in cases:
            if not 0 <= Z < zmax:
                continue
            x = [(Z >> (32 * w)) & 0xFFFFFFFF for w in range(NL)]
            zs = _rn32(_rn32(Fr(x[NL - 2])) * Fr(1, 2**32) + _rn32(Fr(x[NL - 1])))
            if NL == 3:
                zs = _rn32(_rn32(Fr(x[0])) * _rn32(Fr(1, 2**64)) + zs)
            z = _rn32(zs * inv - Fr(1, 256))
            t = _rn32(z + 2**23)
            Q = int(t - 2**23)
            near = abs(z - (t - 2**23)) > Fr(63, 128)
            r = (Z + M // 2) // M
            assert Q in (r, r - 1), (s, Z)
            assert Q == r or near, (s, Z)


def _crt_round_model(X: int, nl: int, D: int):
    """The CRT kernel's rounding of a magnitude X (nl 32-bit words) times 2^-D: the 64-bit
    window from the leading word down, sticky bits below, RN-even, exponent assembly.
    Returns the IEEE bits, or None where the kernel hands over to its subnormal routine."""
    x = [(X >> (32 * w)) & 0xFFFFFFFF for w in range(nl)]
    hw, a, b, cw, below = 0, x[0], 0, 0, 0
    for l in range(1, nl):
        if x[l]:
            hw, a, b = l, x[l], x[l - 1]
            cw = x[l - 2] if l >= 2 else 0
            below = 0
            for q in range(l - 2):
                below |= x[q]
    if a == 0:
        return 0
    lz = 32 - a.bit_length()
    fsl = lambda lo, hi, sh: ((((hi << 32) | lo) << sh) >> 32) & 0xFFFFFFFF
    w1, w0 = fsl(b, a, lz), fsl(cw, b, lz)
    sticky = (((cw << lz) & 0xFFFFFFFF) | below | (w0 & 0x3FF)) != 0
    e_unb = 32 * hw + 31 - lz - D
    if e_unb < -1022:
        return None
    if e_unb > 1023:
        return 0x7FF0000000000000
    mlo = ((((w1 << 32) | w0) >> 11) & 0xFFFFFFFF)
    mhi = w1 >> 11
    inc = ((w0 >> 10) & 1) & (int(sticky) | (mlo & 1))
    m = ((mhi << 32) | mlo) + inc
    return (((e_unb + 1022) << 52) + m) & 0xFFFFFFFFFFFFFFFF


def test_crt_rounding_window_is_round_to_nearest_even():
    rng = random.Random(13)
    handed_over = 0
    for trial in range(20000):
        nl = rng.choice([3, 4, 5, 6])
        top = rng.randint(1, 32 * nl - 1)
        X = rng.getrandbits(top) | (1 << top)  # leading one at bit `top`
        X &= (1 << (32 * nl)) - 1
        shape = rng.random()
        if shape < 0.2 and top > 53:  # exact ties (half a last place, nothing below) and near-ties
            cut = top - 52 - rng.choice([0, 1])
            X = (X >> cut << cut) | (1 << (cut - 1))
        elif shape < 0.3:  # carries through a run of ones
            X = ((1 << (top + 1)) - 1) & ((1 << (32 * nl)) - 1)
        D = rng.randint(-1100, 1300)
        want_val = Fr(X) / Fr(2) ** D
        got = _crt_round_model(X, nl, D)
        if got is None:
            handed_over += 1
            assert want_val < Fr(2) ** -1022
            continue
        try:
            want = _bits(float(want_val))  # Python rounds a Fraction to nearest, ties to even
        except OverflowError:
            want = 0x7FF0000000000000
        assert got == want, (nl, top, D, hex(got), hex(want))
    assert handed_over > 100


def test_split_integer_barrett_step_is_exact_below_2_31():
    # The split's integer path (a' with a power-of-two factor, or above 2^52) takes
    # q = floor(ys / m) as umulhi(ys, ceil(2^39 / m)) >> 7 for 0 <= ys < 2^31.  The estimate
    # is monotone in ys, so it is exact on every [k m, k m + m - 1] when it is exact at both
    # ends; both ends are checked for every k.
    for m in MODULI:
        magic = -(-(1 << 39) // m)
        assert magic < 1 << 32
        k = np.arange(0, ((1 << 31) - 1) // m + 1, dtype=np.uint64)
        for ys in (k * np.uint64(m), k * np.uint64(m) + np.uint64(m - 1)):
            ys = ys[ys < np.uint64(1 << 31)]
            q = ((ys * np.uint64(magic)) >> np.uint64(32)) >> np.uint64(7)
            assert np.array_equal(q, ys // np.uint64(m)), m


def test_gemm_epilogue_quotient_keeps_every_remainder_below_m():
    # The GEMM epilogue takes each exact chunk sum v (|v| <= 2^24) to r = v - q m with
    # q = RN(v fl32(1/m)) (the 1.5 * 2^23 constant) and needs |r| < m.  q is monotone in v,
    # so q(k m) = k for every k with |k m| < 2^25 puts q between floor(v/m) and ceil(v/m)
    # for every v in range, hence |r| < m.
    for m in MODULI:
        n, e = _f32_as_ratio(np.float32(1.0) / np.float32(m))
        k = np.arange(-((1 << 25) // m), (1 << 25) // m + 1, dtype=np.int64)
        v = k * m
        q = _round_half_even(v * n, e)
        assert np.array_equal(q, k), m
    # the 16-bit running lanes: a lane below m gains less than 2m per chunk, 64 chunks
    # between reductions
    assert 256 + 64 * (2 * 256 - 1) < 1 << 16
