"""Pins of the OS II-fast / OS II-accu range estimation in the oracle ([Ozaki II, §9]).

The pages only say that fast uses a cheap (Cauchy-Schwarz) bound of c_max and accu
an extra low-precision GEMM, and that both must keep the CRT result unique
(c_max >= max_ij (|A'||B'|)_ij, c_max <= M/2 - 1, [Ozaki II, §5]).  These tests pin
the oracle's reading to what that fixes, independently of its own code:

* validity: the exact max_ij (|A'||B'|)_ij never exceeds M/2 - 1 (big integers);
* tightness: on inputs where every bound is attained the limit is reached to
  within one bit, so an exponent one too large breaks validity;
* the norm exponent bounds the exact 2-norm (Fractions) and is at most 2 above it;
* the accu magnitudes are the ceiling of |x| 2^(b - E) (Fractions);
* the §9 accuracy claim: on wide exponent distributions accu and fast beat the
  uniform estimate;
* planted mistakes in these functions are caught by one of the above.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

from fp64_gemm_emulation_gb300.inputs import hpl_like, special_matrix
from oracle import ozaki2 as O


def exact_abs_product_max(A, B, s, scaling):
    """max_ij sum_k |A'_ik| |B'_kj| with the oracle's own scaling, in Python integers."""
    cc, k, EA, EB, d, e, Ap, Bp = O.prepare(A, B, s, scaling=scaling)
    absA = np.abs(Ap.astype(object))
    absB = np.abs(Bp.astype(object))
    return int(np.dot(absA, absB).max(initial=0)), cc.M


def frac_norm2_sq(row):
    return sum((Fraction(float(v)) ** 2 for v in row), Fraction(0))


def frac_ceil_log2(x: Fraction) -> int:
    c = 0
    while Fraction(2) ** c < x:
        c += 1
    while Fraction(2) ** (c - 1) >= x:
        c -= 1
    return c


# ------------------------------------------------------------------ parameters
@pytest.mark.parametrize("s", [2, 3, 8, 14, 16, 20])
def test_half_range_and_kappa(s):
    M = math.prod(O.greedy_moduli(s))
    L = O.half_range_log2(M)
    assert Fraction(2) ** L <= Fraction(M, 2) - 1 < Fraction(2) ** (L + 1)
    kap = O.choose_k(M, 1)
    assert 2 * kap <= L < 2 * kap + 2


def test_ceil_log2_int():
    for x in range(1, 3000):
        assert O.ceil_log2_int(x) == frac_ceil_log2(Fraction(x))


def test_accu_bits_table():
    assert O.accu_bits(1) == 7
    assert O.accu_bits(1024) == 7          # 1024 * 4^7 = 2^24
    assert O.accu_bits(1025) == 6
    assert O.accu_bits(4096) == 6
    assert O.accu_bits(16384) == 5
    assert O.accu_bits(262144) == 3
    assert O.accu_bits(2**24) == 0
    for q in (1, 5, 1000, 70000, 2**20 + 1):
        b = O.accu_bits(q)
        assert q * 4**b <= 2**24 and (b == 7 or q * 4 ** (b + 1) > 2**24)
    with pytest.raises(ValueError):
        O.accu_bits(2**24 + 1)


# ------------------------------------------------------------------ OS II-fast norm exponent
def _norm_rows():
    rng = np.random.default_rng(5)
    rows = [
        np.array([3.0]),
        np.array([2.0**-1074, 0.0, -(2.0**-1073)]),          # subnormals only
        np.array([1.0] + [2.0**-17] * 1000),                 # many entries below 2^-G of the max
        np.full(64, -(2.0**10)),                             # equal powers of two (q = 4^3)
        np.array([2.0**900, 2.0**-900, 1.0]),
        (rng.random(333) - 0.5) * np.exp(4.0 * rng.standard_normal(333)),
        (rng.random(1000) - 0.5),
        np.array([0.75, -0.75, 0.75]),
    ]
    return rows


def test_norm_exponent_bounds_the_exact_norm():
    for row in _norm_rows():
        t = O.norm_exponents(row.reshape(1, -1))[0]
        nsq = frac_norm2_sq(row)
        assert Fraction(2) ** (2 * t) >= nsq                         # 2^t >= ||x||_2
        assert t <= math.ceil(frac_ceil_log2(nsq) / 2) + 2           # and not far above it


def test_norm_exponent_closed_forms():
    # a single nonzero: the norm is the maximum
    for v in (1.0, -3.0, 2.0**-1070, 5e300):
        assert O.norm_exponents(np.array([[0.0, v, 0.0]]))[0] == O.ceil_log2_abs(v)
    # q = 4^j equal powers of two 2^c: ||x|| = 2^(c + j) exactly
    for j, c in ((0, 0), (1, 5), (3, -7), (5, 100)):
        assert O.norm_exponents(np.full((1, 4**j), 2.0**c))[0] == c + j


def test_norm_exponent_special_rows_keep_codes():
    X = np.array([[0.0, 0.0], [1.0, np.nan], [np.inf, 1.0], [0.5, 0.25]])
    t = O.norm_exponents(X)
    assert t[0] is O.ZERO_ROW and t[1] == "nan" and t[2] == "nan" and t[3] == 0


# ------------------------------------------------------------------ OS II-accu magnitudes
def test_magnitude_bounds_are_ceilings():
    rng = np.random.default_rng(9)
    X = (rng.random((6, 50)) - 0.5) * np.exp(6.0 * rng.standard_normal((6, 50)))
    X[1, :] = 0.0
    X[2, 3] = 2.0**-1074
    X[3, :] = 2.0**-1000
    X[3, 0] = 2.0**40
    X[4, :] = np.linspace(-1, 1, 50)
    E = O.row_exponents(X)
    for b in (0, 3, 5, 7):
        Xh = O.magnitude_bounds(X, E, b)
        for i in range(X.shape[0]):
            for j in range(X.shape[1]):
                if E[i] is O.ZERO_ROW:
                    assert Xh[i, j] == 0
                    continue
                want = math.ceil(Fraction(abs(float(X[i, j]))) * Fraction(2) ** (b - E[i]))
                assert Xh[i, j] == want
                assert 0 <= Xh[i, j] <= 2**b


# ------------------------------------------------------------------ validity and tightness
RANGE_CASES = [
    ("hpl", 0.0), ("hpl", 0.5), ("hpl", 2.0), ("hpl", 4.0),
    ("zero_rows", None), ("subnormal", None), ("pow2", None), ("ints", None),
]


def _range_inputs(kind, phi, m=9, n=7, q=60, seed=3):
    if kind == "hpl":
        return hpl_like(m, n, q, phi=phi, seed=seed)
    return special_matrix(kind, m, q, seed=seed), special_matrix(kind, q, n, seed=seed + 1)


@pytest.mark.parametrize("scaling", ["fast", "accu", "uniform"])
@pytest.mark.parametrize("kind,phi", RANGE_CASES)
@pytest.mark.parametrize("s", [3, 8, 14])
def test_crt_range_is_never_exceeded(scaling, kind, phi, s):
    A, B = _range_inputs(kind, phi)
    cmax, M = exact_abs_product_max(A, B, s, scaling)
    assert 2 * cmax <= M - 2  # (|A'||B'|)_ij <= M/2 - 1


@pytest.mark.parametrize("s", [3, 8, 14, 20])
def test_fast_attains_its_bound_on_equal_powers_of_two(s):
    # every |a| = 2^3, q = 64 = 4^3: ||A'_i|| ||B'_j|| = (A'B')_ij exactly = 2^(2 kappa)
    A = np.full((3, 64), 8.0)
    B = np.full((64, 2), -0.25)
    cmax, M = exact_abs_product_max(A, B, s, "fast")
    assert cmax == 2 ** (2 * O.choose_k(M, 1))
    assert 2 * cmax <= M - 2 < 4 * 2 * cmax  # one more bit per side would break uniqueness


@pytest.mark.parametrize("s", [3, 8, 14, 20])
@pytest.mark.parametrize("q", [64, 1024, 4096])
def test_accu_reaches_the_limit_within_one_bit(s, q):
    # every |a| a power of two and equal: the magnitudes and C^ carry no rounding
    A = np.full((3, q), 2.0**-5)
    B = np.full((q, 4), 2.0**7)
    cmax, M = exact_abs_product_max(A, B, s, "accu")
    L = O.half_range_log2(M)
    assert 2**(L - 1) <= cmax <= 2**L


def test_scalings_share_codes_for_special_rows():
    A, B = hpl_like(6, 5, 30, seed=4)
    A[1] = 0.0
    A[2, 3] = np.nan
    B[:, 4] = 0.0
    for sc in ("fast", "accu"):
        k, EA, EB = O.scaling_exponents(A, B, math.prod(O.greedy_moduli(14)), sc)
        assert EA[1] is O.ZERO_ROW and EA[2] == "nan" and EB[4] is O.ZERO_ROW


# ------------------------------------------------------------------ method == definition
@pytest.mark.parametrize("scaling", ["fast", "accu"])
@pytest.mark.parametrize("m,n,k,s,phi,seed", [(9, 11, 40, 14, 0.5, 1), (5, 6, 300, 8, 4.0, 2),
                                              (7, 3, 17, 20, 2.0, 3), (4, 4, 2000, 14, 1.0, 4)])
def test_method_equals_definition(scaling, m, n, k, s, phi, seed):
    A, B = hpl_like(m, n, k, phi=phi, seed=seed)
    r = O.ozaki2_dgemm(A, B, s, scaling=scaling)
    D = O.direct_dgemm(A, B, s, scaling=scaling)
    assert np.array_equal(r.C.view(np.int64), D.view(np.int64))
    rows, cols = np.arange(m).repeat(n), np.tile(np.arange(n), m)
    E = O.direct_entries(A, B, s, rows, cols, scaling=scaling)
    assert np.array_equal(E.view(np.int64), r.C[rows, cols].view(np.int64))


def test_sampled_accu_exponents_equal_full_ones():
    A, B = hpl_like(30, 25, 500, phi=2.0, seed=8)
    A[3] = 0.0
    M = math.prod(O.greedy_moduli(14))
    kap, tA, tB = O.accu_exponents(A, B, M)[:3]
    kap2, sA, sB = O.accu_exponents_sampled(A, B, M, range(30), range(25))
    assert kap == kap2
    assert all(sA[i] == tA[i] for i in range(30)) and all(sB[j] == tB[j] for j in range(25))


# ------------------------------------------------------------------ the §9 accuracy claim
def _median_rel_error(A, B, C, samples):
    errs = []
    for i, j in samples:
        exact = sum((Fraction(float(a)) * Fraction(float(b)) for a, b in zip(A[i], B[:, j])), Fraction(0))
        scale = sum((abs(Fraction(float(a)) * Fraction(float(b))) for a, b in zip(A[i], B[:, j])), Fraction(0))
        errs.append(float(abs(Fraction(float(C[i, j])) - exact) / scale))
    return float(np.median(errs))


@pytest.mark.parametrize("phi", [2.0, 4.0])
@pytest.mark.parametrize("s", [8, 12])
def test_accu_and_fast_beat_uniform_on_wide_ranges(phi, s):
    A, B = hpl_like(24, 24, 256, phi=phi, seed=21)
    rng = np.random.default_rng(0)
    samples = list(zip(rng.integers(0, 24, 40), rng.integers(0, 24, 40)))
    err = {sc: _median_rel_error(A, B, O.ozaki2_dgemm(A, B, s, keep=False, scaling=sc).C, samples)
           for sc in O.SCALINGS}
    assert err["accu"] < err["uniform"]
    assert err["fast"] < err["uniform"]
    assert err["accu"] <= err["fast"]


# ------------------------------------------------------------------ planted mistakes
def _norm_without_guard(X):
    X = np.asarray(X, dtype=np.float64)
    out = []
    for i in range(X.shape[0]):
        row = X[i][X[i] != 0]
        c = O._ceil_log2_abs_array(row)
        cmax = int(c.max())
        S = sum(4 ** int(dv) for dv in c - cmax + O.NORM_GUARD if dv >= 0)  # tiny entries dropped
        out.append(cmax - O.NORM_GUARD + (O.ceil_log2_int(S) + 1) // 2)
    return out


def test_planted_norm_mistake_is_caught():
    row = np.array([1.0] + [2.0**-17] * 1000)
    t = _norm_without_guard(row.reshape(1, -1))[0]
    assert Fraction(2) ** (2 * t) < frac_norm2_sq(row)  # the validity pin fails


def test_planted_floor_in_magnitudes_is_caught(monkeypatch):
    orig = O.magnitude_bounds

    def floored(X, E, b):
        out = orig(X, E, b)
        X = np.asarray(X, dtype=np.float64)
        for i in range(X.shape[0]):
            if E[i] is O.ZERO_ROW or E[i] == "nan":
                continue
            for j in range(X.shape[1]):
                out[i, j] = math.floor(Fraction(abs(float(X[i, j]))) * Fraction(2) ** (b - E[i]))
        return out

    X = np.array([[1.0, 0.3, -0.7, 1e-9]])
    E = O.row_exponents(X)
    want = [math.ceil(Fraction(abs(float(v))) * Fraction(2) ** (5 - E[0])) for v in X[0]]
    assert list(orig(X, E, 5)[0]) == want
    monkeypatch.setattr(O, "magnitude_bounds", floored)
    assert list(O.magnitude_bounds(X, E, 5)[0]) != want


@pytest.mark.parametrize("slip", ["x_plus_one", "rho_min"])
def test_planted_accu_exponent_mistakes_break_the_range(slip, monkeypatch):
    orig = O.accu_exponents

    def mutated(A, B, M):
        kap, tA, tB, b, Ah, Bh, Ch = orig(A, B, M)
        if slip == "x_plus_one":
            tA = [t if (t is O.ZERO_ROW or t == "nan") else t - 1 for t in tA]
            tB = [t if (t is O.ZERO_ROW or t == "nan") else t - 1 for t in tB]
        else:  # the row bound taken from the smallest entry of the row of C^
            L = O.half_range_log2(M)
            EA = O.row_exponents(A)
            rho = np.maximum(Ch.min(axis=1), 1)
            tA = [kap - (L - O.ceil_log2_int(int(r))) // 2 + E - b for E, r in zip(EA, rho)]
        return kap, tA, tB, b, Ah, Bh, Ch

    monkeypatch.setattr(O, "accu_exponents", mutated)
    if slip == "x_plus_one":
        A, B = np.full((3, 64), 2.0**-5), np.full((64, 4), 2.0**7)
    else:  # a column of B with one large entry makes the rows of C^ very uneven
        A = np.full((3, 64), 2.0**-5)
        B = np.full((64, 4), 2.0**7)
        B[1:, 1] = 2.0**-20
    cmax, M = exact_abs_product_max(A, B, 14, "accu")
    assert 2 * cmax > M - 2
