"""Pins for the Scheme II oracle: closed forms, invariants, brute force, page values.

Every check here is independent of the oracle's own code path: exact values are
recomputed by brute force with Python integers / fractions, and page-printed
values come from ``tests/golden``.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from fp64_gemm_emulation_gb300.inputs import hpl_like, special_matrix
from oracle import ozaki1, ozaki2

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append([int(x) for x in line.split()])
    return rows


# ---------------------------------------------------------------- brute force
def exact_scaled_int(x: float, shift: int = 1075) -> int:
    """x * 2^shift as an exact integer (every double is a multiple of 2^-1074)."""
    n, den = Fraction(float(x)).as_integer_ratio()
    assert (n << shift) % den == 0
    return (n << shift) // den


def exact_product_fraction(A, B):
    """AB exactly, as a matrix of Fractions (tiny inputs only)."""
    Ai = np.vectorize(exact_scaled_int, otypes=[object])(A)
    Bi = np.vectorize(exact_scaled_int, otypes=[object])(B)
    P = np.dot(Ai, Bi)
    return np.vectorize(lambda v: Fraction(v, 1 << 2150), otypes=[object])(P)


def brute_ceil_log2(x: float) -> int:
    fx = abs(Fraction(x))
    c = 0
    while Fraction(2) ** c < fx:
        c += 1
    while Fraction(2) ** (c - 1) >= fx:
        c -= 1
    return c


def brute_trunc(x: float, d: int) -> int:
    v = Fraction(x) * Fraction(2) ** d
    return math.trunc(v)


# ---------------------------------------------------------------- page values
def test_gemm_count_table_matches_pages():
    for s, count in _golden_rows("gemm_count_table.txt"):
        assert len(ozaki1.triangle_pairs(s)) == count
        assert all(i + j <= s + 1 for i, j in ozaki1.triangle_pairs(s))


def test_workload_moduli_are_the_greedy_list():
    (listed,) = _golden_rows("workload_moduli.txt")
    assert ozaki2.greedy_moduli(14) == listed
    assert ozaki2.greedy_moduli(16)[:14] == listed


@pytest.mark.parametrize("s", range(1, 21))
def test_moduli_pairwise_coprime_bounded_and_greedy(s):
    mods = ozaki2.greedy_moduli(s)
    assert len(mods) == s and all(2 <= m <= 256 for m in mods)
    assert mods == sorted(mods, reverse=True)
    for a in range(s):
        for b in range(a + 1, s):
            assert math.gcd(mods[a], mods[b]) == 1
    # greedy: every integer skipped between picks shares a factor with an earlier pick
    for idx in range(s):
        hi = 256 if idx == 0 else mods[idx - 1] - 1
        for cand in range(mods[idx] + 1, hi + 1):
            assert any(math.gcd(cand, p) > 1 for p in mods[:idx])


def test_int32_exactness_bound_of_section6():
    # [Ozaki II, §6]: residues in [-128, 127] make a length-q dot product at most
    # q * 2^14 in magnitude, which fits INT32 exactly for q < 2^17.
    assert (2**17 - 1) * 128 * 128 < 2**31
    assert not (2**17 * 128 * 128 < 2**31)


def test_log2M_is_linear_in_s_not_M():
    # [Ozaki II, §16]: the printed "M ~ s m_s" is an erratum; log2 M ~ s log2 m_s.
    for s in (8, 14, 16, 20):
        mods = ozaki2.greedy_moduli(s)
        M = ozaki2.crt_constants(mods).M
        assert s * math.log2(mods[-1]) <= math.log2(M) <= s * math.log2(mods[0])
        assert M > 1000 * s * mods[-1]


# ---------------------------------------------------------------- parameters
def test_crt_constants_brute_force():
    for s in (2, 5, 14, 20):
        cc = ozaki2.crt_constants(ozaki2.greedy_moduli(s))
        for t, m in enumerate(cc.moduli):
            w = cc.Mt[t] * cc.yt[t]
            for u, mu in enumerate(cc.moduli):
                assert w % mu == (1 if u == t else 0)


def test_crt_identity_random_big_integers():
    rng = np.random.default_rng(1)
    for s in (2, 7, 14, 16, 20):
        cc = ozaki2.crt_constants(ozaki2.greedy_moduli(s))
        for _ in range(200):
            x = int.from_bytes(rng.bytes(24), "little") % cc.M
            z = sum((x % m) * Mt * y for m, Mt, y in zip(cc.moduli, cc.Mt, cc.yt))
            assert z % cc.M == x


@pytest.mark.parametrize("s", [2, 4, 8, 10, 12, 14, 16, 20])
@pytest.mark.parametrize("q", [1, 7, 256, 4096, 8192, 16384, 2**17, 262144])
def test_choose_k_is_the_largest_valid_k(s, q):
    M = ozaki2.crt_constants(ozaki2.greedy_moduli(s)).M
    if 2 * q > M - 2:
        with pytest.raises(ValueError):
            ozaki2.choose_k(M, q)
        return
    k = ozaki2.choose_k(M, q)
    assert Fraction(q * 4**k) <= Fraction(M, 2) - 1          # c_max bound holds
    assert Fraction(q * 4 ** (k + 1)) > Fraction(M, 2) - 1   # and k + 1 breaks it
    # the pages' floating formula agrees wherever it is not on a boundary
    flt = math.floor(0.5 * math.log2((M / 2 - 1) / q))
    assert abs(flt - k) <= 1


def test_symmetric_residue_range_and_congruence():
    xs = np.arange(-70000, 70001, dtype=np.int64)
    for m in ozaki2.greedy_moduli(20):
        r = ozaki2.symmetric_residue(xs, m)
        assert r.min() >= -128 and r.max() <= 127
        assert np.all((xs - r) % m == 0)
        assert np.all(r >= -(m // 2)) and np.all(r <= (m - 1) // 2)
        # unique: every residue class hit exactly once in one period
        assert len(set(r[:m].tolist())) == m


# ---------------------------------------------------------------- scaling
def test_ceil_log2_matches_brute_force():
    rng = np.random.default_rng(2)
    vals = list(np.ldexp(rng.random(300) - 0.5, rng.integers(-1080, 1020, 300)))
    vals += [1.0, 2.0, 0.5, 3.0, 5e-324, 2.0**-1074 * 3, 2.0**-1022, 2.0**1023, -0.75, 1.5]
    for v in vals:
        if v == 0:
            continue
        assert ozaki2.ceil_log2_abs(float(v)) == brute_ceil_log2(float(v))


def test_scaled_trunc_vectorised_equals_scalar_and_fraction():
    rng = np.random.default_rng(3)
    X = np.ldexp(rng.random((20, 30)) - 0.5, rng.integers(-1070, 30, (20, 30)))
    X[0, :5] = [5e-324, -5e-324, 2.0**-1022, -1.0, 0.0]
    E = ozaki2.row_exponents(X)
    for k in (20, 47, 55):
        d = ozaki2.scale_exponents(E, k)
        V = ozaki2.scaled_trunc_matrix(X, d)
        for i in range(X.shape[0]):
            for j in range(X.shape[1]):
                assert int(V[i, j]) == brute_trunc(X[i, j], d[i]) == ozaki2.scaled_trunc(X[i, j], d[i])


@pytest.mark.parametrize("phi", [0.0, 0.5, 4.0])
def test_truncation_invariants(phi):
    A, _ = hpl_like(40, 1, 300, phi=phi, seed=4)
    k = 47
    E = ozaki2.row_exponents(A)
    d = ozaki2.scale_exponents(E, k)
    Ap = ozaki2.scaled_trunc_matrix(A, d)
    for i in range(A.shape[0]):
        row = [int(v) for v in Ap[i]]
        assert max(abs(v) for v in row) <= 2**k
        assert max(abs(v) for v in row) >= 2 ** (k - 1)   # the scale is the largest allowed
        for j, v in enumerate(row):
            err = Fraction(A[i, j]) - Fraction(v) * Fraction(2) ** (-d[i])
            assert abs(err) < Fraction(2) ** (-d[i])      # truncation loses < 1 unit
            assert v == 0 or (v > 0) == (A[i, j] > 0)      # toward zero keeps the sign


def test_residues_reconstruct_scaled_integers_by_crt():
    A, _ = hpl_like(16, 1, 64, phi=2.0, seed=5)
    for s in (8, 14, 16):
        mods = ozaki2.greedy_moduli(s)
        cc = ozaki2.crt_constants(mods)
        k = ozaki2.choose_k(cc.M, 64)
        d = ozaki2.scale_exponents(ozaki2.row_exponents(A), k)
        Ap = ozaki2.scaled_trunc_matrix(A, d)
        planes = ozaki2.residue_planes(Ap, mods)
        for i in range(A.shape[0]):
            for j in range(A.shape[1]):
                z = sum(int(planes[t, i, j]) % m * Mt * y
                        for t, (m, Mt, y) in enumerate(zip(mods, cc.Mt, cc.yt))) % cc.M
                z = z - cc.M if z > cc.M // 2 else z
                assert z == int(Ap[i, j])


# ---------------------------------------------------------------- whole method
CASES = [
    # (m, n, k, s, phi, seed)
    (5, 7, 9, 14, 0.5, 0),
    (13, 11, 40, 2, 0.5, 1),
    (8, 8, 64, 8, 0.0, 2),
    (9, 6, 33, 10, 2.0, 3),
    (12, 10, 50, 14, 4.0, 4),
    (7, 9, 31, 16, 0.5, 5),
    (6, 5, 17, 20, 1.0, 6),
]


@pytest.mark.parametrize("m,n,k,s,phi,seed", CASES)
def test_method_equals_definition(m, n, k, s, phi, seed):
    A, B = hpl_like(m, n, k, phi=phi, seed=seed)
    r = ozaki2.ozaki2_dgemm(A, B, s)
    # exact A'B' by brute force on Python integers
    direct = np.dot(r.Ap.astype(object), r.Bp.astype(object))
    assert np.array_equal(r.C3, direct)
    C2 = ozaki2.direct_dgemm(A, B, s)
    assert np.array_equal(r.C.view(np.int64), C2.view(np.int64))
    # sampled entries
    rows = [0, m - 1, m // 2]
    cols = [n - 1, 0, n // 2]
    E = ozaki2.direct_entries(A, B, s, rows, cols)
    assert np.array_equal(E.view(np.int64), r.C[rows, cols].view(np.int64))


@pytest.mark.parametrize("kind", ["zeros", "pow2", "subnormal", "zero_rows", "ints"])
def test_method_equals_definition_special_inputs(kind):
    A = special_matrix(kind, 9, 21, seed=7)
    B = special_matrix(kind, 21, 8, seed=8)
    r = ozaki2.ozaki2_dgemm(A, B, 14)
    C2 = ozaki2.direct_dgemm(A, B, 14)
    assert np.array_equal(r.C.view(np.int64), C2.view(np.int64))
    if kind == "zeros":
        assert np.all(r.C.view(np.int64) == 0)   # +0.0 everywhere
    if kind == "zero_rows":
        assert np.all(r.C[::3, :] == 0) and np.all(r.C[:, ::3] == 0)


def test_integer_inputs_give_the_exact_product():
    # special case that reduces to a textbook routine: small-integer matrices
    # are represented without truncation, so C is the exact integer product.
    A = special_matrix("ints", 20, 30, seed=9)
    B = special_matrix("ints", 30, 15, seed=10)
    r = ozaki2.ozaki2_dgemm(A, B, 6)
    assert r.k >= 6  # 2^k >= 20: no bit of |a| <= 20 is truncated
    expect = A.astype(np.int64) @ B.astype(np.int64)
    assert np.array_equal(r.C, expect.astype(np.float64))


def test_non_finite_rows_and_columns_give_nan():
    A, B = hpl_like(6, 5, 12, seed=11)
    A[2, 3] = np.inf
    B[4, 1] = np.nan
    r = ozaki2.ozaki2_dgemm(A, B, 14)
    assert np.all(np.isnan(r.C[2, :])) and np.all(np.isnan(r.C[:, 1]))
    mask = np.ones_like(r.C, dtype=bool)
    mask[2, :] = False
    mask[:, 1] = False
    assert np.all(np.isfinite(r.C[mask]))


@pytest.mark.parametrize("s,phi", [(8, 0.5), (14, 0.5), (14, 4.0), (20, 0.5)])
def test_error_within_truncation_bound(s, phi):
    A, B = hpl_like(6, 7, 45, phi=phi, seed=12)
    r = ozaki2.ozaki2_dgemm(A, B, s)
    exact = exact_product_fraction(A, B)
    for i in range(6):
        for j in range(7):
            scale = Fraction(2) ** (-(r.d[i] + r.e[j]))
            bound = sum(abs(int(r.Ap[i, kk])) + abs(int(r.Bp[kk, j])) + 1 for kk in range(45)) * scale
            c = Fraction(float(r.C[i, j]))
            half_ulp = Fraction(math.ulp(abs(float(r.C[i, j])))) / 2
            assert abs(c - exact[i, j]) <= bound + half_ulp
            # C is the rounding of C''' 2^-(d+e): at most half an ulp from it
            assert abs(c - Fraction(int(r.C3[i, j])) * scale) <= half_ulp


def test_accuracy_versus_moduli_count_matches_section10():
    # [Ozaki II, §10]: at phi = 0.5, about 14-15 moduli reach DGEMM-like
    # accuracy; fewer moduli are markedly less accurate.
    m, n, k = 16, 16, 512
    A, B = hpl_like(m, n, k, phi=0.5, seed=13)
    exact = exact_product_fraction(A, B)
    absAB = np.abs(A) @ np.abs(B)

    def err(C):
        return max(float(abs(Fraction(float(C[i, j])) - exact[i, j])) / absAB[i, j]
                   for i in range(m) for j in range(n))

    e_dgemm = err(A @ B)
    e = {s: err(ozaki2.ozaki2_dgemm(A, B, s, keep=False).C) for s in (8, 12, 14, 15, 16)}
    assert e[14] <= 16 * e_dgemm
    assert e[15] <= 2 * e_dgemm
    assert e[16] <= e_dgemm
    assert e[8] > 1e4 * e_dgemm
    assert e[8] > e[12] > e[14] > e[15] > e[16]


def test_zero_inner_dimension_is_rejected_by_parameter_choice():
    with pytest.raises(ValueError):
        ozaki2.choose_k(ozaki2.crt_constants(ozaki2.greedy_moduli(14)).M, 0)
