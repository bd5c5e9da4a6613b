"""Pins of the Scheme I EF / Hybrid variants in the oracle ([Ozaki notes]: group-wise
error-free accumulation, the Hybrid split), against what the pages and arithmetic fix:

* the INT32 sums of a batch of r products are exact, and r is the largest power of two
  for which the worst case still fits (brute force on the worst-case input);
* the groups cover the triangular products i + j <= s + 1 exactly once, in order;
* the bitmask split is |a| truncated to the grid 2^(e + 1 - s beta), cut into beta-bit
  fields (Fractions); the Hybrid split reconstructs A exactly with its residual and
  keeps every slice within 2^(beta - 1);
* on inputs the slices hold exactly, the result is the exact product;
* the error against the exact product stays inside the truncation plus dropped-term
  plus FP64-accumulation bound, and falls as s grows;
* planted mistakes are caught by one of the above.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

from fp64_gemm_emulation_gb300.inputs import hpl_like
from oracle import ozaki1 as O1


@pytest.mark.parametrize("q", [1, 2, 3, 255, 256, 4095, 4096, 4097, 16384, 65536, 2**17, 2**17 + 1, 262144])
def test_group_r_is_the_largest_exact_batch(q):
    beta = O1.beta_rn(q)
    r = O1.group_r(q, beta)
    worst = (2**beta - 1) ** 2 * q      # one product of two worst-case slice rows
    if r > 1:
        assert r & (r - 1) == 0          # a power of two
        assert r * worst < 2**31
        cq = math.ceil(math.log2(q)) if q > 1 else 0
        assert r * 2 ** (2 * beta + cq) <= 2**31 < 2 * r * 2 ** (2 * beta + cq)
    else:
        assert 2 ** (2 * beta + (math.ceil(math.log2(q)) if q > 1 else 0)) * 2 > 2**31 or worst < 2**31


@pytest.mark.parametrize("s", [1, 2, 5, 7, 9])
@pytest.mark.parametrize("r", [1, 2, 3, 32])
def test_group_batches_cover_the_triangle_in_order(s, r):
    batches = O1.group_batches(s, r)
    flat = [p for g, pairs in batches for p in pairs]
    assert sorted(flat) == sorted(O1.triangle_pairs(s))
    assert len(flat) == len(set(flat))
    gs = [g for g, _ in batches]
    assert gs == sorted(gs)
    for g, pairs in batches:
        assert 1 <= len(pairs) <= r and all(i + j == g for i, j in pairs)
        assert [i for i, _ in pairs] == sorted(i for i, _ in pairs)


def _split_inputs():
    rng = np.random.default_rng(3)
    X = (rng.random((6, 40)) - 0.5) * np.exp(3.0 * rng.standard_normal((6, 40)))
    X[1] = 0.0
    X[2, :5] = [2.0**-1074, -(2.0**-1060), 1.0, -1.0, 2.0**-30]
    X[3] = np.full(40, -(2.0 - 2.0**-52))
    X[4] = np.ldexp(1.0, rng.integers(-60, 60, 40)) * np.sign(rng.standard_normal(40))
    return X


@pytest.mark.parametrize("s,beta", [(1, 7), (3, 7), (7, 7), (9, 6), (20, 3)])
def test_bitmask_split_is_the_truncated_fields(s, beta):
    X = _split_inputs()
    S, E = O1.bitmask_split_rows(X, s, beta)
    assert np.abs(S).max() <= 2**beta - 1
    for i in range(X.shape[0]):
        row = X[i]
        if not row.any():
            assert not S[:, i].any()
            continue
        mx = max(abs(Fraction(float(v))) for v in row)
        e = 0  # floor(log2 mx) by brute force
        while Fraction(2) ** e > mx:
            e -= 1
        while Fraction(2) ** (e + 1) <= mx:
            e += 1
        grid = Fraction(2) ** (e + 1 - s * beta)
        for j, v in enumerate(row):
            a = Fraction(float(v))
            want = math.floor(abs(a) / grid) * grid * (1 if a >= 0 else -1)
            got = sum(Fraction(int(S[p, i, j])) * Fraction(2) ** int(E[p, i]) for p in range(s))
            assert got == want
            assert all(int(E[p, i]) == e + 1 - (p + 1) * beta for p in range(s))
        jmax = int(np.argmax(np.abs(row)))
        assert abs(int(S[0, i, jmax])) >= 2 ** (beta - 1)   # the leading bit sits in slice 1


@pytest.mark.parametrize("s,beta", [(1, 7), (4, 7), (7, 7), (9, 6)])
def test_hybrid_split_reconstructs_and_stays_in_range(s, beta):
    X = _split_inputs()
    X[2, :2] = 0.0  # keep the last grids normal
    S, E, R = O1.hybrid_split_rows(X, s, beta)
    assert np.abs(S).max() <= 2 ** (beta - 1)
    for i in range(X.shape[0]):
        for j in range(X.shape[1]):
            got = sum(Fraction(int(S[p, i, j])) * Fraction(2) ** int(E[p, i]) for p in range(s))
            assert got + Fraction(float(R[i, j])) == Fraction(float(X[i, j]))
        if X[i].any():
            # fixed grids mu'' 2^(-beta (p-1)); the residual is at most half the last grid
            assert all(int(E[p, i]) == int(E[0, i]) - beta * p for p in range(s))
            assert np.abs(R[i]).max() <= 2.0 ** (int(E[s - 1, i]) - 1)


@pytest.mark.parametrize("variant", ["ef", "hybrid"])
def test_exactly_representable_inputs_give_the_exact_product(variant):
    rng = np.random.default_rng(4)
    A = rng.integers(-100, 101, (7, 50)).astype(np.float64)
    B = rng.integers(-100, 101, (50, 6)).astype(np.float64)
    C = O1.ozaki1_dgemm_variant(A, B, 4, variant)[0]
    assert np.array_equal(C, A @ B)


def test_int32_batches_at_the_worst_case():
    # q = 2^17: beta = 7, r = 1; every slice field is 127, so one product sums to
    # q 127^2 < 2^31 and two would not fit
    q = 2**17
    A = np.full((2, q), 2.0 - 2.0**-52)
    B = np.full((q, 2), 2.0 - 2.0**-52)
    beta = O1.beta_rn(q)
    assert beta == 7 and O1.group_r(q, beta) == 1
    S, _ = O1.bitmask_split_rows(A[:, :8], 2, beta)
    assert (np.abs(S) == 127).all()
    assert q * 127**2 < 2**31 < 2 * q * 127**2
    O1.ozaki1_dgemm_variant(A, B, 2, "ef")  # the oracle's own INT32 assertion holds


def _exact_product(A, B, i, j):
    return sum((Fraction(float(a)) * Fraction(float(b)) for a, b in zip(A[i], B[:, j])), Fraction(0))


@pytest.mark.parametrize("variant", ["ef", "hybrid"])
@pytest.mark.parametrize("phi", [0.5, 2.0])
def test_error_within_the_bound_and_falling_with_s(variant, phi):
    A, B = hpl_like(6, 5, 64, phi=phi, seed=12)
    prev = None
    for s in (3, 5, 7, 9):
        C, SA, XA, SBt, XB, beta = O1.ozaki1_dgemm_variant(A, B, s, variant)
        worst = Fraction(0)
        for i in range(6):
            for j in range(5):
                exact = _exact_product(A, B, i, j)
                # kept terms, exactly; what the triangle drops; what the slices leave out
                kept = Fraction(0)
                for (p, q_) in O1.triangle_pairs(s):
                    kept += sum(Fraction(int(SA[p - 1, i, k]) * int(SBt[q_ - 1, j, k])) for k in range(64)) \
                        * Fraction(2) ** (int(XA[p - 1, i]) + int(XB[q_ - 1, j]))
                absterms = sum(abs(Fraction(float(a)) * Fraction(float(b))) for a, b in zip(A[i], B[:, j]))
                nb = len(O1.group_batches(s, O1.group_r(64, beta)))
                acc_bound = nb * Fraction(2) ** -53 * 2 * absterms         # FP64 additions of the batches
                assert abs(Fraction(float(C[i, j])) - kept) <= acc_bound
                err = abs(Fraction(float(C[i, j])) - exact) / absterms
                worst = max(worst, err)
        if prev is not None:
            assert worst <= prev
        prev = worst
    assert prev < Fraction(2) ** -40


def test_hybrid_is_at_least_as_accurate_as_ef():
    A, B = hpl_like(16, 16, 128, phi=1.0, seed=13)
    ex = np.array([[float(_exact_product(A, B, i, j)) for j in range(16)] for i in range(16)])
    scale = np.abs(A) @ np.abs(B)
    for s in (4, 6):
        e_ef = np.median(np.abs(O1.ozaki1_dgemm_variant(A, B, s, "ef")[0] - ex) / scale)
        e_h = np.median(np.abs(O1.ozaki1_dgemm_variant(A, B, s, "hybrid")[0] - ex) / scale)
        assert e_h <= e_ef  # round-to-nearest slices lose less than truncated ones


# ------------------------------------------------------------------ planted mistakes
def test_planted_ceil_exponent_in_the_bitmask_split_is_caught(monkeypatch):
    # taking ceil(log2 max) instead of floor for the leading bit pushes powers of two
    # out of the first field
    def ceil_rows(X):
        E, nz = O1._ceil_log2_rows(X)
        return np.where(nz, E, 0), nz

    monkeypatch.setattr(O1, "_floor_log2_rows", ceil_rows)
    X = np.array([[3.0, 1.0, -2.5]])
    S, E = O1.bitmask_split_rows(X, 3, 7)
    assert abs(int(S[0, 0, 0])) < 2**6  # the leading bit is no longer in slice 1


def test_planted_batch_size_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(O1, "group_r", lambda q, beta: 2)
    q = 2**17
    A = np.full((2, q), 2.0 - 2.0**-52)
    B = np.full((q, 2), 2.0 - 2.0**-52)
    with pytest.raises(AssertionError):
        O1.ozaki1_dgemm_variant(A, B, 2, "ef")  # two worst-case products overflow INT32


def test_planted_constant_sigma_in_hybrid_is_caught(monkeypatch):
    # without the 2^(-beta (p-1)) decay every later slice rounds to zero and the
    # error stops falling with s
    def no_decay(A, s, beta):
        R = np.array(A, dtype=np.float64, copy=True)
        E, nz = O1._ceil_log2_rows(R)
        slices = np.zeros((s,) + R.shape, dtype=np.int64)
        exps = np.zeros((s, R.shape[0]), dtype=np.int64)
        for p in range(1, s + 1):
            ex = np.where(nz, E + 1 - beta * p, 0)
            sigma = np.where(nz, 0.75 * np.ldexp(1.0, E + 1 - beta + 53), 0.0)
            S = (R + sigma[:, None]) - sigma[:, None]
            slices[p - 1] = (S / np.ldexp(1.0, ex)[:, None]).astype(np.int64)
            exps[p - 1] = ex
            R = R - S
        return slices, exps, R

    A, B = hpl_like(6, 5, 64, phi=0.5, seed=12)
    good = O1.ozaki1_dgemm_variant(A, B, 6, "hybrid")[0]
    monkeypatch.setattr(O1, "hybrid_split_rows", no_decay)
    bad = O1.ozaki1_dgemm_variant(A, B, 6, "hybrid")[0]
    ex = A @ B
    assert np.abs(bad - ex).max() > 1e6 * np.abs(good - ex).max()
