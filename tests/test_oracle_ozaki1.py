"""Pins for the Scheme I oracle (RN split, triangular products, FP64 accumulation)."""
import math
from fractions import Fraction

import numpy as np
import pytest

from fp64_gemm_emulation_gb300.inputs import hpl_like, special_matrix
from oracle import ozaki1

from test_oracle_ozaki2 import exact_product_fraction


def test_beta_values_from_the_rn_split_formula():
    # beta = min(7, floor((31 - log2 n)/2)): INT8 limits 7 bits, INT32 the rest.
    assert ozaki1.beta_rn(4096) == 7
    assert ozaki1.beta_rn(16384) == 7
    assert ozaki1.beta_rn(2**17) == 7
    assert ozaki1.beta_rn(262144) == 6
    assert ozaki1.beta_rn(2**21) == 5
    # SplitFP alpha with an FP32 accumulator (u_acc = 2^-24) and an INT32 one (2^-31)
    assert ozaki1.alpha_splitfp(4096, 24) == 6
    assert ozaki1.alpha_splitfp(4096, 31) == 9


def test_int32_never_overflows_for_the_chosen_beta():
    for q in (1, 100, 4096, 65536, 2**17, 262144, 2**20):
        b = ozaki1.beta_rn(q)
        assert q * (2 ** (b - 1)) ** 2 <= 2**31


def test_magic_constant_rounds_to_nearest_even():
    # (a + 1.5 2^52) - 1.5 2^52 == RN-even(a) for |a| < 2^51; on a grid
    # delta = 2^t the constant scales to 1.5 2^52 delta.
    rng = np.random.default_rng(20)
    a = (rng.random(20000) - 0.5) * 2.0**52
    a = np.concatenate([a, np.arange(-20, 20) + 0.5, [2.0**51 - 0.5, -(2.0**51) + 0.5]])
    sigma = 1.5 * 2.0**52
    assert np.array_equal((a + sigma) - sigma, np.rint(a))
    for t in (-30, 0, 17):
        delta = 2.0**t
        sig = 1.5 * 2.0**52 * delta
        assert np.array_equal((a * delta + sig) - sig, np.rint(a) * delta)


@pytest.mark.parametrize("phi", [0.0, 0.5, 4.0])
def test_rn_slices_are_bounded_and_error_free(phi):
    A, _ = hpl_like(12, 1, 200, phi=phi, seed=21)
    A[3, :] = 0.0
    beta = ozaki1.beta_rn(200)
    S, X, R = ozaki1.rn_split_rows(A, 6, beta)
    assert np.abs(S).max() <= 2 ** (beta - 1)
    assert np.all(S[:, 3, :] == 0)
    for i in range(A.shape[0]):
        for j in range(A.shape[1]):
            total = sum(Fraction(int(S[p, i, j])) * Fraction(2) ** int(X[p, i]) for p in range(6))
            assert total + Fraction(R[i, j]) == Fraction(A[i, j])   # exact split
    # each slice shrinks the residual by about beta bits
    assert np.all(np.abs(R) <= np.ldexp(np.abs(A).max(axis=1), -6 * (beta - 1))[:, None] + 0)


def test_gemm_count_for_seven_slices():
    assert len(ozaki1.triangle_pairs(7)) == 28


def test_scheme1_accuracy_improves_with_slices_to_dgemm_level():
    # [Ozaki II, §10]: Scheme I needs about 7-8 slices (28-36 GEMMs) for
    # DGEMM-like accuracy on phi = 0.5 data.
    m, n, k = 12, 12, 256
    A, B = hpl_like(m, n, k, phi=0.5, seed=22)
    exact = exact_product_fraction(A, B)
    absAB = np.abs(A) @ np.abs(B)

    def err(C):
        return max(float(abs(Fraction(float(C[i, j])) - exact[i, j])) / absAB[i, j]
                   for i in range(m) for j in range(n))

    e_dgemm = err(A @ B)
    e = {s: err(ozaki1.ozaki1_dgemm(A, B, s)[0]) for s in (4, 6, 7, 8)}
    assert e[4] > e[6] > e[7] > e[8]
    assert e[8] <= 4 * e_dgemm
    assert e[4] > 1e5 * e_dgemm


def test_integer_inputs_are_exact():
    A = special_matrix("ints", 10, 20, seed=23)
    B = special_matrix("ints", 20, 9, seed=24)
    C = ozaki1.ozaki1_dgemm(A, B, 2)[0]
    assert np.array_equal(C, (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float64))
