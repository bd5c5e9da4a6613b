"""Pins of the FP64 summation order of the Scheme I oracle.

[Ozaki notes], FP matrix-multiplication algorithm, step 3: the kept slice products
are added to C for i = 1..s (outer) and j = 1..s-i+1 (inner), starting from C = 0.
Every term mu_i (A'_i B'_j) nu_j is an exact double (an integer below 2^31 times a
power of two), so only the additions round, and the order fixes every bit of C.

[Ozaki notes], group-wise error-free accumulation, steps 4-11: for g = 2..s+1 the
products with i + j = g (i = 1..g-1) are summed exactly in INT32, r at a time, and
each batch is scaled by the group's power of two and added to C with one FP64
addition; again the order of those additions fixes C.

The expected values here are computed from scratch: exact Python-integer dot
products of the slices, exact scaling through Fractions, and plain Python float
additions in the pages' order.  The slices themselves are pinned elsewhere (exact
reconstruction, range, Fraction brute force).  Planted orders (reversed, j outer,
groups reversed) must be caught.
"""
from fractions import Fraction

import numpy as np
import pytest

from fp64_gemm_emulation_gb300.inputs import hpl_like
from oracle import ozaki1 as O1


def _int_dot(x, y):
    return sum(int(a) * int(b) for a, b in zip(x, y))


def _exact_term(v, e):
    """v * 2^e as a double, asserting that the conversion is exact."""
    f = Fraction(v) * Fraction(2) ** int(e)
    d = float(f)
    assert Fraction(d) == f
    return d


def scheme1_rn_in_page_order(SA, XA, SBt, XB, s):
    """C_ij = sum over i = 1..s, j = 1..s-i+1 (i outer) of the exact terms, Python floats."""
    m, n = SA.shape[1], SBt.shape[1]
    C = np.zeros((m, n))
    for r in range(m):
        for c in range(n):
            acc = 0.0
            for i in range(1, s + 1):
                for j in range(1, s - i + 2):
                    v = _int_dot(SA[i - 1, r], SBt[j - 1, c])
                    acc = acc + _exact_term(v, XA[i - 1, r] + XB[j - 1, c])
            C[r, c] = acc
    return C


def scheme1_groupwise_in_page_order(SA, XA, SBt, XB, s, r):
    """Group-wise: for g = 2..s+1, pairs i = 1..g-1 in batches of r; one FP64 add per batch."""
    m, n = SA.shape[1], SBt.shape[1]
    C = np.zeros((m, n))
    for a in range(m):
        for b in range(n):
            acc = 0.0
            for g in range(2, s + 2):
                pairs = [(i, g - i) for i in range(1, g)]
                for b0 in range(0, len(pairs), r):
                    batch = pairs[b0 : b0 + r]
                    v = sum(_int_dot(SA[i - 1, a], SBt[j - 1, b]) for i, j in batch)
                    assert abs(v) < 2**31
                    i1, j1 = batch[0]
                    acc = acc + _exact_term(v, XA[i1 - 1, a] + XB[j1 - 1, b])
            C[a, b] = acc
    return C


CASES = [(9, 7, 96, 0.5, 41), (6, 10, 200, 2.0, 42), (12, 5, 64, 2.0, 43), (16, 16, 128, 0.5, 46)]
# a case on which a slip in the order changes dozens of result bits at s = 7 and 8
SLIP_CASE = (16, 16, 128, 0.5, 46)


@pytest.mark.parametrize("s", [3, 7, 8])
@pytest.mark.parametrize("m,n,k,phi,seed", CASES)
def test_rn_accumulation_is_in_the_pages_order(m, n, k, phi, seed, s):
    A, B = hpl_like(m, n, k, phi=phi, seed=seed)
    C, SA, XA, SBt, XB, _ = O1.ozaki1_dgemm(A, B, s)
    want = scheme1_rn_in_page_order(SA, XA, SBt, XB, s)
    assert np.array_equal(C.view(np.int64), want.view(np.int64))


@pytest.mark.parametrize("variant", ["ef", "hybrid"])
@pytest.mark.parametrize("s", [3, 7, 8])
@pytest.mark.parametrize("m,n,k,phi,seed", CASES[:2])
def test_groupwise_accumulation_is_in_the_pages_order(m, n, k, phi, seed, s, variant):
    A, B = hpl_like(m, n, k, phi=phi, seed=seed)
    C, SA, XA, SBt, XB, beta = O1.ozaki1_dgemm_variant(A, B, s, variant)
    want = scheme1_groupwise_in_page_order(SA, XA, SBt, XB, s, O1.group_r(k, beta))
    assert np.array_equal(C.view(np.int64), want.view(np.int64))


# groups cut into several batches: beta is forced to 10 at q = 1024, so
# r = max(1, 2^(31 - 20 - 10)) = 2 and the groups of three or more pairs are cut
BATCH_CASE = (12, 12, 1024, 1.0, 45)
BATCH_BETA = 10


def test_groupwise_order_with_several_batches_per_group():
    m, n, k, phi, seed = BATCH_CASE
    A, B = hpl_like(m, n, k, phi=phi, seed=seed)
    s = 6
    r = O1.group_r(k, BATCH_BETA)
    assert r == 2
    for variant in ("ef", "hybrid"):
        C, SA, XA, SBt, XB, _ = O1.ozaki1_dgemm_variant(A, B, s, variant, beta=BATCH_BETA)
        want = scheme1_groupwise_in_page_order(SA, XA, SBt, XB, s, r)
        assert np.array_equal(C.view(np.int64), want.view(np.int64))


# ------------------------------------------------------------------ planted orders
def _bits_differ(X, Y):
    return not np.array_equal(X.view(np.int64), Y.view(np.int64))


RN_SLIPS = {
    "reversed": lambda s: list(reversed([(i, j) for i in range(1, s + 1) for j in range(1, s - i + 2)])),
    "j outer": lambda s: [(i, j) for j in range(1, s + 1) for i in range(1, s - j + 2)],
}


@pytest.mark.parametrize("slip", sorted(RN_SLIPS))
@pytest.mark.parametrize("s", [7, 8])
def test_planted_rn_order_is_caught(slip, s, monkeypatch):
    m, n, k, phi, seed = SLIP_CASE
    A, B = hpl_like(m, n, k, phi=phi, seed=seed)
    _, SA, XA, SBt, XB, _ = O1.ozaki1_dgemm(A, B, s)
    want = scheme1_rn_in_page_order(SA, XA, SBt, XB, s)
    monkeypatch.setattr(O1, "triangle_pairs", RN_SLIPS[slip])
    got = O1.ozaki1_dgemm(A, B, s)[0]
    assert _bits_differ(got, want)


def _groups_reversed(s, r):
    out = []
    for g in range(s + 1, 1, -1):
        pairs = [(i, g - i) for i in range(1, g)]
        for b0 in range(0, len(pairs), r):
            out.append((g, pairs[b0 : b0 + r]))
    return out


def _batches_reversed_inside_groups(s, r):
    out = []
    for g in range(2, s + 2):
        pairs = [(i, g - i) for i in range(1, g)]
        cut = [pairs[b0 : b0 + r] for b0 in range(0, len(pairs), r)]
        out.extend((g, b) for b in reversed(cut))
    return out


@pytest.mark.parametrize("variant", ["ef", "hybrid"])
def test_planted_group_order_is_caught(variant, monkeypatch):
    m, n, k, phi, seed = SLIP_CASE
    s = 8
    A, B = hpl_like(m, n, k, phi=phi, seed=seed)
    _, SA, XA, SBt, XB, beta = O1.ozaki1_dgemm_variant(A, B, s, variant)
    want = scheme1_groupwise_in_page_order(SA, XA, SBt, XB, s, O1.group_r(k, beta))
    monkeypatch.setattr(O1, "group_batches", _groups_reversed)
    got = O1.ozaki1_dgemm_variant(A, B, s, variant)[0]
    assert _bits_differ(got, want)


@pytest.mark.parametrize("variant", ["ef", "hybrid"])
def test_planted_batch_order_inside_a_group_is_caught(variant, monkeypatch):
    m, n, k, phi, seed = BATCH_CASE
    A, B = hpl_like(m, n, k, phi=phi, seed=seed)
    s = 6
    r = O1.group_r(k, BATCH_BETA)
    _, SA, XA, SBt, XB, _ = O1.ozaki1_dgemm_variant(A, B, s, variant, beta=BATCH_BETA)
    want = scheme1_groupwise_in_page_order(SA, XA, SBt, XB, s, r)
    monkeypatch.setattr(O1, "group_batches", _batches_reversed_inside_groups)
    got = O1.ozaki1_dgemm_variant(A, B, s, variant, beta=BATCH_BETA)[0]
    assert _bits_differ(got, want)
