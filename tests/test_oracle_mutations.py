"""Planted mistakes in the oracle (CPU only) must be caught by an independent brute force.

Each case patches one step of the Scheme II oracle with a plausible slip and
checks that the result no longer matches a from-scratch brute force written
here with Fractions (exponents, truncation, exact dot products, one rounding).
"""
import math
from fractions import Fraction

import numpy as np
import pytest

from fp64_gemm_emulation_gb300.inputs import hpl_like
from oracle import ozaki2


def brute_result(A, B, s):
    mods = ozaki2.greedy_moduli(s)
    M = math.prod(mods)
    q = A.shape[1]
    k = 0
    while Fraction(q * 4 ** (k + 1)) <= Fraction(M, 2) - 1:
        k += 1

    def ceil_log2(x):
        fx, c = abs(Fraction(x)), 0
        while Fraction(2) ** c < fx:
            c += 1
        while Fraction(2) ** (c - 1) >= fx:
            c -= 1
        return c

    def scaled(row):
        nz = [v for v in row if v != 0]
        d = k - max(ceil_log2(v) for v in nz) if nz else 0
        return d, [math.trunc(Fraction(v) * Fraction(2) ** d) for v in row]

    rows = [scaled(A[i, :]) for i in range(A.shape[0])]
    cols = [scaled(B[:, j]) for j in range(B.shape[1])]
    C = np.empty((A.shape[0], B.shape[1]))
    for i, (di, a) in enumerate(rows):
        for j, (ej, b) in enumerate(cols):
            C[i, j] = float(Fraction(sum(x * y for x, y in zip(a, b))) * Fraction(2) ** (-(di + ej)))
    return C


def _case():
    return hpl_like(7, 6, 40, phi=1.0, seed=31)


def test_unmutated_oracle_matches_brute_force():
    A, B = _case()
    for s in (6, 14):
        C = ozaki2.ozaki2_dgemm(A, B, s).C
        assert np.array_equal(C.view(np.int64), brute_result(A, B, s).view(np.int64))


def _floor_instead_of_trunc(X, d_rows):
    X = np.asarray(X, dtype=np.float64)
    out = np.empty(X.shape, dtype=object)
    for i in range(X.shape[0]):
        for j in range(X.shape[1]):
            out[i, j] = math.floor(Fraction(X[i, j]) * Fraction(2) ** d_rows[i])
    return out


_orig_sym = ozaki2.symmetric_residue
_orig_choose = ozaki2.choose_k
_orig_exps = ozaki2.scale_exponents
_orig_round = ozaki2.round_scaled


def _crt_drop_last(Cres, cc):
    Z = np.zeros(Cres.shape[1:], dtype=object)
    for t in range(len(cc.moduli) - 1):
        Z = Z + Cres[t].astype(object) * (cc.Mt[t] * cc.yt[t])
    Z = np.mod(Z, cc.M)
    return np.where(Z > cc.M // 2, Z - cc.M, Z)


def _products_transposed(Ares, Bres, moduli):
    out = np.empty((len(moduli), Ares.shape[1], Bres.shape[2]), dtype=np.int64)
    for t, m in enumerate(moduli):
        out[t] = np.mod(ozaki2.exact_int_matmul(Ares[t], Bres[t][::-1, :]), m)
    return out


MUTATIONS = {
    "floor instead of trunc": ("scaled_trunc_matrix", _floor_instead_of_trunc),
    "residue of |x| (sign dropped)": ("symmetric_residue", lambda x, m: _orig_sym(np.abs(np.asarray(x)), m)),
    "k one too large": ("choose_k", lambda M, q: _orig_choose(M, q) + 1),
    "dropped CRT term": ("crt_reconstruct", _crt_drop_last),
    "reversed inner index": ("residue_products", _products_transposed),
    "exponent sign slip": ("scale_exponents", lambda E, k: [-v for v in _orig_exps(E, k)]),
    "round after unscale twice": ("round_scaled", lambda n, e: float(np.float32(_orig_round(n, e)))),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    A, B = _case()
    want = brute_result(A, B, 14)
    monkeypatch.setattr(ozaki2, attr, fn)
    try:
        got = ozaki2.ozaki2_dgemm(A, B, 14).C
    except (ValueError, OverflowError, IndexError):
        return  # the slip broke the method outright: caught
    assert not np.array_equal(got.view(np.int64), want.view(np.int64))


def test_residue_range_slip_is_caught_by_the_range_pin(monkeypatch):
    # Any representative of the right class leaves C unchanged (CRT needs only
    # congruence), so a threshold slip must be caught by the INT8 range pin.
    slip = lambda x, m: np.where(_orig_sym(x, m) == (m - 1) // 2, _orig_sym(x, m) - m, _orig_sym(x, m))
    monkeypatch.setattr(ozaki2, "symmetric_residue", slip)
    xs = np.arange(-1000, 1001)
    bad = [m for m in ozaki2.greedy_moduli(14)
           if not (np.all(ozaki2.symmetric_residue(xs, m) >= -(m // 2))
                   and np.all(ozaki2.symmetric_residue(xs, m) <= (m - 1) // 2))]
    assert bad
