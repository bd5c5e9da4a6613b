"""Seeded synthetic inputs (shared by the tests, the benchmark and the oracle checks).

This module holds only the input recipe, none of the emulation's arithmetic.

The workload is the HPL-like distribution used to measure Ozaki Scheme II's
accuracy and speed (the explainer "Ozaki Scheme II: mapping high-precision GEMM
to a few INT8 GEMMs with CRT", §10, at phi = 0.5): every entry is
``(U(0,1) - 0.5) * exp(phi * N(0,1))``, so ``phi`` widens the spread of
exponents within a row (phi = 0: uniform in (-0.5, 0.5); phi = 4: many
binades).  A is drawn first, then B, from one numpy PCG64 generator; both are
returned column-major (Fortran order), the layout the C ABI takes.
"""
from __future__ import annotations

import numpy as np


def hpl_like(m: int, n: int, k: int, phi: float = 0.5, seed: int = 0):
    """Return column-major float64 A (m x k) and B (k x n)."""
    rng = np.random.default_rng(seed)
    A = (rng.random((m, k)) - 0.5) * np.exp(phi * rng.standard_normal((m, k)))
    B = (rng.random((k, n)) - 0.5) * np.exp(phi * rng.standard_normal((k, n)))
    return np.asfortranarray(A), np.asfortranarray(B)


def special_matrix(kind: str, rows: int, cols: int, seed: int = 0) -> np.ndarray:
    """Edge-case operands (column-major float64) for correctness tests.

    kinds: ``zeros``, ``pow2`` (signed powers of two over a wide range),
    ``subnormal`` (entries around 2^-1060), ``huge`` (entries near 2^1000),
    ``zero_rows`` (HPL-like with every third row and column zeroed),
    ``ints`` (small integers, exactly representable products).
    """
    rng = np.random.default_rng(seed)
    if kind == "zeros":
        X = np.zeros((rows, cols))
    elif kind == "pow2":
        X = np.ldexp(rng.choice([-1.0, 1.0], (rows, cols)), rng.integers(-40, 40, (rows, cols)))
    elif kind == "subnormal":
        X = np.ldexp(rng.random((rows, cols)) - 0.5, rng.integers(-1062, -1050, (rows, cols)))
    elif kind == "huge":
        X = np.ldexp(rng.random((rows, cols)) - 0.5, rng.integers(990, 1000, (rows, cols)))
    elif kind == "zero_rows":
        X = (rng.random((rows, cols)) - 0.5) * np.exp(0.5 * rng.standard_normal((rows, cols)))
        X[::3, :] = 0.0
        X[:, ::3] = 0.0
    elif kind == "ints":
        X = rng.integers(-20, 21, (rows, cols)).astype(np.float64)
    else:
        raise ValueError(kind)
    return np.asfortranarray(X)
