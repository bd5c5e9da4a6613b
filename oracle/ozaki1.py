"""Ozaki Scheme I oracle (TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__``).

Pages: [Ozaki notes] -- SplitFP (steps 1-9), the FP matrix-multiplication
algorithm (the triangular loop i + j <= s + 1), the RN split of Uchino et al.
(beta, mu, sigma = 0.75 * 2^53 * mu) and the magic-constant rounding
paragraph; [Ozaki II, §2] for the GEMM-count table.

What this oracle computes (readings listed in the design doc):

* slice width beta = min(7, floor((31 - log2 q) / 2)) with log2 taken real
  valued (RN split, step 1);
* per slice p = 1..s and per row i of the current residual R:
  mu_i = 2^(ceil(log2 max_j |R_ij|) + 1 - beta), sigma_i = 0.75 * 2^53 * mu_i
  (identical to SplitFP's sigma = 0.75 * 2^ceil(log2 m_i) * 2^(54 - alpha)
  with alpha = beta), slice S = (R + sigma) - sigma in float64 round-to-nearest,
  integer slice S / mu (|.| <= 2^(beta-1)), R <- R - S;  a zero row gives
  sigma = 0, a zero slice and mu = 1;
* all s slices are integer slices and the final residual is dropped (the
  RN split extracts s INT8 slices; SplitFP's last slice is the raw residual,
  which no integer unit could multiply);
* C = sum over i = 1..s, j = 1..s-i+1 (in that order, i outer) of
  diag(mu_A^(i)) (A'_i B'_j) diag(mu_B^(j)), every term exact, accumulated in
  float64 with round-to-nearest additions starting from C = 0.
"""
from __future__ import annotations

import math

import numpy as np

from .ozaki2 import exact_int_matmul


def beta_rn(q: int) -> int:
    """beta = min(7, floor((31 - log2 q) / 2))  ([Ozaki notes, RN split step 1])."""
    return min(7, math.floor((31 - math.log2(q)) / 2))


def alpha_splitfp(q: int, acc_bits: int) -> int:
    """alpha = floor((-log2 u_acc - log2 q) / 2)  ([Ozaki notes, SplitFP step 1])."""
    return math.floor((acc_bits - math.log2(q)) / 2)


def triangle_pairs(s: int) -> list[tuple[int, int]]:
    """(i, j) with i = 1..s, j = 1..s-i+1: the products kept by i + j <= s + 1."""
    return [(i, j) for i in range(1, s + 1) for j in range(1, s - i + 2)]


def _ceil_log2_rows(R: np.ndarray) -> np.ndarray:
    """ceil(log2 max_j |R_ij|) per row; rows that are all zero give a marker."""
    mx = np.abs(R).max(axis=1) if R.shape[1] else np.zeros(R.shape[0])
    f, e = np.frexp(mx)
    c = e.astype(np.int64) - (f == 0.5).astype(np.int64)
    return np.where(mx > 0, c, np.iinfo(np.int64).min // 4), mx > 0


def rn_split_rows(A: np.ndarray, s: int, beta: int):
    """s integer slices of the rows of A by the RN split ([Ozaki notes, RN split]).

    Returns (slices int64 s x m x q, exps int64 s x m, residual float64) with
    A = sum_p 2^exps[p][i] * slices[p][i, :] + residual exactly.
    """
    R = np.array(A, dtype=np.float64, copy=True)
    m = R.shape[0]
    slices = np.zeros((s,) + R.shape, dtype=np.int64)
    exps = np.zeros((s, m), dtype=np.int64)
    for p in range(s):
        E, nz = _ceil_log2_rows(R)
        ex = np.where(nz, E + 1 - beta, 0)
        mu = np.ldexp(1.0, ex)                                  # mu_i
        sigma = np.where(nz, 0.75 * np.ldexp(1.0, ex + 53), 0.0)  # 0.75 2^53 mu_i
        S = (R + sigma[:, None]) - sigma[:, None]               # round to the mu grid
        slices[p] = (S / mu[:, None]).astype(np.int64)          # exact: S is on the grid
        exps[p] = ex
        R = R - S
    return slices, exps, R


def ozaki1_dgemm(A: np.ndarray, B: np.ndarray, s: int, beta: int | None = None):
    """Scheme I product with s RN-split slices per operand and fixed-order accumulation."""
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    q = A.shape[1]
    if beta is None:
        beta = beta_rn(q)
    SA, XA, _ = rn_split_rows(A, s, beta)
    SBt, XB, _ = rn_split_rows(B.T, s, beta)
    C = np.zeros((A.shape[0], B.shape[1]), dtype=np.float64)
    for i, j in triangle_pairs(s):
        Cij = exact_int_matmul(SA[i - 1], SBt[j - 1].T)  # exact INT product
        term = np.ldexp(Cij.astype(np.float64), XA[i - 1][:, None] + XB[j - 1][None, :])
        C = C + term
    return C, SA, XA, SBt, XB, beta
