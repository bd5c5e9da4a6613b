"""Ozaki Scheme I oracle (TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__``).

Pages: [Ozaki notes] -- SplitFP (steps 1-9), the FP matrix-multiplication
algorithm (the triangular loop i + j <= s + 1), the RN split of Uchino et al.
(beta, mu, sigma = 0.75 * 2^53 * mu) and the magic-constant rounding
paragraph; [Ozaki II, §2] for the GEMM-count table.

What this oracle computes (the readings taken where the notes leave a step open):

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

The two variants of [Ozaki notes, "group-wise error-free accumulation" and
"Hybrid"] (variant names "ef" and "hybrid"):

* EF: the bitmask split (SplitInt): with e_i = floor(log2 max_j |a_ij|) the row's
  leading bit, |a| is truncated to the grid 2^(e_i + 1 - s beta) and its s
  consecutive beta-bit fields below 2^(e_i + 1) are the slices (sign applied),
  slice p carrying the scale 2^(e_i + 1 - p beta);
* Hybrid: the RN split with mu''_i = 2^(ceil(log2 max_j |a_ij|) + 1 - beta) fixed
  from the input and sigma_i = 0.75 * 2^(53 - beta (p - 1)) mu''_i for slice p, so
  slice p carries the fixed scale mu''_i 2^(-beta (p - 1));
* both accumulate group-wise: for g = 2..s+1 the products of slice i of A with
  slice g - i of B (i = 1..g-1, in that order) share the scale of the group and
  are summed exactly in INT32, r = max(1, 2^(31 - 2 beta - ceil(log2 q))) products
  at a time; each batch is converted to float64, scaled (exact) and added to C.
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


# --------------------------------------------------------------------------
# Group-wise error-free accumulation and the EF / Hybrid splits ([Ozaki notes])
# --------------------------------------------------------------------------
VARIANTS = ("rn", "ef", "hybrid")


def group_r(q: int, beta: int) -> int:
    """r = max(1, 2^(31 - 2 beta - ceil(log2 q))): products an INT32 sum holds exactly."""
    e = 31 - 2 * beta - (q - 1).bit_length()  # (q - 1).bit_length() = ceil(log2 q), q >= 1
    return 2**e if e > 0 else 1


def group_batches(s: int, r: int) -> list[tuple[int, list[tuple[int, int]]]]:
    """[(g, [(i, j), ...]), ...]: groups g = 2..s+1 of the pairs i + j = g (i = 1..g-1),
    cut into consecutive batches of at most r pairs."""
    out = []
    for g in range(2, s + 2):
        pairs = [(i, g - i) for i in range(1, g)]
        for b0 in range(0, len(pairs), r):
            out.append((g, pairs[b0 : b0 + r]))
    return out


def _floor_log2_rows(X: np.ndarray):
    """floor(log2 max_j |x_ij|) per row and a nonzero-row mask (exact: frexp)."""
    mx = np.abs(X).max(axis=1) if X.shape[1] else np.zeros(X.shape[0])
    f, e = np.frexp(mx)  # mx = f 2^e, f in [1/2, 1)
    return np.where(mx > 0, e.astype(np.int64) - 1, 0), mx > 0


def bitmask_split_rows(A: np.ndarray, s: int, beta: int):
    """EF split (SplitInt): s beta-bit fields of |a| below the row's leading bit.

    Returns (slices int64 s x m x q, exps int64 s x m): slice p of row i has scale
    2^exps[p][i] = 2^(e_i + 1 - p beta), and sum_p slices * scale is |a| truncated to
    the grid 2^(e_i + 1 - s beta), with the sign of a.
    """
    A = np.asarray(A, dtype=np.float64)
    m, q = A.shape
    e, nz = _floor_log2_rows(A)
    slices = np.zeros((s, m, q), dtype=np.int64)
    exps = np.zeros((s, m), dtype=np.int64)
    mask = (1 << beta) - 1
    for i in range(m):
        if not nz[i]:
            continue
        for p in range(1, s + 1):
            exps[p - 1, i] = e[i] + 1 - p * beta
        for j in range(q):
            x = float(A[i, j])
            if x == 0.0:
                continue
            num, den = abs(x).as_integer_ratio()  # |x| = num / den, den a power of two
            sh = s * beta - int(e[i]) - 1          # N = floor(|x| 2^sh) < 2^(s beta)
            N = (num << sh) // den if sh >= 0 else num // (den << (-sh))
            sg = -1 if x < 0 else 1
            for p in range(1, s + 1):
                slices[p - 1, i, j] = sg * ((N >> ((s - p) * beta)) & mask)
    return slices, exps


def hybrid_split_rows(A: np.ndarray, s: int, beta: int):
    """Hybrid split: RN to the fixed grids mu''_i 2^(-beta (p - 1)) (sigma decays instead of mu).

    Returns (slices, exps, residual) with A = sum_p 2^exps[p][i] slices[p][i, :] + residual.
    """
    R = np.array(A, dtype=np.float64, copy=True)
    m = R.shape[0]
    E, nz = _ceil_log2_rows(R)
    slices = np.zeros((s,) + R.shape, dtype=np.int64)
    exps = np.zeros((s, m), dtype=np.int64)
    for p in range(1, s + 1):
        ex = np.where(nz, E + 1 - beta * p, 0)                   # log2 of mu''_i 2^(-beta (p-1))
        grid = np.ldexp(1.0, ex)
        sigma = np.where(nz, 0.75 * np.ldexp(1.0, ex + 53), 0.0)  # 0.75 2^(53 - beta(p-1)) mu''_i
        S = (R + sigma[:, None]) - sigma[:, None]                # round to the grid
        slices[p - 1] = (S / grid[:, None]).astype(np.int64)     # exact: S is on the grid
        exps[p - 1] = ex
        R = R - S
    return slices, exps, R


def ozaki1_dgemm_variant(A: np.ndarray, B: np.ndarray, s: int, variant: str, beta: int | None = None):
    """Scheme I with the EF or Hybrid split and group-wise accumulation (or "rn")."""
    if variant == "rn":
        return ozaki1_dgemm(A, B, s, beta)
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    q = A.shape[1]
    if beta is None:
        beta = beta_rn(q)
    if variant == "ef":
        SA, XA = bitmask_split_rows(A, s, beta)
        SBt, XB = bitmask_split_rows(B.T, s, beta)
    elif variant == "hybrid":
        SA, XA, _ = hybrid_split_rows(A, s, beta)
        SBt, XB, _ = hybrid_split_rows(B.T, s, beta)
    else:
        raise ValueError(f"unknown variant {variant!r}")
    r = group_r(q, beta)
    C = np.zeros((A.shape[0], B.shape[1]), dtype=np.float64)
    for g, pairs in group_batches(s, r):
        acc = np.zeros_like(C, dtype=np.int64)
        for i, j in pairs:
            acc = acc + exact_int_matmul(SA[i - 1], SBt[j - 1].T)   # exact INT products
        assert np.abs(acc).max(initial=0) < 2**31                     # the INT32 sum is exact
        x = XA[pairs[0][0] - 1][:, None] + XB[pairs[0][1] - 1][None, :]
        for i, j in pairs:  # every pair of the group has the same scale where the batch is nonzero
            assert not ((XA[i - 1][:, None] + XB[j - 1][None, :] != x) & (acc != 0)).any()
        C = C + np.ldexp(acc.astype(np.float64), x)
    return C, SA, XA, SBt, XB, beta
