"""Ozaki Scheme II oracle (TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__``).

Notation follows [Ozaki II]: A is p x q, B is q x r (here m x k and k x n),
s pairwise-coprime moduli m_1 > ... > m_s, M = prod m_t, M_t = M / m_t,
y_t = M_t^{-1} mod m_t, D = diag(2^d_i), E = diag(2^e_j), A' = trunc(DA),
B' = trunc(BE).

The result this oracle defines (and the GPU path must reproduce bit for bit):

    C_ij = RN( 2^-(d_i + e_j) * sum_k A'_ik B'_kj )

i.e. the exact integer product of the truncated scaled matrices, rounded once
(round-to-nearest-even, including into the subnormal range) after the inverse
scaling.  :func:`ozaki2_dgemm` reaches it the method's way (residues, one exact
product per modulus, CRT, range reduction) and :func:`direct_dgemm` reaches it
from the definition; tests require both to agree.

Readings taken where the pages leave a step open:

* moduli: the greedy descending pairwise-coprime list starting at 256
  ([Ozaki II, §6] only fixes 2 <= m_t <= 256 and pairwise coprimality);
* k_A = k_B = the largest integer k with q * 2^(2k) <= M/2 - 1, which is the
  exact integer form of floor(1/2 * log2((M/2 - 1)/q)) ([Ozaki II, §5]);
* d_i = k_A - ceil(log2 max_j |a_ij|), the largest power of two that keeps
  |D_ii a_ij| <= 2^k_A ([Ozaki II, §3], with the bound c_max <= q 2^(k_A+k_B)
  of §5); zero rows get d_i = 0;
* trunc is rounding toward zero ([Ozaki II, §7 step 2]);
* the symmetric residue of x mod m is r = x mod m in [0, m), minus m when
  r >= ceil(m/2); for m = 256 this is [-128, 127] ([Ozaki II, §6]);
* C''_t is taken in [0, m_t) ([Ozaki II, §7 step 3]);
* rows of A / columns of B that hold a non-finite value produce NaN rows /
  columns of C (the pages are silent).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# Largest modulus allowed on the GPU: residues must fit signed INT8 [Ozaki II, §6].
MODULUS_MAX = 256


# --------------------------------------------------------------------------
# Step 1 of Algorithm 1: parameters
# --------------------------------------------------------------------------
def greedy_moduli(s: int, top: int = MODULUS_MAX) -> list[int]:
    """First ``s`` pairwise-coprime integers taken greedily downward from ``top``.

    [Ozaki II, §4] needs pairwise-coprime moduli; [Ozaki II, §6] bounds them
    by 2 <= m_t <= 256 so symmetric residues fit INT8.  Which ones is not
    stated; the greedy list keeps each m_t as large as possible, which
    maximises M for a given s.
    """
    if s < 1:
        raise ValueError("need at least one modulus")
    out: list[int] = []
    cand = top
    while len(out) < s:
        if cand < 2:
            raise ValueError(f"only {len(out)} pairwise-coprime moduli <= {top}")
        if all(math.gcd(cand, prev) == 1 for prev in out):
            out.append(cand)
        cand -= 1
    return out


@dataclass
class CrtConstants:
    """M, M_t and y_t of [Ozaki II, §4] for one moduli list."""

    moduli: list[int]
    M: int
    Mt: list[int] = field(default_factory=list)
    yt: list[int] = field(default_factory=list)


def crt_constants(moduli: list[int]) -> CrtConstants:
    """M = prod m_t, M_t = M/m_t, y_t = M_t^{-1} mod m_t  ([Ozaki II, §4])."""
    M = 1
    for m in moduli:
        M *= m
    Mt = [M // m for m in moduli]
    yt = [pow(Mt_t % m, -1, m) for Mt_t, m in zip(Mt, moduli)]
    return CrtConstants(list(moduli), M, Mt, yt)


def choose_k(M: int, q: int) -> int:
    """k_A = k_B = floor(1/2 * log2((M/2 - 1) / q))  ([Ozaki II, §5]).

    Computed exactly: the largest integer k with q * 2^(2k) <= M/2 - 1.
    (Both sides doubled so M odd is handled without fractions.)
    Raises ValueError when not even k = 0 satisfies the bound.
    """
    if q < 1:
        raise ValueError("inner dimension must be positive")
    # q * 4^k <= M/2 - 1   <=>   2 q 4^k <= M - 2
    if 2 * q > M - 2:
        raise ValueError("M too small for this inner dimension")
    k = 0
    while 2 * q * 4 ** (k + 1) <= M - 2:
        k += 1
    return k


# --------------------------------------------------------------------------
# Step 2 of Algorithm 1: scaling and truncation
# --------------------------------------------------------------------------
def ceil_log2_abs(x: float) -> int:
    """ceil(log2 |x|) for finite nonzero x, exact (frexp: |x| = f 2^e, f in [1/2, 1))."""
    f, e = math.frexp(abs(x))
    return e - 1 if f == 0.5 else e


def _ceil_log2_abs_array(X: np.ndarray) -> np.ndarray:
    """Element-wise ceil(log2|x|) as int64; 0 entries map to a very small value."""
    f, e = np.frexp(np.abs(X))
    c = e.astype(np.int64) - (f == 0.5).astype(np.int64)
    return np.where(X != 0, c, np.iinfo(np.int64).min // 4)


ZERO_ROW = None  # marker for an all-zero row / column in the exponent vectors


def row_exponents(A: np.ndarray) -> list:
    """E_i = ceil(log2 max_j |a_ij|) per row (None for a zero row, 'nan' if non-finite)."""
    A = np.asarray(A, dtype=np.float64)
    out: list = []
    finite = np.isfinite(A).all(axis=1)
    c = _ceil_log2_abs_array(np.where(np.isfinite(A), A, 0.0))
    mx = c.max(axis=1) if A.shape[1] > 0 else np.full(A.shape[0], np.iinfo(np.int64).min // 4)
    for i in range(A.shape[0]):
        if not finite[i]:
            out.append("nan")
        elif mx[i] <= np.iinfo(np.int64).min // 8:
            out.append(ZERO_ROW)
        else:
            out.append(int(mx[i]))
    return out


def scale_exponents(E: list, k: int) -> list[int]:
    """d_i = k - E_i (0 for zero or non-finite rows)  ([Ozaki II, §3, §7 step 2])."""
    return [0 if (e is ZERO_ROW or e == "nan") else k - e for e in E]


def scaled_trunc(x: float, d: int) -> int:
    """trunc(x * 2^d) as an exact integer (rounding toward zero)."""
    n, den = float(x).as_integer_ratio()  # x = n / den, den a power of two
    if d >= 0:
        num = n * (1 << d)
        return num // den if num >= 0 else -((-num) // den)
    den = den << (-d)
    return n // den if n >= 0 else -((-n) // den)


def scaled_trunc_matrix(X: np.ndarray, d_rows: list[int]) -> np.ndarray:
    """A' = trunc(D X) with D = diag(2^d_i) applied to rows; exact.

    Returns int64 when every |A'| fits comfortably (vectorised), else an object
    array of Python integers computed element by element.  Non-finite entries are treated as 0 (their rows are
    flagged separately and produce NaN).
    """
    X = np.asarray(X, dtype=np.float64)
    Xf = np.where(np.isfinite(X), X, 0.0)
    d = np.asarray(d_rows, dtype=np.int64).reshape(-1, 1)
    f, e = np.frexp(np.abs(Xf))
    # |x| = sig * 2^(e-53) with sig = f * 2^53 an integer < 2^53 (exact).
    sig = np.ldexp(f, 53).astype(np.int64)
    sh = e.astype(np.int64) - 53 + d  # |x| 2^d = sig 2^sh
    if np.all(sh <= 62 - 53):
        right = np.clip(-sh, 0, 63)
        mag = np.where(right >= 63, 0, sig >> np.minimum(right, 62))
        left = np.clip(sh, 0, None)
        mag = mag << left
        return np.where(Xf < 0, -mag, mag).astype(np.int64)
    out = np.empty(X.shape, dtype=object)
    for i in range(X.shape[0]):
        for j in range(X.shape[1]):
            out[i, j] = scaled_trunc(float(Xf[i, j]), int(d_rows[i]))
    return out


# --------------------------------------------------------------------------
# Step 3 of Algorithm 1: residues, one exact product per modulus, re-modulo
# --------------------------------------------------------------------------
def symmetric_residue(x, m: int):
    """Symmetric representative of x mod m: [0, m) shifted down by m above ceil(m/2)."""
    x = np.asarray(x)
    r = np.mod(x, m).astype(np.int64)  # floor mod: [0, m) for m > 0
    return np.where(r >= (m + 1) // 2, r - m, r).astype(np.int64)


def residue_planes(Xp: np.ndarray, moduli: list[int]) -> np.ndarray:
    """A'_t = A' mod m_t (symmetric, int8) for every t  ([Ozaki II, §7 step 3])."""
    planes = np.empty((len(moduli),) + Xp.shape, dtype=np.int8)
    for t, m in enumerate(moduli):
        planes[t] = symmetric_residue(Xp, m).astype(np.int8)
    return planes


def exact_int_matmul(Ai: np.ndarray, Bi: np.ndarray) -> np.ndarray:
    """Exact integer product of two small-integer matrices via a float64 matmul.

    Exact because every entry is an integer and every partial sum stays below
    2^53 in magnitude (the caller's inputs are bounded by 128 in magnitude and
    q < 2^39, so |sum| <= q 2^14 < 2^53).
    """
    Ai = np.asarray(Ai, dtype=np.int64)
    Bi = np.asarray(Bi, dtype=np.int64)
    q = Ai.shape[1]
    bound = int(np.abs(Ai).max(initial=0)) * int(np.abs(Bi).max(initial=0)) * max(q, 1)
    if bound >= 2**53:
        raise ValueError("float64 product would not be exact")
    return (Ai.astype(np.float64) @ Bi.astype(np.float64)).astype(np.int64)


def residue_products(Ares: np.ndarray, Bres: np.ndarray, moduli: list[int]) -> np.ndarray:
    """C''_t = (A'_t B'_t) mod m_t in [0, m_t)  ([Ozaki II, §7 step 3])."""
    out = np.empty((len(moduli), Ares.shape[1], Bres.shape[2]), dtype=np.int64)
    for t, m in enumerate(moduli):
        Ct = exact_int_matmul(Ares[t], Bres[t])  # C'_t, exact INT
        out[t] = np.mod(Ct, m)
    return out


# --------------------------------------------------------------------------
# Steps 4-5 of Algorithm 1: CRT accumulation and range reduction
# --------------------------------------------------------------------------
def crt_reconstruct(Cres: np.ndarray, cc: CrtConstants) -> np.ndarray:
    """C''' = (sum_t C''_t M_t y_t) mod M, symmetric representative (object ints).

    [Ozaki II, §7 steps 4-5]; unique because |A'B'| <= c_max < M/2 ([Ozaki II, §5]).
    """
    Z = np.zeros(Cres.shape[1:], dtype=object)
    for t in range(len(cc.moduli)):
        Z = Z + Cres[t].astype(object) * (cc.Mt[t] * cc.yt[t])
    Z = np.mod(Z, cc.M)
    half = cc.M // 2
    return np.where(Z > half, Z - cc.M, Z)


# --------------------------------------------------------------------------
# Step 6 of Algorithm 1: inverse scaling with one rounding
# --------------------------------------------------------------------------
def round_scaled(n: int, e: int) -> float:
    """RN-even of the exact value n * 2^e (one rounding; +-inf on overflow)."""
    n = int(n)
    if n == 0:
        return 0.0
    try:
        if e >= 0:
            return float(n << e)
        return n / (1 << (-e))  # int/int true division is correctly rounded
    except OverflowError:
        return math.copysign(math.inf, n)


def unscale(C3: np.ndarray, d: list[int], e: list[int], rowflag=None, colflag=None) -> np.ndarray:
    """C = D^{-1} C''' E^{-1}, rounded once  ([Ozaki II, §7 step 6])."""
    m, n = C3.shape
    C = np.empty((m, n), dtype=np.float64)
    for i in range(m):
        for j in range(n):
            C[i, j] = round_scaled(C3[i, j], -(d[i] + e[j]))
    if rowflag is not None:
        C[np.asarray(rowflag, dtype=bool), :] = np.nan
    if colflag is not None:
        C[:, np.asarray(colflag, dtype=bool)] = np.nan
    return C


# --------------------------------------------------------------------------
# Range estimation variants ([Ozaki II, §9]): OS II-fast and OS II-accu
# --------------------------------------------------------------------------
# The CRT result is unique when c_max >= max_ij (|A'||B'|)_ij stays <= M/2 - 1
# ([Ozaki II, §5, §9]).  The uniform estimate above takes c_max = q 2^(k_A+k_B).
# OS II-fast bounds (|A'||B'|)_ij by the Cauchy-Schwarz product of a row norm of A'
# and a column norm of B'; OS II-accu bounds it entry by entry with an exact
# low-precision product of rounded-up magnitudes.  Both keep the form
# d_i = kappa - t_i with kappa the largest k such that 2^(2k) <= M/2 - 1 (the k of
# q = 1) and a per-row exponent t_i; everything after the exponents is unchanged.
SCALINGS = ("uniform", "fast", "accu")
NORM_GUARD = 16  # G: entries below 2^-G of the row maximum count as 4^-G of its square


def half_range_log2(M: int) -> int:
    """L = floor(log2(M/2 - 1)): the largest L with 2^L <= M/2 - 1 (i.e. 2^(L+1) <= M - 2)."""
    if M - 2 < 2:
        raise ValueError("M too small")
    return (M - 2).bit_length() - 2


def ceil_log2_int(x: int) -> int:
    """ceil(log2 x) for an integer x >= 1."""
    if x < 1:
        raise ValueError("need x >= 1")
    return (int(x) - 1).bit_length()


def norm_exponents(X: np.ndarray) -> list:
    """OS II-fast: per row, an integer t with 2^t >= ||x_i||_2 (None / 'nan' as in row_exponents).

    Each |x_ik| <= 2^c_k with c_k = ceil(log2 |x_ik|) exact from the bits, so
    ||x_i||^2 <= sum_k 4^c_k <= 4^(c_max - G) S,  S = sum_k max(1, 4^(c_k - c_max + G)),
    an integer (order-free), and ||x_i|| <= 2^(c_max - G + ceil(ceil(log2 S) / 2)) = 2^t.
    """
    X = np.asarray(X, dtype=np.float64)
    finite = np.isfinite(X).all(axis=1)
    out: list = []
    for i in range(X.shape[0]):
        if not finite[i]:
            out.append("nan")
            continue
        row = X[i][X[i] != 0]
        if row.size == 0:
            out.append(ZERO_ROW)
            continue
        c = _ceil_log2_abs_array(row)
        cmax = int(c.max())
        delta = c - cmax + NORM_GUARD  # <= G
        S = sum(4 ** int(dv) if dv >= 0 else 1 for dv in delta)
        L = ceil_log2_int(S)
        out.append(cmax - NORM_GUARD + (L + 1) // 2)
    return out


def accu_bits(q: int) -> int:
    """OS II-accu: b = the largest integer in [0, 7] with q 4^b <= 2^24.

    Bound entries are integers in [0, 2^b]; their products (<= 4^b) summed over q
    stay <= 2^24, so one FP32 accumulation (or any integer arithmetic) is exact.
    """
    if q < 1 or q > 2**24:
        raise ValueError("OS II-accu needs 1 <= q <= 2^24")
    b = 0
    while b < 7 and q * 4 ** (b + 1) <= 2**24:
        b += 1
    return b


def magnitude_bounds(X: np.ndarray, E: list, b: int) -> np.ndarray:
    """X^_ik = ceil(|x_ik| 2^(b - E_i)) in [0, 2^b] (int64); rows without an exponent are 0.

    With E_i = ceil(log2 max_k |x_ik|) this is |x_ik| rounded up to b bits of the
    row's range: |x_ik| <= X^_ik 2^(E_i - b).
    """
    X = np.asarray(X, dtype=np.float64)
    out = np.zeros(X.shape, dtype=np.int64)
    f, e = np.frexp(np.abs(np.where(np.isfinite(X), X, 0.0)))
    sig = np.ldexp(f, 53).astype(np.int64)  # |x| = sig 2^(e - 53), exact
    for i in range(X.shape[0]):
        if E[i] is ZERO_ROW or E[i] == "nan":
            continue
        sh = e[i].astype(np.int64) - 53 + b - int(E[i])  # |x| 2^(b - E) = sig 2^sh
        right = -sh
        small = right >= 62
        r = np.clip(right, 0, 61)
        up = np.where(right > 0, (sig[i] + (np.int64(1) << r) - 1) >> r, sig[i] << np.clip(sh, 0, 61))
        up = np.where(small, (sig[i] > 0).astype(np.int64), up)
        out[i] = np.where(sig[i] > 0, up, 0)
    return out


def accu_exponents(A: np.ndarray, B: np.ndarray, M: int):
    """OS II-accu exponents: (kappa, tA, tB, b, Ahat, Bhat, Chat).

    C^ = A^ B^ (exact integers) bounds sum_k |a_ik||b_kj| <= 2^(E_i + F_j - 2b) C^_ij.
    With rho_i = max(1, max_j C^_ij), gamma_j = max(1, max_i C^_ij), L as in
    half_range_log2 and x_i = floor((L - ceil(log2 rho_i)) / 2), y_j likewise,
    d_i = x_i - E_i + b and e_j = y_j - F_j + b give
    (|A'||B'|)_ij <= 2^(x_i + y_j) C^_ij <= 2^L <= M/2 - 1, because
    C^_ij <= min(rho_i, gamma_j) <= 2^((ceil log2 rho_i + ceil log2 gamma_j) / 2).
    Returned as t_i = kappa - d_i (kappa = floor(L/2)).
    """
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    q = A.shape[1]
    b = accu_bits(q)
    EA = row_exponents(A)
    EB = row_exponents(B.T)
    Ahat = magnitude_bounds(A, EA, b)
    Bhat = magnitude_bounds(B.T, EB, b)  # n x q
    Chat = exact_int_matmul(Ahat, Bhat.T)
    L = half_range_log2(M)
    kap = L // 2
    rho = np.maximum(Chat.max(axis=1, initial=0), 1)
    gamma = np.maximum(Chat.max(axis=0, initial=0), 1)
    tA = [E if (E is ZERO_ROW or E == "nan") else kap - (L - ceil_log2_int(int(r))) // 2 + E - b
          for E, r in zip(EA, rho)]
    tB = [F if (F is ZERO_ROW or F == "nan") else kap - (L - ceil_log2_int(int(g))) // 2 + F - b
          for F, g in zip(EB, gamma)]
    return kap, tA, tB, b, Ahat, Bhat, Chat


def accu_exponents_sampled(A: np.ndarray, B: np.ndarray, M: int, rows, cols):
    """accu_exponents for selected rows of A and columns of B only (same values).

    rho_i needs row i of C^ in full and gamma_j column j, i.e. A^[i] B^ and A^ B^[:, j]:
    vector-matrix products, cheap enough for sampled checks of large problems.
    """
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    q = A.shape[1]
    b = accu_bits(q)
    EA = row_exponents(A)
    EB = row_exponents(B.T)
    Ahat = magnitude_bounds(A, EA, b).astype(np.float64)  # integers <= 2^7: exact
    BhatT = magnitude_bounds(B.T, EB, b).astype(np.float64)
    L = half_range_log2(M)
    kap = L // 2
    tA, tB = {}, {}
    for i in set(int(r) for r in rows):
        E = EA[i]
        if E is ZERO_ROW or E == "nan":
            tA[i] = E
            continue
        rho = max(int((BhatT @ Ahat[i]).max(initial=0)), 1)  # sums <= 2^24: exact in float64
        tA[i] = kap - (L - ceil_log2_int(rho)) // 2 + E - b
    for j in set(int(c) for c in cols):
        F = EB[j]
        if F is ZERO_ROW or F == "nan":
            tB[j] = F
            continue
        gamma = max(int((Ahat @ BhatT[j]).max(initial=0)), 1)
        tB[j] = kap - (L - ceil_log2_int(gamma)) // 2 + F - b
    return kap, tA, tB


def scaling_exponents(A: np.ndarray, B: np.ndarray, M: int, scaling: str):
    """(k, EA, EB) of a scaling mode: d_i = k - EA_i, e_j = k - EB_j."""
    q = np.asarray(A).shape[1]
    if scaling == "uniform":
        return choose_k(M, q), row_exponents(A), row_exponents(np.asarray(B).T)
    if scaling == "fast":
        return choose_k(M, 1), norm_exponents(A), norm_exponents(np.asarray(B).T)
    if scaling == "accu":
        kap, tA, tB = accu_exponents(A, B, M)[:3]
        return kap, tA, tB
    raise ValueError(f"unknown scaling {scaling!r}")


# --------------------------------------------------------------------------
# Whole method and the direct definition
# --------------------------------------------------------------------------
@dataclass
class Ozaki2Result:
    C: np.ndarray
    k: int
    moduli: list[int]
    EA: list
    EB: list
    d: list[int]
    e: list[int]
    Ap: np.ndarray = None      # A' (object ints)
    Bp: np.ndarray = None      # B' (object ints)
    Ares: np.ndarray = None    # s x m x q int8, symmetric residues of A'
    Bres: np.ndarray = None    # s x q x n int8, symmetric residues of B'
    Cres: np.ndarray = None    # s x m x n, C''_t in [0, m_t)
    C3: np.ndarray = None      # C''' (object ints)


def prepare(A: np.ndarray, B: np.ndarray, s: int, moduli=None, scaling: str = "uniform"):
    """Steps 1-2: parameters, exponents and the truncated integer matrices."""
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    moduli = list(moduli) if moduli is not None else greedy_moduli(s)
    cc = crt_constants(moduli)
    k, EA, EB = scaling_exponents(A, B, cc.M, scaling)
    d = scale_exponents(EA, k)
    e = scale_exponents(EB, k)
    Ap = scaled_trunc_matrix(A, d)
    Bp = scaled_trunc_matrix(B.T, e).T
    return cc, k, EA, EB, d, e, Ap, Bp


def ozaki2_dgemm(A: np.ndarray, B: np.ndarray, s: int, moduli=None, keep=True,
                 scaling: str = "uniform") -> Ozaki2Result:
    """Algorithm 1 of [Ozaki II, §7], steps 1-6, in the pages' order (scaling: §5 or §9)."""
    cc, k, EA, EB, d, e, Ap, Bp = prepare(A, B, s, moduli, scaling)
    Ares = residue_planes(Ap, cc.moduli)
    Bres = residue_planes(Bp, cc.moduli)
    Cres = residue_products(Ares, Bres, cc.moduli)
    C3 = crt_reconstruct(Cres, cc)
    C = unscale(C3, d, e, [x == "nan" for x in EA], [x == "nan" for x in EB])
    r = Ozaki2Result(C, k, cc.moduli, EA, EB, d, e)
    if keep:
        r.Ap, r.Bp, r.Ares, r.Bres, r.Cres, r.C3 = Ap, Bp, Ares, Bres, Cres, C3
    return r


def direct_dgemm(A: np.ndarray, B: np.ndarray, s: int, moduli=None, scaling: str = "uniform") -> np.ndarray:
    """The same result from its definition: RN(2^-(d_i+e_j) * (A'B')_ij), exact integers."""
    cc, k, EA, EB, d, e, Ap, Bp = prepare(A, B, s, moduli, scaling)
    C3 = np.dot(Ap.astype(object), Bp.astype(object))
    return unscale(C3, d, e, [x == "nan" for x in EA], [x == "nan" for x in EB])


def direct_entries(A: np.ndarray, B: np.ndarray, s: int, rows, cols, moduli=None,
                   scaling: str = "uniform") -> np.ndarray:
    """C_ij from the definition for selected (rows[p], cols[p]) pairs only.

    Uses the full row i of A and column j of B (their exponents span all of q),
    so it is cheap enough for sampled checks of large products.
    """
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    moduli = list(moduli) if moduli is not None else greedy_moduli(s)
    cc = crt_constants(moduli)
    if scaling == "accu":
        k, tA, tB = accu_exponents_sampled(A, B, cc.M, rows, cols)
        rowexp = lambda i: tA[int(i)]
        colexp = lambda j: tB[int(j)]
    else:
        if scaling == "uniform":
            k, f = choose_k(cc.M, A.shape[1]), row_exponents
        elif scaling == "fast":
            k, f = choose_k(cc.M, 1), norm_exponents
        else:
            raise ValueError(f"unknown scaling {scaling!r}")
        rowexp = lambda i: f(A[i : i + 1, :])[0]
        colexp = lambda j: f(B[:, j : j + 1].T)[0]
    out = np.empty(len(rows), dtype=np.float64)
    for p, (i, j) in enumerate(zip(rows, cols)):
        Ei = rowexp(i)
        Fj = colexp(j)
        if Ei == "nan" or Fj == "nan":
            out[p] = np.nan
            continue
        di = scale_exponents([Ei], k)[0]
        ej = scale_exponents([Fj], k)[0]
        a = scaled_trunc_matrix(A[i : i + 1, :], [di])[0]
        b = scaled_trunc_matrix(B[:, j : j + 1].T, [ej])[0]
        c3 = int(np.dot(a.astype(object), b.astype(object)))
        out[p] = round_scaled(c3, -(di + ej))
    return out
