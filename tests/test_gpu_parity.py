"""GPU path vs the CPU oracle, element by element, through the C ABI (Scheme II).

Bar: bit-exact everywhere.  Exponents, residue planes and C''_t are integer data;
the final C is the single rounding of an exact integer, which both sides take
the same way, so C is compared bit for bit as well (the tolerance
|dC| <= 2^-50 (|A||B|) stated for the emulated product is checked on top as a sanity bound).
"""
from fractions import Fraction

import numpy as np
import pytest

from fp64_gemm_emulation_gb300.inputs import hpl_like, special_matrix
from oracle import ozaki2 as O

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def oz():
    from fp64_gemm_emulation_gb300 import ozaki

    return ozaki


def dev(X):
    """Column-major float64 CUDA tensor from a numpy array."""
    X = np.asfortranarray(X, dtype=np.float64)
    return torch.from_numpy(X.T.copy()).cuda().t()


def host(T):
    return T.t().contiguous().cpu().numpy().T


def exps_as_int32(E):
    out = []
    for e in E:
        if e is O.ZERO_ROW:
            out.append(int(np.int32(np.uint32(0x80808080).view(np.int32))))
        elif e == "nan":
            out.append(0x7FFFFFFF)
        else:
            out.append(e)
    return np.array(out, dtype=np.int32)


def exact_entry(A, B, i, j):
    """(AB)_ij exactly, as a Fraction."""
    return sum((Fraction(float(a)) * Fraction(float(b)) for a, b in zip(A[i, :], B[:, j])), Fraction(0))


def bits(x):
    return np.ascontiguousarray(x, dtype=np.float64).view(np.int64)


def bf16_planes_to_int(P):
    """bf16 bit patterns (int16 tensor) -> integer values."""
    u = P.cpu().numpy().astype(np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.int64)


# ------------------------------------------------------------------ step by step
STEP_CASES = [
    # m, n, k, s, phi, seed
    (256, 256, 256, 14, 0.5, 0),      # the 256^3 workload
    (300, 520, 2100, 14, 0.5, 1),     # several tiles, ragged, 3 k-chunks
    (129, 257, 961, 8, 2.0, 2),       # one past every tile edge, 2 chunks
    (64, 40, 960, 16, 0.0, 3),        # exactly one chunk
    (200, 300, 3000, 20, 4.0, 4),     # widest exponent spread, 20 moduli, 4 chunks
    (17, 9, 5, 2, 0.5, 5),            # tiny, 2 moduli
]


@pytest.mark.parametrize("m,n,k,s,phi,seed", STEP_CASES)
def test_steps_bit_exact(oz, m, n, k, s, phi, seed):
    A, B = hpl_like(m, n, k, phi=phi, seed=seed)
    ref = O.ozaki2_dgemm(A, B, s)
    dA, dB = dev(A), dev(B)

    rowexp, colexp = oz.ozaki2_exponents(dA, dB)
    assert np.array_equal(rowexp.cpu().numpy(), exps_as_int32(ref.EA))
    assert np.array_equal(colexp.cpu().numpy(), exps_as_int32(ref.EB))

    Ap, Bp = oz.ozaki2_split(dA, dB, s, rowexp, colexp)
    Ai, Bi = bf16_planes_to_int(Ap), bf16_planes_to_int(Bp)
    assert np.array_equal(Ai[:, :m, :k], ref.Ares.astype(np.int64))
    assert np.array_equal(Bi[:, :n, :k], np.transpose(ref.Bres, (0, 2, 1)).astype(np.int64))
    assert not Ai[:, m:, :].any() and not Ai[:, :, k:].any()      # zero padding
    assert not Bi[:, n:, :].any() and not Bi[:, :, k:].any()

    # steps a1 + a2 in one call (one pass over each column of B): the same bits
    re2, ce2, Ap2, Bp2 = oz.ozaki2_scale_split(dA, dB, s)
    assert torch.equal(re2, rowexp) and torch.equal(ce2, colexp)
    assert torch.equal(Ap2, Ap) and torch.equal(Bp2, Bp)

    Cr = oz.ozaki2_residue_gemm(m, n, k, s, Ap, Bp)
    got = Cr.cpu().numpy()[:, :n, :m]                               # [s][j][i]
    assert np.array_equal(got, np.transpose(ref.Cres, (0, 2, 1)).astype(np.uint8))

    C = oz.ozaki2_crt(m, n, k, s, Cr, rowexp, colexp)
    assert np.array_equal(bits(host(C)), bits(ref.C))
    assert oz.ozaki_get_device_status() == oz.OZ_OK


# ------------------------------------------------------------------ whole call
E2E_CASES = [
    (256, 256, 256, 14, 0.5, 0),
    (333, 444, 1234, 14, 1.0, 6),
    (96, 80, 70, 10, 0.5, 7),
    (511, 257, 1919, 12, 2.0, 8),
]


@pytest.mark.parametrize("m,n,k,s,phi,seed", E2E_CASES)
def test_dgemm_bit_exact(oz, m, n, k, s, phi, seed):
    A, B = hpl_like(m, n, k, phi=phi, seed=seed)
    ref = O.ozaki2_dgemm(A, B, s, keep=False).C
    C = oz.ozaki2_dgemm(dev(A), dev(B), s)
    assert np.array_equal(bits(host(C)), bits(ref))
    # The stated tolerance |dC| <= 2^-50 (|A||B|) is about GPU vs oracle: dC = 0 here.
    # Against the exact product, the error must stay inside the truncation bound
    # 2^-(d_i+e_j) sum_k (|a'_ik| + |b'_kj| + 1) plus half an ulp (sampled entries).
    cc, kA, EA, EB, d, e, Ap, Bp = O.prepare(A, B, s)
    Ch = host(C)
    rng = np.random.default_rng(seed)
    for i, j in zip(rng.integers(0, m, 16), rng.integers(0, n, 16)):
        exact = exact_entry(A, B, i, j)
        bound = Fraction(sum(abs(int(Ap[i, q])) + abs(int(Bp[q, j])) + 1 for q in range(k))) \
            * Fraction(2) ** -(d[i] + e[j])
        half_ulp = Fraction(np.spacing(abs(Ch[i, j]))) / 2
        assert abs(Fraction(float(Ch[i, j])) - exact) <= bound + half_ulp


@pytest.mark.parametrize("s", list(range(2, 21)))
def test_every_moduli_count(oz, s):
    m, n, k = 70, 90, 40
    A, B = hpl_like(m, n, k, phi=0.5, seed=100 + s)
    ref = O.ozaki2_dgemm(A, B, s, keep=False).C
    C = oz.ozaki2_dgemm(dev(A), dev(B), s)
    assert np.array_equal(bits(host(C)), bits(ref))


@pytest.mark.parametrize("kind", ["zeros", "pow2", "subnormal", "zero_rows", "ints", "huge"])
def test_special_inputs(oz, kind):
    A = special_matrix(kind, 130, 270, seed=11)
    B = special_matrix(kind if kind != "huge" else "pow2", 270, 70, seed=12)
    ref = O.ozaki2_dgemm(A, B, 14, keep=False).C
    C = oz.ozaki2_dgemm(dev(A), dev(B), 14)
    assert np.array_equal(bits(host(C)), bits(ref))


def test_overflow_and_underflow_edges(oz):
    # products beyond DBL_MAX give inf; products far below the subnormal range give 0
    A = np.asfortranarray(np.full((3, 2), 2.0**600))
    B = np.asfortranarray(np.array([[2.0**500, 2.0**-700, -(2.0**-1000)], [2.0**500, 2.0**-700, 0.0]]))
    A[2, :] = [2.0**-600, -(2.0**-600)]
    ref = O.ozaki2_dgemm(A, B, 14, keep=False).C
    C = oz.ozaki2_dgemm(dev(A), dev(B), 14)
    assert np.array_equal(bits(host(C)), bits(ref))
    assert np.isinf(ref[0, 0])


def test_non_finite_inputs(oz):
    A, B = hpl_like(40, 30, 50, seed=13)
    A[5, 7] = np.inf
    A[9, 0] = np.nan
    B[3, 11] = -np.inf
    ref = O.ozaki2_dgemm(A, B, 14, keep=False).C
    C = host(oz.ozaki2_dgemm(dev(A), dev(B), 14))
    assert np.array_equal(bits(C), bits(ref))
    assert np.isnan(C[5]).all() and np.isnan(C[:, 11]).all()


def test_k_zero_gives_zeros(oz):
    dA = torch.empty((5, 0), dtype=torch.float64, device="cuda")
    dB = torch.empty((0, 4), dtype=torch.float64, device="cuda")
    C = torch.full((4, 5), 7.0, dtype=torch.float64, device="cuda").t()
    lib = oz._lib
    rc = lib.ozaki2_dgemm(5, 4, 0, dA.data_ptr(), 5, dB.data_ptr(), 1, C.data_ptr(), 5, 14,
                          torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    assert np.all(bits(host(C)) == 0)


def test_leading_dimensions_and_views(oz):
    m, n, k = 150, 130, 300
    A, B = hpl_like(m, n, k, seed=14)
    big_A = np.zeros((m + 13, k), order="F")
    big_A[:m] = A
    big_B = np.zeros((k + 5, n), order="F")
    big_B[:k] = B
    dA = dev(big_A)[:m]
    dB = dev(big_B)[:k]
    Cbig = torch.full((n, m + 7), -1.0, dtype=torch.float64, device="cuda").t()
    C = oz.ozaki2_dgemm(dA, dB, 14, C=Cbig[:m])
    ref = O.ozaki2_dgemm(A, B, 14, keep=False).C
    assert np.array_equal(bits(host(C)), bits(ref))
    assert torch.all(Cbig[m:] == -1.0)          # padding rows of C untouched


def test_ws_and_host_variants_agree(oz):
    m, n, k = 200, 210, 900
    A, B = hpl_like(m, n, k, seed=15)
    ref = O.ozaki2_dgemm(A, B, 14, keep=False).C
    ws = torch.empty(oz.ozaki2_workspace_bytes(m, n, k, 14), dtype=torch.uint8, device="cuda")
    C1 = host(oz.ozaki2_dgemm_ws(dev(A), dev(B), 14, ws))
    C2 = oz.ozaki2_dgemm_host(A, B, 14)
    assert np.array_equal(bits(C1), bits(ref))
    assert np.array_equal(bits(C2), bits(ref))


def test_deterministic_repeats(oz):
    A, B = hpl_like(640, 520, 2000, seed=16)
    dA, dB = dev(A), dev(B)
    outs = [bits(host(oz.ozaki2_dgemm(dA, dB, 14))) for _ in range(3)]
    assert all(np.array_equal(outs[0], o) for o in outs[1:])


def test_host_pipeline_blocks_match_device_path(oz):
    # m >= 4096 and n >= 2048: the host entry point splits A into 2 row blocks and B into
    # 2 column blocks (ragged last blocks) and overlaps copies with compute; the result
    # must equal the device-resident entry point bit for bit, with padded leading dims.
    m, n, k = 4300, 2600, 700
    A, B = hpl_like(m, n, k, phi=1.0, seed=17)
    Ah = np.zeros((m + 5, k), order="F")
    Ah[:m] = A
    Bh = np.zeros((k + 3, n), order="F")
    Bh[:k] = B
    Ch = np.full((m + 7, n), -2.0, order="F")
    rc = oz._lib.ozaki2_dgemm_host(m, n, k, Ah.ctypes.data, m + 5, Bh.ctypes.data, k + 3, Ch.ctypes.data, m + 7, 14)
    assert rc == 0
    ref = host(oz.ozaki2_dgemm(dev(A), dev(B), 14))
    assert np.array_equal(bits(Ch[:m]), bits(ref))
    assert np.all(Ch[m:] == -2.0)
    # sampled entries against the oracle as well
    rows, cols = [0, m - 1, 4095, 4096, 17], [n - 1, 0, 2047, 2048, 1000]
    want = O.direct_entries(A, B, 14, rows, cols)
    assert np.array_equal(bits(Ch[rows, cols]), bits(want))


def test_host_pipeline_four_by_two_blocks(oz):
    # m >= 12288: four row blocks (ragged last), n = 2100: two column blocks; the blocks are
    # computed in the order their operands arrive (A_0, B_0, A_1, B_1, A_2, A_3)
    m, n, k = 12300, 2100, 300
    A, B = hpl_like(m, n, k, phi=0.5, seed=18)
    Ch = np.empty((m, n), order="F")
    rc = oz._lib.ozaki2_dgemm_host(m, n, k, A.ctypes.data, m, B.ctypes.data, k, Ch.ctypes.data, m, 14)
    assert rc == 0
    ref = host(oz.ozaki2_dgemm(dev(A), dev(B), 14))
    assert np.array_equal(bits(Ch), bits(ref))


def test_concurrent_calls_on_two_streams(oz):
    # two products at once on two streams (the second launch's CTA pairs wait for SMs the first
    # one holds): both results exact, no device-status error
    pairs = [hpl_like(1300, 1200, 2100, phi=0.5, seed=19), hpl_like(1000, 1500, 1700, phi=2.0, seed=20)]
    refs = [O.ozaki2_dgemm(A, B, 14, keep=False).C for A, B in pairs]
    dev_in = [(dev(A), dev(B)) for A, B in pairs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [None, None]
    torch.cuda.synchronize()
    for i in range(2):
        with torch.cuda.stream(streams[i]):
            outs[i] = oz.ozaki2_dgemm(dev_in[i][0], dev_in[i][1], 14)
    torch.cuda.synchronize()
    for C, ref in zip(outs, refs):
        assert np.array_equal(bits(host(C)), bits(ref))
    assert oz.ozaki_get_device_status() == oz.OZ_OK


@pytest.mark.parametrize("s", [2, 8, 14, 16, 20])
def test_crt_on_random_residue_tuples(oz, s):
    # Any residue tuple is a valid input of the CRT step.  With uniform residues Z/M has a
    # uniform fractional part, so about 1 element in 128 lies near +-M/2 (the quotient
    # estimate's corrected case), and the rows at the ends of the exponent range put the
    # results across the subnormal and the overflow boundaries.
    m, n, k = 301, 203, 1024
    moduli = O.greedy_moduli(s)
    cc = O.crt_constants(moduli)
    kA = O.choose_k(cc.M, k)
    bm = cc.M.bit_length()
    rng = np.random.default_rng(1000 + s)
    Cres = np.stack([rng.integers(0, mt, size=(m, n)) for mt in moduli])
    E = rng.integers(-40, 41, m)
    F = rng.integers(-40, 41, n)
    # D = 2 kA - E - F: about bm + 1074 puts |X| 2^-D at the bottom of the subnormals,
    # about bm - 1025 at the top of the normal range
    E[:80] = 2 * kA - (bm + 1030) - rng.integers(-45, 46, 80)
    E[80:140] = 2 * kA - (bm - 1026) - rng.integers(-3, 4, 60)
    F[:40] = 0
    E[140], E[141] = oz.OZ_EXP_EMPTY, oz.OZ_EXP_NONFINITE
    F[50], F[51] = oz.OZ_EXP_EMPTY, oz.OZ_EXP_NONFINITE
    X = O.crt_reconstruct(Cres, cc)
    live_r = (E != oz.OZ_EXP_EMPTY) & (E != oz.OZ_EXP_NONFINITE)
    live_c = (F != oz.OZ_EXP_EMPTY) & (F != oz.OZ_EXP_NONFINITE)
    d = [int(kA - e) if ok else 0 for e, ok in zip(E, live_r)]
    e = [int(kA - f) if ok else 0 for f, ok in zip(F, live_c)]
    ref = O.unscale(X, d, e)
    ref[E == oz.OZ_EXP_EMPTY, :] = 0.0
    ref[:, F == oz.OZ_EXP_EMPTY] = 0.0
    ref[E == oz.OZ_EXP_NONFINITE, :] = np.nan
    ref[:, F == oz.OZ_EXP_NONFINITE] = np.nan
    mp, np_, _ = oz.ozaki2_plane_dims(m, n, k)
    Cr = np.zeros((s, np_, mp), dtype=np.uint8)
    Cr[:, :n, :m] = np.transpose(Cres, (0, 2, 1))
    rowexp = torch.from_numpy(E.astype(np.int32)).cuda()
    colexp = torch.from_numpy(F.astype(np.int32)).cuda()
    C = host(oz.ozaki2_crt(m, n, k, s, torch.from_numpy(Cr).cuda(), rowexp, colexp))
    got, want = bits(C), bits(ref)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(C), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # the sample really spans the cases: subnormal, infinite and near-M/2 results
    fin = ref[live_r][:, live_c]
    assert (np.abs(fin[fin != 0]) < 2.0**-1022).any() and np.isinf(fin).any()
    near = np.abs(np.abs(X.astype(float)) / float(cc.M) - 0.5) < 2.0**-8
    assert near.sum() > 20


@pytest.mark.parametrize("s,k", [(20, 3000), (20, 40), (16, 16), (17, 4096)])
def test_split_with_large_shifts(oz, s, k):
    # k_A above 62 (17 or more moduli, or 16 with a small k) makes a' = u 2^p with p > 10
    # (the six-limb residue path); rows and columns whose maximum is a small subnormal reach
    # p close to k_A, past 43 at 20 moduli (the per-bit fallback)
    m, n = 96, 72
    A, B = hpl_like(m, n, k, phi=4.0, seed=s + k)
    rng = np.random.default_rng(s * k)
    A[3, :] = rng.integers(-3, 4, k) * 2.0**-1074
    A[5, :] = rng.integers(-(2**20), 2**20, k) * 2.0**-1074
    A[6, :] *= 2.0**-1060
    B[:, 7] = rng.integers(-3, 4, k) * 2.0**-1074
    B[:, 9] *= 2.0**-1050
    ref = O.ozaki2_dgemm(A, B, s)
    assert ref.k > 52
    dA, dB = dev(A), dev(B)
    rowexp, colexp = oz.ozaki2_exponents(dA, dB)
    Ap, Bp = oz.ozaki2_split(dA, dB, s, rowexp, colexp)
    assert np.array_equal(bf16_planes_to_int(Ap)[:, :m, :k], ref.Ares.astype(np.int64))
    assert np.array_equal(bf16_planes_to_int(Bp)[:, :n, :k], np.transpose(ref.Bres, (0, 2, 1)).astype(np.int64))
    C = oz.ozaki2_dgemm(dA, dB, s)
    assert np.array_equal(bits(host(C)), bits(ref.C))


# the one-pass split of B holds 8, 16 or 32 values a thread (Kp up to 4096, 8192, 16384); above
# that the two-pass path runs.  Every width, ragged k, special values and padding columns:
@pytest.mark.parametrize("m,n,k,s,seed", [(40, 300, 4000, 14, 11), (70, 257, 8100, 12, 12),
                                          (33, 130, 16384, 16, 13), (20, 70, 16400, 14, 14)])
def test_scale_split_matches_the_oracle_at_every_width(oz, m, n, k, s, seed):
    A, B = hpl_like(m, n, k, phi=1.0, seed=seed)
    B[:, 3] = 0.0                                   # an empty column
    B[5, 7] = 2.0**-1070                            # a subnormal, and a column led by one
    B[:, 9] = 0.0
    B[123, 9] = -(2.0**-1060)
    B[17, 11] = np.inf                              # a non-finite column
    ref = O.prepare(A, B, s)
    cc, kA, EA, EB, d, e, Apv, Bpv = ref
    dA, dB = dev(A), dev(B)
    rowexp, colexp, Ap, Bp = oz.ozaki2_scale_split(dA, dB, s)
    assert np.array_equal(rowexp.cpu().numpy(), exps_as_int32(EA))
    assert np.array_equal(colexp.cpu().numpy(), exps_as_int32(EB))
    Bi = bf16_planes_to_int(Bp)
    want = np.transpose(O.residue_planes(Bpv, cc.moduli), (0, 2, 1)).astype(np.int64)
    ok_cols = [j for j in range(n) if EB[j] != "nan"]  # a non-finite column's planes are not used
    assert np.array_equal(Bi[:, ok_cols, :k], want[:, ok_cols, :])
    assert not Bi[:, n:, :].any() and not Bi[:, :, k:].any()
    Ai = bf16_planes_to_int(Ap)
    assert np.array_equal(Ai[:, :m, :k], O.residue_planes(Apv, cc.moduli).astype(np.int64))
    assert oz.ozaki_get_device_status() == oz.OZ_OK
