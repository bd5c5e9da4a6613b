"""OS II-fast and OS II-accu on the GPU vs the oracle, bit for bit, through the C ABI.

The exponents are integer data and every later step is exact, so the bar is
bit-exact everywhere: exponent codes, residue planes, final C.
"""
import numpy as np
import pytest

from fp64_gemm_emulation_gb300.inputs import hpl_like, special_matrix
from oracle import ozaki2 as O

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

SCALINGS = ["fast", "accu"]


@pytest.fixture(scope="module")
def oz():
    from fp64_gemm_emulation_gb300 import ozaki

    return ozaki


def dev(X):
    X = np.asfortranarray(X, dtype=np.float64)
    return torch.from_numpy(X.T.copy()).cuda().t()


def host(T):
    return T.t().contiguous().cpu().numpy().T


def bits(x):
    return np.ascontiguousarray(x, dtype=np.float64).view(np.int64)


def codes(E):
    out = []
    for e in E:
        if e is O.ZERO_ROW:
            out.append(int(np.uint32(0x80808080).view(np.int32)))
        elif e == "nan":
            out.append(0x7FFFFFFF)
        else:
            out.append(e)
    return np.array(out, dtype=np.int32)


def bf16_to_int(P):
    u = P.cpu().numpy().astype(np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.int64)


STEP_CASES = [
    # m, n, k, s, phi, seed
    (256, 256, 256, 14, 0.5, 0),
    (300, 520, 2100, 14, 4.0, 1),     # several tiles, ragged, wide exponent range
    (129, 257, 961, 8, 2.0, 2),
    (17, 9, 5, 3, 0.5, 5),
    (200, 300, 3000, 20, 4.0, 4),
]


@pytest.mark.parametrize("scaling", SCALINGS)
@pytest.mark.parametrize("m,n,k,s,phi,seed", STEP_CASES)
def test_steps_bit_exact(oz, scaling, m, n, k, s, phi, seed):
    A, B = hpl_like(m, n, k, phi=phi, seed=seed)
    ref = O.ozaki2_dgemm(A, B, s, scaling=scaling)
    dA, dB = dev(A), dev(B)
    rowexp, colexp = oz.ozaki2_exponents_ex(dA, dB, s, scaling)
    assert np.array_equal(rowexp.cpu().numpy(), codes(ref.EA))
    assert np.array_equal(colexp.cpu().numpy(), codes(ref.EB))
    Ap, Bp = oz.ozaki2_split_ex(dA, dB, s, rowexp, colexp, scaling)
    assert np.array_equal(bf16_to_int(Ap)[:, :m, :k], ref.Ares.astype(np.int64))
    assert np.array_equal(bf16_to_int(Bp)[:, :n, :k], np.transpose(ref.Bres, (0, 2, 1)).astype(np.int64))
    Cr = oz.ozaki2_residue_gemm(m, n, k, s, Ap, Bp)
    assert np.array_equal(Cr.cpu().numpy()[:, :n, :m], np.transpose(ref.Cres, (0, 2, 1)).astype(np.uint8))
    C = oz.ozaki2_crt_ex(m, n, k, s, Cr, rowexp, colexp, scaling)
    assert np.array_equal(bits(host(C)), bits(ref.C))
    assert oz.ozaki_get_device_status() == oz.OZ_OK


@pytest.mark.parametrize("scaling", SCALINGS)
@pytest.mark.parametrize("s", list(range(2, 21)))
def test_every_moduli_count(oz, scaling, s):
    A, B = hpl_like(70, 90, 40, phi=1.0, seed=200 + s)
    ref = O.ozaki2_dgemm(A, B, s, keep=False, scaling=scaling).C
    C = oz.ozaki2_dgemm_ex(dev(A), dev(B), s, scaling)
    assert np.array_equal(bits(host(C)), bits(ref))


@pytest.mark.parametrize("scaling", SCALINGS)
@pytest.mark.parametrize("kind", ["zeros", "pow2", "subnormal", "zero_rows", "ints", "huge"])
def test_special_inputs(oz, scaling, kind):
    A = special_matrix(kind, 130, 270, seed=11)
    B = special_matrix(kind if kind != "huge" else "pow2", 270, 70, seed=12)
    ref = O.ozaki2_dgemm(A, B, 14, keep=False, scaling=scaling).C
    C = oz.ozaki2_dgemm_ex(dev(A), dev(B), 14, scaling)
    assert np.array_equal(bits(host(C)), bits(ref))


@pytest.mark.parametrize("scaling", SCALINGS)
def test_non_finite_inputs(oz, scaling):
    A, B = hpl_like(40, 30, 50, seed=13)
    A[5, 7] = np.inf
    A[9, 0] = np.nan
    B[3, 11] = -np.inf
    ref = O.ozaki2_dgemm(A, B, 14, keep=False, scaling=scaling).C
    C = host(oz.ozaki2_dgemm_ex(dev(A), dev(B), 14, scaling))
    assert np.array_equal(bits(C), bits(ref))
    assert np.isnan(C[5]).all() and np.isnan(C[:, 11]).all()


@pytest.mark.parametrize("q", [1024, 4096, 16384])
def test_accu_bound_product_at_the_fp32_limit(oz, q):
    # every magnitude is 2^b: C^ = q 4^b = 2^24 exactly, the largest value the single
    # FP32 accumulation must hold
    A = np.full((300, q), 2.0**-5)
    B = np.full((q, 260), -(2.0**7))
    A[7, 3] = 0.75 * 2.0**-5  # one row slightly below the bound
    b = O.accu_bits(q)
    assert q * 4**b == 2**24
    ref = O.ozaki2_dgemm(A, B, 14, keep=False, scaling="accu")
    rowexp, colexp = oz.ozaki2_exponents_ex(dev(A), dev(B), 14, "accu")
    assert np.array_equal(rowexp.cpu().numpy(), codes(ref.EA))
    assert np.array_equal(colexp.cpu().numpy(), codes(ref.EB))
    C = oz.ozaki2_dgemm_ex(dev(A), dev(B), 14, "accu")
    assert np.array_equal(bits(host(C)), bits(ref.C))


@pytest.mark.parametrize("scaling", SCALINGS)
def test_leading_dimensions_and_workspace(oz, scaling):
    m, n, k = 150, 130, 300
    A, B = hpl_like(m, n, k, phi=2.0, seed=14)
    big_A = np.zeros((m + 13, k), order="F")
    big_A[:m] = A
    big_B = np.zeros((k + 5, n), order="F")
    big_B[:k] = B
    dA = dev(big_A)[:m]
    dB = dev(big_B)[:k]
    Cbig = torch.full((n, m + 7), -1.0, dtype=torch.float64, device="cuda").t()
    ws = torch.empty(oz.ozaki2_workspace_bytes_ex(m, n, k, 14, scaling), dtype=torch.uint8, device="cuda")
    C = oz.ozaki2_dgemm_ex_ws(dA, dB, 14, scaling, ws, C=Cbig[:m])
    ref = O.ozaki2_dgemm(A, B, 14, keep=False, scaling=scaling).C
    assert np.array_equal(bits(host(C)), bits(ref))
    assert torch.all(Cbig[m:] == -1.0)


def test_uniform_mode_of_ex_equals_the_plain_entry_point(oz):
    A, B = hpl_like(333, 444, 1234, phi=1.0, seed=6)
    dA, dB = dev(A), dev(B)
    C1 = host(oz.ozaki2_dgemm(dA, dB, 14))
    C2 = host(oz.ozaki2_dgemm_ex(dA, dB, 14, "uniform"))
    assert np.array_equal(bits(C1), bits(C2))


@pytest.mark.parametrize("phi", [2.0, 4.0])
def test_accuracy_order_on_the_gpu(oz, phi):
    # the section 9 claim on the GPU results: accu <= fast < uniform in error vs A B
    A, B = hpl_like(256, 256, 1024, phi=phi, seed=31)
    dA, dB = dev(A), dev(B)
    exact = A @ B  # float64: far more accurate than 8 moduli
    scale = np.abs(A) @ np.abs(B)
    err = {sc: np.median(np.abs(host(oz.ozaki2_dgemm_ex(dA, dB, 8, sc)) - exact) / scale)
           for sc in ("uniform", "fast", "accu")}
    assert err["accu"] <= err["fast"] < err["uniform"]


# ------------------------------------------------------------------ full sizes, sampled
FULL = [
    # m, n, k, s, phi, scaling
    (4096, 4096, 4096, 14, 0.5, "accu"),
    (4096, 4096, 4096, 14, 0.5, "fast"),
    (8192, 8192, 8192, 14, 4.0, "accu"),
    (16384, 16384, 16384, 14, 0.5, "accu"),
    (16384, 16384, 16384, 14, 4.0, "fast"),
    (2048, 2048, 262144, 14, 0.5, "accu"),
]


@pytest.mark.parametrize("m,n,k,s,phi,scaling", FULL)
def test_full_size_sampled(oz, m, n, k, s, phi, scaling):
    A, B = hpl_like(m, n, k, phi=phi, seed=0)
    dA, dB = dev(A), dev(B)
    ws = torch.empty(oz.ozaki2_workspace_bytes_ex(m, n, k, s, scaling), dtype=torch.uint8, device="cuda")
    C = oz.ozaki2_dgemm_ex_ws(dA, dB, s, scaling, ws)
    rowexp, colexp = oz.ozaki2_exponents_ex(dA, dB, s, scaling)
    assert oz.ozaki_get_device_status() == oz.OZ_OK
    rng = np.random.default_rng(1)
    rows = [0, m - 1] + list(rng.integers(0, m, 10))
    cols = [n - 1, 0] + list(rng.integers(0, n, 10))
    want = O.direct_entries(A, B, s, rows, cols, scaling=scaling)
    got = C[rows, cols].cpu().numpy()
    assert np.array_equal(bits(got), bits(want))
    # the sampled rows' and columns' exponents themselves
    M = O.crt_constants(O.greedy_moduli(s)).M
    if scaling == "accu":
        _, tA, tB = O.accu_exponents_sampled(A, B, M, rows, cols)
        assert all(int(rowexp[i]) == tA[int(i)] for i in rows)
        assert all(int(colexp[j]) == tB[int(j)] for j in cols)
    else:
        assert all(int(rowexp[i]) == O.norm_exponents(A[i : i + 1])[0] for i in rows)
        assert all(int(colexp[j]) == O.norm_exponents(B[:, j : j + 1].T)[0] for j in cols)
    del ws, C
    torch.cuda.empty_cache()
