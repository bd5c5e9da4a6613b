"""Scheme I EF / Hybrid on the GPU vs the oracle, bit for bit, through the C ABI.

Slices and their exponents are integer data, the group batches are exact INT32 sums,
and the FP64 accumulation follows the oracle's order, so the bar is bit-exact for the
slices, the products and C.
"""
import numpy as np
import pytest

from fp64_gemm_emulation_gb300.inputs import hpl_like, special_matrix
from oracle import ozaki1 as O1

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

VARIANTS = ["ef", "hybrid"]


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


def bf16_to_int(P):
    u = P.cpu().numpy().astype(np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.int64)


def oracle_pair_products(SA, SBt, s, q, beta):
    """The pair products in the variant's order (groups ascending), exact."""
    return [O1.exact_int_matmul(SA[i - 1], SBt[j - 1].T)
            for g, pairs in O1.group_batches(s, O1.group_r(q, beta)) for i, j in pairs]


CASES = [
    # m, n, k, s, phi, seed
    (256, 256, 256, 7, 0.5, 0),
    (300, 200, 1100, 7, 1.0, 1),     # several tiles, ragged, more than one EF chunk
    (129, 257, 4100, 5, 2.0, 2),     # k past a RN/Hybrid chunk
    (40, 33, 17, 9, 0.5, 3),
    (64, 70, 300, 12, 0.5, 4),
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("m,n,k,s,phi,seed", CASES)
def test_steps_bit_exact(oz, variant, m, n, k, s, phi, seed):
    A, B = hpl_like(m, n, k, phi=phi, seed=seed)
    C_ref, SA, XA, SBt, XB, beta = O1.ozaki1_dgemm_variant(A, B, s, variant)
    Ap, Bp, Ae, Be = oz.ozaki1_split_ex(dev(A), dev(B), s, variant)
    assert np.array_equal(bf16_to_int(Ap)[:, :m, :k], SA)
    assert np.array_equal(bf16_to_int(Bp)[:, :n, :k], SBt)
    assert not bf16_to_int(Ap)[:, m:, :].any() and not bf16_to_int(Ap)[:, :, k:].any()
    assert np.array_equal(Ae.cpu().numpy(), XA.astype(np.int32))
    assert np.array_equal(Be.cpu().numpy(), XB.astype(np.int32))
    P = oz.ozaki1_slice_gemm_ex(m, n, k, s, variant, Ap, Bp)
    want = oracle_pair_products(SA, SBt, s, k, beta)
    assert P.shape[0] == len(want)
    for t, w in enumerate(want):
        assert np.array_equal(P[t].cpu().numpy()[:n, :m].T, w.astype(np.int32))
    C = oz.ozaki1_accumulate_ex(m, n, k, s, variant, P, Ae, Be)
    assert np.array_equal(bits(host(C)), bits(C_ref))
    assert oz.ozaki_get_device_status() == oz.OZ_OK


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("s", list(range(1, 13)))
def test_every_slice_count(oz, variant, s):
    A, B = hpl_like(70, 90, 40, phi=1.0, seed=300 + s)
    C_ref = O1.ozaki1_dgemm_variant(A, B, s, variant)[0]
    C = oz.ozaki1_dgemm_ex(dev(A), dev(B), s, variant)
    assert np.array_equal(bits(host(C)), bits(C_ref))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("kind", ["zeros", "pow2", "zero_rows", "ints"])
def test_special_inputs(oz, variant, kind):
    A = special_matrix(kind, 130, 270, seed=11)
    B = special_matrix(kind, 270, 70, seed=12)
    C_ref = O1.ozaki1_dgemm_variant(A, B, 6, variant)[0]
    C = oz.ozaki1_dgemm_ex(dev(A), dev(B), 6, variant)
    assert np.array_equal(bits(host(C)), bits(C_ref))


def test_ef_subnormal_inputs(oz):
    A = special_matrix("subnormal", 130, 270, seed=11)
    B = special_matrix("subnormal", 270, 70, seed=12)
    C_ref = O1.ozaki1_dgemm_variant(A, B, 4, "ef")[0]
    C = oz.ozaki1_dgemm_ex(dev(A), dev(B), 4, "ef")
    assert np.array_equal(bits(host(C)), bits(C_ref))


@pytest.mark.parametrize("k", [1024, 2048, 4096])
def test_ef_worst_case_fields_stay_exact(oz, k):
    # every field 127: EF chunks of 2^(24 - 2 beta) = 1024 k hold 1024 * 127^2 < 2^24
    A = np.full((256, k), 2.0 - 2.0**-52)
    B = np.full((k, 256), -(2.0 - 2.0**-52))
    A[3, :5] = 1.5
    C_ref, SA, XA, SBt, XB, beta = O1.ozaki1_dgemm_variant(A, B, 3, "ef")
    assert beta == 7 and (np.abs(SA[:, 4]) == 127).all()
    C = oz.ozaki1_dgemm_ex(dev(A), dev(B), 3, "ef")
    assert np.array_equal(bits(host(C)), bits(C_ref))


def test_ef_int32_batches_at_the_limit(oz):
    # q = 2^17: beta = 7, r = 1, one worst-case product sums to q 127^2 (just below 2^31)
    q = 2**17
    A = np.full((256, q), 2.0 - 2.0**-52)
    B = np.full((q, 256), 2.0 - 2.0**-52)
    C_ref = O1.ozaki1_dgemm_variant(A[:2], B[:, :2], 2, "ef")[0]
    C = host(oz.ozaki1_dgemm_ex(dev(A), dev(B), 2, "ef"))
    assert np.array_equal(bits(C[:2, :2]), bits(C_ref))


@pytest.mark.parametrize("variant", VARIANTS + ["rn"])
def test_leading_dimensions_and_workspace(oz, variant):
    m, n, k = 150, 130, 300
    A, B = hpl_like(m, n, k, phi=1.0, seed=14)
    big_A = np.zeros((m + 13, k), order="F")
    big_A[:m] = A
    big_B = np.zeros((k + 5, n), order="F")
    big_B[:k] = B
    Cbig = torch.full((n, m + 7), -1.0, dtype=torch.float64, device="cuda").t()
    ws = torch.empty(oz.ozaki1_workspace_bytes_ex(m, n, k, 7, variant), dtype=torch.uint8, device="cuda")
    C = oz.ozaki1_dgemm_ex_ws(dev(big_A)[:m], dev(big_B)[:k], 7, variant, ws, C=Cbig[:m])
    C_ref = O1.ozaki1_dgemm_variant(A, B, 7, variant)[0]
    assert np.array_equal(bits(host(C)), bits(C_ref))
    assert torch.all(Cbig[m:] == -1.0)


@pytest.mark.parametrize("m,n,k,s,variant", [(4096, 4096, 4096, 7, "ef"), (4096, 4096, 4096, 7, "hybrid"),
                                             (8192, 8192, 8192, 8, "ef"), (2048, 2048, 65536, 6, "hybrid")])
def test_full_size_sampled(oz, m, n, k, s, variant):
    A, B = hpl_like(m, n, k, phi=0.5, seed=0)
    C = oz.ozaki1_dgemm_ex(dev(A), dev(B), s, variant)
    assert oz.ozaki_get_device_status() == oz.OZ_OK
    rng = np.random.default_rng(2)
    rows = np.array([0, m - 1] + list(rng.integers(0, m, 8)))
    cols = np.array([n - 1, 0] + list(rng.integers(0, n, 8)))
    # C_ij depends on row i of A and column j of B only (their own maxima)
    want = O1.ozaki1_dgemm_variant(A[rows], B[:, cols], s, variant)[0]
    got = C[torch.as_tensor(rows, device="cuda")][:, torch.as_tensor(cols, device="cuda")].cpu().numpy()
    assert np.array_equal(bits(got), bits(want))
    del C
    torch.cuda.empty_cache()
