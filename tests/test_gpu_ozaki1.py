"""Scheme I on the GPU vs the CPU oracle (RN split, triangular products, FP64 sum).

Slices, slice exponents and the INT32 products are integer data and compared bit
for bit; the result C is the same fixed-order sequence of FP64 additions of exact
terms on both sides, so it is compared bit for bit too.
"""
import numpy as np
import pytest

from fp64_gemm_emulation_gb300.inputs import hpl_like, special_matrix
from oracle import ozaki1 as O1
from oracle import ozaki2 as O2

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def oz():
    from fp64_gemm_emulation_gb300 import ozaki

    return ozaki


def dev(X):
    return torch.from_numpy(np.asfortranarray(X).T.copy()).cuda().t()


def host(T):
    return T.t().contiguous().cpu().numpy().T


def bits(x):
    return np.ascontiguousarray(x, dtype=np.float64).view(np.int64)


def bf16_to_int(P):
    u = P.cpu().numpy().astype(np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.int64)


STEP_CASES = [
    # m, n, k, s, phi, seed
    (256, 256, 256, 7, 0.5, 0),
    (300, 520, 1100, 7, 0.5, 1),     # ragged tiles
    (130, 70, 5000, 4, 2.0, 2),      # k > 4096: two exact INT32 chunks
    (64, 96, 40, 10, 4.0, 3),
    (17, 9, 5, 1, 0.5, 4),           # one slice
]


@pytest.mark.parametrize("m,n,k,s,phi,seed", STEP_CASES)
def test_scheme1_steps_bit_exact(oz, m, n, k, s, phi, seed):
    A, B = hpl_like(m, n, k, phi=phi, seed=seed)
    A[3 % m, :] = 0.0  # a zero row
    C_ref, SA, XA, SBt, XB, beta = O1.ozaki1_dgemm(A, B, s)
    assert oz.ozaki1_beta(k) == beta
    dA, dB = dev(A), dev(B)
    Ap, Bp, Ae, Be = oz.ozaki1_split(dA, dB, s)
    Ai, Bi = bf16_to_int(Ap), bf16_to_int(Bp)
    assert np.array_equal(Ai[:, :m, :k], SA)
    assert np.array_equal(Bi[:, :n, :k], SBt)
    assert not Ai[:, m:, :].any() and not Ai[:, :, k:].any()
    assert np.array_equal(Ae.cpu().numpy(), XA)
    assert np.array_equal(Be.cpu().numpy(), XB)

    P = oz.ozaki1_slice_gemm(m, n, k, s, Ap, Bp).cpu().numpy()
    for q, (i, j) in enumerate(O1.triangle_pairs(s)):
        want = O2.exact_int_matmul(SA[i - 1], SBt[j - 1].T)
        assert np.array_equal(P[q, :n, :m].T, want)

    C = oz.ozaki1_accumulate(m, n, k, s, torch.from_numpy(P).cuda(), Ae, Be)
    assert np.array_equal(bits(host(C)), bits(C_ref))
    assert oz.ozaki_get_device_status() == oz.OZ_OK


@pytest.mark.parametrize("s", [1, 2, 3, 7, 8, 12, 20])
def test_scheme1_dgemm_bit_exact(oz, s):
    m, n, k = 150, 110, 700
    A, B = hpl_like(m, n, k, phi=0.5, seed=10 + s)
    C_ref = O1.ozaki1_dgemm(A, B, s)[0]
    C = host(oz.ozaki1_dgemm(dev(A), dev(B), s))
    assert np.array_equal(bits(C), bits(C_ref))


@pytest.mark.parametrize("kind", ["zeros", "pow2", "zero_rows", "ints"])
def test_scheme1_special_inputs(oz, kind):
    A = special_matrix(kind, 130, 270, seed=21)
    B = special_matrix(kind, 270, 70, seed=22)
    C_ref = O1.ozaki1_dgemm(A, B, 7)[0]
    C = host(oz.ozaki1_dgemm(dev(A), dev(B), 7))
    assert np.array_equal(bits(C), bits(C_ref))


def test_scheme1_4096_cube_seven_slices_sampled(oz):
    # the comparison workload: 4096^3, phi = 0.5, s = 7 (28 products)
    m = n = k = 4096
    A, B = hpl_like(m, n, k, phi=0.5, seed=0)
    ws = torch.empty(oz.ozaki1_workspace_bytes(m, n, k, 7), dtype=torch.uint8, device="cuda")
    C = oz.ozaki1_dgemm_ws(dev(A), dev(B), 7, ws)
    rows = np.arange(0, m, 97)[:40]
    cols = np.arange(5, n, 101)[:40]
    # oracle on the sampled rows / columns (slices of a row depend on that row only)
    C_ref = O1.ozaki1_dgemm(A[rows, :], B[:, cols], 7)[0]
    got = C[torch.as_tensor(rows, device="cuda")][:, torch.as_tensor(cols, device="cuda")].cpu().numpy()
    assert np.array_equal(bits(got), bits(C_ref))
    assert oz.ozaki_get_device_status() == oz.OZ_OK
