"""Full-size workloads on the GPU, in the launch configuration the benchmark times.

At these sizes the oracle cannot compute all of C, so sampled entries are
computed one by one from the definition (full row of A, full column of B, exact
integers) and compared bit for bit; the rest of C is checked through properties
that hold at any size (finite, NaN-free, and within the float64 product's own error
envelope).
"""
import numpy as np
import pytest

from fp64_gemm_emulation_gb300.inputs import hpl_like
from oracle import ozaki2 as O

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def oz():
    from fp64_gemm_emulation_gb300 import ozaki

    return ozaki


def run_ws(oz, A, B, s):
    """The benchmark's configuration: resident inputs, preallocated workspace."""
    m, k = A.shape
    n = B.shape[1]
    dA = torch.from_numpy(A.T.copy()).cuda().t()
    dB = torch.from_numpy(B.T.copy()).cuda().t()
    ws = torch.empty(oz.ozaki2_workspace_bytes(m, n, k, s), dtype=torch.uint8, device="cuda")
    C = oz.ozaki2_dgemm_ws(dA, dB, s, ws)
    torch.cuda.synchronize()
    assert oz.ozaki_get_device_status() == oz.OZ_OK
    del ws
    return C


def sampled_check(oz, A, B, s, C, nsamp=48, seed=0):
    m, n = A.shape[0], B.shape[1]
    rng = np.random.default_rng(seed)
    rows = np.concatenate([[0, m - 1], rng.integers(0, m, nsamp - 2)])
    cols = np.concatenate([[n - 1, 0], rng.integers(0, n, nsamp - 2)])
    got = C[torch.as_tensor(rows, device=C.device), torch.as_tensor(cols, device=C.device)].cpu().numpy()
    want = O.direct_entries(A, B, s, rows, cols)
    assert np.array_equal(got.view(np.int64), want.view(np.int64))
    assert torch.isfinite(C).all()


def test_4096_cube_s14(oz):
    A, B = hpl_like(4096, 4096, 4096, phi=0.5, seed=0)
    C = run_ws(oz, A, B, 14)
    sampled_check(oz, A, B, 14, C)
    # whole-matrix property: error vs the float64 product stays within its envelope
    ref = torch.from_numpy(A.T.copy()).cuda().t() @ torch.from_numpy(B.T.copy()).cuda().t()
    absAB = torch.from_numpy(np.abs(A).T.copy()).cuda().t() @ torch.from_numpy(np.abs(B).T.copy()).cuda().t()
    assert torch.all((C - ref).abs() <= 4096 * 2.0**-52 * absAB)


@pytest.mark.parametrize("phi", [0.0, 1.0, 2.0])
def test_8192_cube_moduli_sweep(oz, phi):
    A, B = hpl_like(8192, 8192, 8192, phi=phi, seed=1)
    for s in (8, 10, 12, 14, 16):
        C = run_ws(oz, A, B, s)
        sampled_check(oz, A, B, s, C, nsamp=24, seed=s)
        del C


@pytest.mark.parametrize("s,phi", [(14, 0.5), (16, 0.5), (14, 4.0)])
def test_16384_cube(oz, s, phi):
    A, B = hpl_like(16384, 16384, 16384, phi=phi, seed=0)
    C = run_ws(oz, A, B, s)
    sampled_check(oz, A, B, s, C, nsamp=32, seed=s)


def test_tall_inner_dimension(oz):
    # k = 2^18 >= 2^17: the INT32 path of the pages would need k-blocking here
    A, B = hpl_like(2048, 2048, 262144, phi=0.5, seed=0)
    C = run_ws(oz, A, B, 14)
    sampled_check(oz, A, B, 14, C, nsamp=16)
