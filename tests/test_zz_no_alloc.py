"""ozaki2_dgemm_noalloc: the product without any device allocation.

Callers that cannot allocate device memory when they multiply (their memory manager
owns the GPU, or they must not allocate after start-up) use this entry point; its
workspace is a fixed 64 MiB buffer inside the library.  It must give exactly the
result of the oracle and of the allocating entry point ozaki2_dgemm, call after call,
even though each call finds the previous call's data in the shared buffer.

This file is collected last on purpose, so that a run stopping at the first failure
has already run every other test.
"""
import numpy as np
import pytest

from fp64_gemm_emulation_gb300.inputs import hpl_like
from oracle import ozaki2 as O

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _dev(X):
    return torch.from_numpy(np.asfortranarray(X).T.copy()).cuda().t()


def _call(lib, name, A, B, s):
    m, k = A.shape
    n = B.shape[1]
    C = torch.full((n, m), np.nan, dtype=torch.float64, device="cuda").t()
    rc = getattr(lib, name)(m, n, k, A.data_ptr(), m, B.data_ptr(), max(1, k), C.data_ptr(), m, s,
                            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return rc, C.t().contiguous().cpu().numpy().T


def _bits(X):
    return np.ascontiguousarray(X).view(np.int64)


def test_noalloc_matches_the_oracle_and_the_allocating_entry_point_on_two_calls_in_a_row():
    from fp64_gemm_emulation_gb300 import ozaki as oz

    lib = oz._lib
    # first a larger problem, then a smaller one that lands on the first one's leftovers
    for (m, n, k, s, phi, seed) in [(700, 650, 760, 14, 0.5, 1), (300, 130, 1000, 12, 2.0, 2)]:
        assert oz.ozaki2_workspace_bytes(m, n, k, s) <= oz.OZ_NOALLOC_SCRATCH_BYTES
        A, B = hpl_like(m, n, k, phi=phi, seed=seed)
        dA, dB = _dev(A), _dev(B)
        rc_ref, C_ref = _call(lib, "ozaki2_dgemm", dA, dB, s)
        rc, C = _call(lib, "ozaki2_dgemm_noalloc", dA, dB, s)
        assert rc_ref == 0 and rc == 0
        # same tolerance as every other parity test here: bit for bit
        assert np.array_equal(_bits(C), _bits(C_ref))
        assert np.array_equal(_bits(C), _bits(O.ozaki2_dgemm(A, B, s).C))
    assert oz.ozaki_get_device_status() == oz.OZ_OK


def test_noalloc_through_the_binding_and_with_an_empty_inner_dimension():
    from fp64_gemm_emulation_gb300 import ozaki as oz

    A, B = hpl_like(257, 300, 130, phi=1.0, seed=3)
    C = oz.ozaki2_dgemm_noalloc(_dev(A), _dev(B), 13)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(C.cpu().numpy()), _bits(O.ozaki2_dgemm(A, B, 13).C))
    # k = 0: C = +0 (BLAS with beta = 0), as ozaki2_dgemm gives, on leftovers of the call above
    dA = torch.empty((0, 40), dtype=torch.float64, device="cuda").t()
    dB = torch.empty((33, 0), dtype=torch.float64, device="cuda").t()
    rc_ref, C_ref = _call(oz._lib, "ozaki2_dgemm", dA, dB, 14)
    rc, C0 = _call(oz._lib, "ozaki2_dgemm_noalloc", dA, dB, 14)
    assert rc_ref == 0 and rc == 0 and C0.shape == (40, 33)
    assert np.array_equal(_bits(C0), _bits(np.zeros((40, 33))))
    assert np.array_equal(_bits(C0), _bits(C_ref))
    assert oz.ozaki_get_device_status() == oz.OZ_OK


def test_noalloc_rejects_problems_beyond_its_buffer():
    from fp64_gemm_emulation_gb300 import ozaki as oz

    m = n = k = 1024
    assert oz.ozaki2_workspace_bytes(m, n, k, 14) > oz.OZ_NOALLOC_SCRATCH_BYTES
    dA = torch.zeros((k, m), dtype=torch.float64, device="cuda").t()
    dB = torch.zeros((n, k), dtype=torch.float64, device="cuda").t()
    C = torch.full((n, m), 3.0, dtype=torch.float64, device="cuda").t()
    rc = oz._lib.ozaki2_dgemm_noalloc(m, n, k, dA.data_ptr(), m, dB.data_ptr(), k, C.data_ptr(), m, 14,
                                      torch.cuda.current_stream().cuda_stream)
    assert rc == oz.OZ_ENOMEM
    assert bool(torch.all(C == 3.0))  # nothing ran
