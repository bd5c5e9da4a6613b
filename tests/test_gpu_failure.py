"""Failure detection on the GPU without a fault: a bounded wait made to expire.

Every wait inside the tensor-core GEMM is bounded; when one expires the kernel records
OZ_ETIMEOUT in the device status word, stops both CTAs of its pair, accounts for every
copy and MMA it issued, frees its tensor memory and returns, so the context stays usable.
Here the epilogue's accumulator wait is given a zero limit (it gives up as soon as the
accumulator is not ready, which it never is at a tile's first chunk), the status word
must report the expiry, and the next call with the default limit must be bit-exact
against the oracle.  Nothing faults, traps or hangs: the limit only shortens a wait.
"""
import numpy as np
import pytest

from fp64_gemm_emulation_gb300.inputs import hpl_like
from oracle import ozaki1 as O1
from oracle import ozaki2 as O

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _dev(X):
    return torch.from_numpy(np.asfortranarray(X).T.copy()).cuda().t()


def _host(T):
    return T.t().contiguous().cpu().numpy().T


def _bits(X):
    return np.ascontiguousarray(X).view(np.int64)


@pytest.fixture
def oz():
    from fp64_gemm_emulation_gb300 import ozaki

    assert ozaki.ozaki_get_device_status() == ozaki.OZ_OK
    yield ozaki
    ozaki.ozaki_set_epilogue_wait_ns(-1)
    ozaki.ozaki_get_device_status()


def test_expired_epilogue_wait_in_scheme2_is_reported_and_the_next_call_is_exact(oz):
    m, n, k, s = 600, 520, 3000, 14
    A, B = hpl_like(m, n, k, phi=0.5, seed=71)
    dA, dB = _dev(A), _dev(B)
    oz.ozaki_set_epilogue_wait_ns(0)
    for _ in range(2):  # twice in a row: the first expiry leaves nothing behind
        oz.ozaki2_dgemm(dA, dB, s)
        assert oz.ozaki_get_device_status() == oz.OZ_ETIMEOUT
        assert oz.ozaki_get_device_status() == oz.OZ_OK  # the read cleared it
    oz.ozaki_set_epilogue_wait_ns(-1)
    C = oz.ozaki2_dgemm(dA, dB, s)
    assert oz.ozaki_get_device_status() == oz.OZ_OK
    assert np.array_equal(_bits(_host(C)), _bits(O.ozaki2_dgemm(A, B, s, keep=False).C))


def test_expired_epilogue_wait_in_scheme1_is_reported_and_the_next_call_is_exact(oz):
    m, n, k, s = 300, 280, 2500, 7
    A, B = hpl_like(m, n, k, phi=0.5, seed=72)
    dA, dB = _dev(A), _dev(B)
    oz.ozaki_set_epilogue_wait_ns(0)
    oz.ozaki1_dgemm_ex(dA, dB, s, "hybrid")
    assert oz.ozaki_get_device_status() == oz.OZ_ETIMEOUT
    oz.ozaki_set_epilogue_wait_ns(-1)
    C = oz.ozaki1_dgemm_ex(dA, dB, s, "hybrid")
    assert oz.ozaki_get_device_status() == oz.OZ_OK
    assert np.array_equal(_bits(_host(C)), _bits(O1.ozaki1_dgemm_variant(A, B, s, "hybrid")[0]))
