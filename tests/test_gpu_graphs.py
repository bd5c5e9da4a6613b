"""The workspace entry points under CUDA graph capture: a captured call replays bit for bit,
and replays on new operand values (same buffers) give the oracle's result for those values.
Every step is a stream-ordered memset or kernel launch, so the whole path captures."""
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


def bits(x):
    return np.ascontiguousarray(x, dtype=np.float64).view(np.int64)


def col(X):
    return torch.from_numpy(np.asfortranarray(X).T.copy()).cuda().t()


@pytest.mark.parametrize("m,n,k,s,scaling", [(256, 256, 256, 14, "uniform"), (300, 520, 1100, 14, "uniform"),
                                             (200, 130, 700, 12, "accu"), (200, 130, 700, 12, "fast")])
def test_captured_call_replays_bit_exact(oz, m, n, k, s, scaling):
    A, B = hpl_like(m, n, k, phi=1.0, seed=40)
    dA, dB = col(A), col(B)
    C = torch.empty((n, m), dtype=torch.float64, device="cuda").t()
    ws = torch.empty(oz.ozaki2_workspace_bytes_ex(m, n, k, s, scaling), dtype=torch.uint8, device="cuda")
    oz.ozaki2_dgemm_ex_ws(dA, dB, s, scaling, ws, C=C)  # warm: module loading, tensor-map encoder lookup
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        oz.ozaki2_dgemm_ex_ws(dA, dB, s, scaling, ws, C=C)
    C.fill_(0.0)
    g.replay()
    torch.cuda.synchronize()
    ref = O.ozaki2_dgemm(A, B, s, keep=False, scaling=scaling).C
    assert np.array_equal(bits(C.t().contiguous().cpu().numpy().T), bits(ref))
    # new values in the same buffers
    A2, B2 = hpl_like(m, n, k, phi=2.0, seed=41)
    dA.copy_(col(A2))
    dB.copy_(col(B2))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    ref2 = O.ozaki2_dgemm(A2, B2, s, keep=False, scaling=scaling).C
    assert np.array_equal(bits(C.t().contiguous().cpu().numpy().T), bits(ref2))
    assert oz.ozaki_get_device_status() == oz.OZ_OK


def test_captured_scheme1_hybrid(oz):
    from oracle import ozaki1 as O1

    m, n, k = 260, 300, 900
    A, B = hpl_like(m, n, k, phi=0.5, seed=42)
    dA, dB = col(A), col(B)
    C = torch.empty((n, m), dtype=torch.float64, device="cuda").t()
    ws = torch.empty(oz.ozaki1_workspace_bytes_ex(m, n, k, 7, "hybrid"), dtype=torch.uint8, device="cuda")
    oz.ozaki1_dgemm_ex_ws(dA, dB, 7, "hybrid", ws, C=C)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        oz.ozaki1_dgemm_ex_ws(dA, dB, 7, "hybrid", ws, C=C)
    C.fill_(0.0)
    g.replay()
    torch.cuda.synchronize()
    ref = O1.ozaki1_dgemm_variant(A, B, 7, "hybrid")[0]
    assert np.array_equal(bits(C.t().contiguous().cpu().numpy().T), bits(ref))
