"""Full-size intermediates against the oracle, element by element.

At the benchmark's sizes some code paths exist only there: the GEMM's pair pacing
over many waves of 76 CTA pairs, the reduction of the 16-bit running lanes every 64
chunks of 1024 k (first reached at k = 65,536), and the widest C_res layout.  So at
16384^3 (s = 14) and 2048 x 2048 x 262144 (s = 14) this test compares, with the
oracle ([Ozaki II] section 7, Algorithm 1 steps 2-3):

* the row / column exponents, in full;
* every residue plane of A and B, in full (the oracle's truncation and symmetric
  residues computed on the host in row blocks), plus the zero padding;
* the C''_t planes of every modulus on sampled 128 x 128 output tiles, including
  the last row and column tiles, against the oracle's exact products mod m_t over
  the whole k.

The steps run through the C ABI in the benchmark's launch configuration.
"""
import math

import numpy as np
import pytest

from fp64_gemm_emulation_gb300.inputs import hpl_like
from oracle import ozaki2 as O

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


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


def plane_block_to_int8(P, r0, r1, k):
    """Rows r0..r1 of every bf16 plane (int16 bit patterns) as int8 values, on the host."""
    return P[:, r0:r1, :k].view(torch.bfloat16).to(torch.int8).cpu().numpy()


def check_planes(P, X, d, moduli, rows_total, k, block):
    """Every plane of X's rows (rows of A, or columns of B as rows of B^T) against the oracle."""
    for r0 in range(0, rows_total, block):
        r1 = min(rows_total, r0 + block)
        want = O.residue_planes(O.scaled_trunc_matrix(X[r0:r1], d[r0:r1]), moduli)
        got = plane_block_to_int8(P, r0, r1, k)
        if not np.array_equal(got, want):
            bad = np.argwhere(got != want)[0]
            raise AssertionError(f"plane mismatch at (t, row, k) = ({bad[0]}, {r0 + bad[1]}, {bad[2]})")
    assert not bool(P[:, rows_total:, :].any()) and not bool(P[:, :, k:].any())  # zero padding


def tile_origins(m, n, count, seed):
    rng = np.random.default_rng(seed)
    tm, tn = m // 128, n // 128
    picks = {(0, 0), (tm - 1, tn - 1), (tm - 1, 0), (0, tn - 1)}
    while len(picks) < count:
        picks.add((int(rng.integers(0, tm)), int(rng.integers(0, tn))))
    return sorted(picks)


@pytest.mark.parametrize("m,n,k,s,phi,row_block", [
    (16384, 16384, 16384, 14, 0.5, 512),
    (2048, 2048, 262144, 14, 0.5, 32),
])
def test_full_size_intermediates_match_the_oracle(m, n, k, s, phi, row_block):
    from fp64_gemm_emulation_gb300 import ozaki as oz

    A, B = hpl_like(m, n, k, phi=phi, seed=0)
    Bt = np.ascontiguousarray(B.T)
    moduli = O.greedy_moduli(s)
    kA = O.choose_k(math.prod(moduli), k)
    EA, EB = O.row_exponents(A), O.row_exponents(Bt)
    dA_, eB_ = O.scale_exponents(EA, kA), O.scale_exponents(EB, kA)

    dA = torch.from_numpy(A.T.copy()).cuda().t()
    dB = torch.from_numpy(Bt).cuda().t()
    rowexp, colexp = oz.ozaki2_exponents(dA, dB)
    assert np.array_equal(rowexp.cpu().numpy(), exps_as_int32(EA))
    assert np.array_equal(colexp.cpu().numpy(), exps_as_int32(EB))
    Ap, Bp = oz.ozaki2_split(dA, dB, s, rowexp, colexp)
    del dA, dB
    Cr = oz.ozaki2_residue_gemm(m, n, k, s, Ap, Bp)
    torch.cuda.synchronize()
    assert oz.ozaki_get_device_status() == oz.OZ_OK

    check_planes(Ap, A, dA_, moduli, m, k, row_block)
    check_planes(Bp, Bt, eB_, moduli, n, k, row_block)
    del Ap, Bp
    torch.cuda.empty_cache()

    for ti, tj in tile_origins(m, n, 8, seed=k):
        rows = slice(128 * ti, 128 * ti + 128)
        cols = slice(128 * tj, 128 * tj + 128)
        Ares = O.residue_planes(O.scaled_trunc_matrix(A[rows], dA_[rows]), moduli)
        Bres = O.residue_planes(O.scaled_trunc_matrix(Bt[cols], eB_[cols]), moduli)
        want = O.residue_products(Ares, np.transpose(Bres, (0, 2, 1)), moduli)   # [t][i][j]
        got = Cr[:, cols, rows].cpu().numpy().transpose(0, 2, 1)                # C_res is [t][j][i]
        assert np.array_equal(got.astype(np.int64), want), f"C''_t tile ({ti}, {tj})"
