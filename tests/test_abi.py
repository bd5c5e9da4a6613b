"""The C-ABI library loads and exports what include/ozaki.h declares; host logic matches the oracle.

No GPU is used here: only host-side queries and argument checks that return before
any CUDA call.
"""
import ctypes
import os
import re

import pytest

from fp64_gemm_emulation_gb300 import build_lib
from oracle import ozaki2 as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def oz():
    if not os.path.exists(build_lib.LIB):
        build_lib.build()
    from fp64_gemm_emulation_gb300 import ozaki

    return ozaki


def declared_functions():
    names = []
    for hdr in os.listdir(os.path.join(ROOT, "include")):
        if hdr.endswith(".h"):
            with open(os.path.join(ROOT, "include", hdr)) as f:
                names += re.findall(r"^(?:int|size_t|const char\*)\s+(\w+)\s*\(", f.read(), flags=re.M)
    return names


def test_every_declared_symbol_is_exported(oz):
    names = declared_functions()
    assert len(names) >= 13
    lib = ctypes.CDLL(build_lib.LIB)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_moduli_match_the_oracle(oz):
    for s in range(1, 21):
        assert oz.ozaki2_moduli(s) == O.greedy_moduli(s)


@pytest.mark.parametrize("s", [2, 3, 8, 10, 12, 14, 16, 18, 20])
@pytest.mark.parametrize("q", [1, 63, 256, 960, 4096, 8192, 16384, 131071, 131072, 262144, 2**31 - 1])
def test_choose_k_matches_the_oracle(oz, s, q):
    M = O.crt_constants(O.greedy_moduli(s)).M
    try:
        want = O.choose_k(M, q)
    except ValueError:
        want = None
    if want is None or want < 1:
        with pytest.raises(oz.OzakiError) as e:
            oz.ozaki2_choose_k(s, q)
        assert e.value.code == oz.OZ_ERANGE
    else:
        assert oz.ozaki2_choose_k(s, q) == want


def test_plane_dims_and_workspace(oz):
    assert oz.ozaki2_plane_dims(1, 1, 1) == (256, 256, 64)
    assert oz.ozaki2_plane_dims(300, 520, 2100) == (512, 768, 2112)
    assert oz.ozaki2_plane_dims(16384, 16384, 16384) == (16384, 16384, 16384)
    ws = oz.ozaki2_workspace_bytes(300, 520, 2100, 14)
    assert ws >= 14 * (512 + 768) * 2112 * 2 + 14 * 512 * 768
    assert oz.ozaki2_workspace_bytes(300, 520, 2100, 1) == 0   # fewer than 2 moduli
    assert oz.ozaki2_workspace_bytes(-1, 5, 5, 14) == 0


def test_argument_errors_are_synchronous(oz):
    lib = oz._lib
    null = None
    # negative dimension, bad leading dimensions, moduli count out of range
    assert lib.ozaki2_dgemm(-1, 4, 4, null, 1, null, 4, null, 1, 14, null) == oz.OZ_EINVAL
    assert lib.ozaki2_dgemm(8, 4, 4, null, 7, null, 4, null, 8, 14, null) == oz.OZ_EINVAL
    assert lib.ozaki2_dgemm(8, 4, 4, null, 8, null, 3, null, 8, 14, null) == oz.OZ_EINVAL
    assert lib.ozaki2_dgemm(8, 4, 4, null, 8, null, 4, null, 7, 14, null) == oz.OZ_EINVAL
    assert lib.ozaki2_dgemm(8, 4, 4, null, 8, null, 4, null, 8, 1, null) == oz.OZ_EINVAL
    assert lib.ozaki2_dgemm(8, 4, 4, null, 8, null, 4, null, 8, 21, null) == oz.OZ_EINVAL
    # empty problems return at once
    assert lib.ozaki2_dgemm(0, 4, 4, null, 1, null, 4, null, 1, 14, null) == oz.OZ_OK
    assert lib.ozaki2_dgemm(4, 0, 4, null, 4, null, 4, null, 4, 14, null) == oz.OZ_OK
    # too few moduli for the inner dimension
    assert lib.ozaki2_dgemm_ws(8, 8, 2**30, 1, 8, 1, 2**30, 1, 8, 2, 1, 1 << 40, null) == oz.OZ_ERANGE
    # workspace too small
    assert lib.ozaki2_dgemm_ws(8, 8, 8, 1, 8, 1, 8, 1, 8, 14, 256, 16, null) == oz.OZ_ENOMEM
    assert oz.ozaki_status_string(oz.OZ_ETIMEOUT).startswith("OZ_ETIMEOUT")


def test_noalloc_checks_arguments_in_the_order_of_ozaki2_dgemm(oz):
    # every one of these returns before any CUDA call: null pointers and OZ_ERANGE come
    # before the buffer's size limit, as in ozaki2_dgemm
    lib = oz._lib
    null = None
    big = 4096  # its workspace is far beyond the fixed buffer
    assert oz.ozaki2_workspace_bytes(big, big, big, 14) > oz.OZ_NOALLOC_SCRATCH_BYTES
    assert lib.ozaki2_dgemm_noalloc(-1, 4, 4, null, 1, null, 4, null, 1, 14, null) == oz.OZ_EINVAL
    assert lib.ozaki2_dgemm_noalloc(8, 4, 4, null, 8, null, 4, null, 8, 21, null) == oz.OZ_EINVAL
    assert lib.ozaki2_dgemm_noalloc(0, 4, 4, null, 1, null, 4, null, 1, 14, null) == oz.OZ_OK
    assert lib.ozaki2_dgemm_noalloc(big, big, big, 1, big, 1, big, null, big, 14, null) == oz.OZ_EINVAL
    assert lib.ozaki2_dgemm_noalloc(big, big, big, null, big, 1, big, 1, big, 14, null) == oz.OZ_EINVAL
    assert lib.ozaki2_dgemm_noalloc(big, big, big, 1, big, null, big, 1, big, 14, null) == oz.OZ_EINVAL
    assert lib.ozaki2_dgemm_noalloc(8, 8, 2**30, 1, 8, 1, 2**30, 1, 8, 2, null) == oz.OZ_ERANGE
    assert lib.ozaki2_dgemm(8, 8, 2**30, 1, 8, 1, 2**30, 1, 8, 2, null) == oz.OZ_ERANGE
    assert lib.ozaki2_dgemm_noalloc(big, big, big, 1, big, 1, big, 1, big, 14, null) == oz.OZ_ENOMEM


def test_binding_names_follow_the_header(oz):
    for name in declared_functions():
        if name.startswith("ozaki"):
            assert hasattr(oz, name), name


@pytest.mark.parametrize("q", [1, 2, 3, 255, 256, 4095, 4096, 4097, 16384, 65536, 2**17, 2**17 + 1,
                               262144, 2**20, 2**25, 2**29])
def test_ozaki1_beta_matches_the_oracle(oz, q):
    from oracle import ozaki1 as O1

    want = O1.beta_rn(q)
    if want < 1:
        with pytest.raises(oz.OzakiError):
            oz.ozaki1_beta(q)
    else:
        assert oz.ozaki1_beta(q) == want


def test_ozaki1_workspace(oz):
    s = 7
    ws = oz.ozaki1_workspace_bytes(300, 520, 2100, s)
    mp, np_, kp = oz.ozaki2_plane_dims(300, 520, 2100)
    assert ws >= 2 * s * (mp + np_) * kp + 4 * (s * (s + 1) // 2) * mp * np_
    assert oz.ozaki1_workspace_bytes(300, 520, 2100, 0) == 0
    assert oz.ozaki1_workspace_bytes(300, 520, 2100, 21) == 0
    assert oz.ozaki1_split_scratch_bytes(300, 520, 2100) >= 8 * (300 * 2100 + 2100 * 520)


# ------------------------------------------------------------------ range estimation modes
@pytest.mark.parametrize("s", [2, 3, 8, 14, 16, 20])
@pytest.mark.parametrize("q", [1, 256, 1025, 16384, 262144, 2**24, 2**24 + 1, 2**30])
@pytest.mark.parametrize("scaling", ["uniform", "fast", "accu"])
def test_scaling_k_matches_the_oracle(oz, s, q, scaling):
    M = O.crt_constants(O.greedy_moduli(s)).M
    if scaling == "accu" and q > 2**24:
        with pytest.raises(oz.OzakiError) as e:
            oz.ozaki2_scaling_k(s, q, scaling)
        assert e.value.code == oz.OZ_EINVAL
        return
    try:
        want = O.choose_k(M, q if scaling == "uniform" else 1)
    except ValueError:
        want = None
    if want is None or want < 1:
        with pytest.raises(oz.OzakiError):
            oz.ozaki2_scaling_k(s, q, scaling)
    else:
        assert oz.ozaki2_scaling_k(s, q, scaling) == want
        if scaling != "uniform":
            assert want == O.half_range_log2(M) // 2


def test_scaling_workspace_sizes(oz):
    m, n, k = 300, 520, 2100
    mp, np_, kp = oz.ozaki2_plane_dims(m, n, k)
    assert oz.ozaki2_exponents_workspace_bytes(m, n, k, "uniform") == 0
    assert oz.ozaki2_exponents_workspace_bytes(m, n, k, "fast") >= 8 * (m + n)
    assert oz.ozaki2_exponents_workspace_bytes(m, n, k, "accu") >= 2 * kp * (mp + np_) + 4 * (mp + np_)
    base = oz.ozaki2_workspace_bytes(m, n, k, 14)
    assert oz.ozaki2_workspace_bytes_ex(m, n, k, 14, "uniform") == base
    assert oz.ozaki2_workspace_bytes_ex(m, n, k, 14, "fast") >= base
    # the exponent scratch overlays the C_res region: the total grows only when it is larger
    tall = oz.ozaki2_workspace_bytes_ex(256, 256, 262144, 14, "accu")
    assert tall >= oz.ozaki2_workspace_bytes(256, 256, 262144, 14)
    assert oz.ozaki2_workspace_bytes_ex(m, n, k, 14, 7) == 0


def test_scaling_argument_errors(oz):
    lib = oz._lib
    null = None
    # unknown scaling mode
    assert lib.ozaki2_dgemm_ex(8, 4, 4, 1, 8, 1, 4, 1, 8, 14, 3, null) == oz.OZ_EINVAL
    assert lib.ozaki2_dgemm_ex(8, 4, 4, 1, 8, 1, 4, 1, 8, 14, -1, null) == oz.OZ_EINVAL
    # accu needs k <= 2^24 and both operands
    assert lib.ozaki2_dgemm_ex_ws(8, 8, 2**24 + 1, 1, 8, 1, 2**24 + 1, 1, 8, 14, 2, 256, 1 << 40, null) == oz.OZ_EINVAL
    assert lib.ozaki2_exponents_ex(8, 8, 8, 1, 8, null, 8, 14, 2, 1, 1, 256, 1 << 30, null) == oz.OZ_EINVAL
    # fast / accu scratch too small
    assert lib.ozaki2_exponents_ex(8, 8, 8, 1, 8, 1, 8, 14, 1, 1, 1, 256, 8, null) == oz.OZ_ENOMEM
    assert lib.ozaki2_dgemm_ex_ws(8, 8, 8, 1, 8, 1, 8, 1, 8, 14, 2, 256, 16, null) == oz.OZ_ENOMEM
    # split / crt reject an unknown mode
    assert lib.ozaki2_split_ex(8, 8, 8, 1, 8, 1, 8, 14, 5, 1, 1, 1, 1, null) == oz.OZ_EINVAL
    assert lib.ozaki2_crt_ex(8, 8, 8, 14, 5, 1, 1, 1, 1, 8, null) == oz.OZ_EINVAL


# ------------------------------------------------------------------ Scheme I variants
@pytest.mark.parametrize("q", [1, 2, 255, 4096, 4097, 16384, 2**17, 2**17 + 1, 262144])
def test_ozaki1_group_r_and_products_match_the_oracle(oz, q):
    from oracle import ozaki1 as O1

    beta = O1.beta_rn(q)
    if beta < 1:
        return
    assert oz.ozaki1_group_r(q) == O1.group_r(q, beta)
    for s in (1, 3, 7, 9, 20):
        assert oz.ozaki1_num_batches(s, q, "rn") == s * (s + 1) // 2
        want = len(O1.group_batches(s, O1.group_r(q, beta)))
        assert oz.ozaki1_num_batches(s, q, "ef") == want
        assert oz.ozaki1_num_batches(s, q, "hybrid") == want


def test_ozaki1_variant_workspace_and_errors(oz):
    lib, null = oz._lib, None
    m, n, k = 300, 520, 2100
    assert oz.ozaki1_workspace_bytes_ex(m, n, k, 7, "rn") == oz.ozaki1_workspace_bytes(m, n, k, 7)
    # EF and Hybrid split in one pass: no residual arrays
    assert oz.ozaki1_split_scratch_bytes_ex(m, n, k, "ef") < oz.ozaki1_split_scratch_bytes_ex(m, n, k, "rn")
    assert oz.ozaki1_workspace_bytes_ex(m, n, k, 7, "ef") < oz.ozaki1_workspace_bytes_ex(m, n, k, 7, "rn")
    assert oz.ozaki1_workspace_bytes_ex(m, n, k, 7, "hybrid") == oz.ozaki1_workspace_bytes_ex(m, n, k, 7, "ef")
    assert oz.ozaki1_workspace_bytes_ex(m, n, k, 7, 3) == 0
    assert lib.ozaki1_dgemm_ex(8, 4, 4, 1, 8, 1, 4, 1, 8, 7, 3, null) == oz.OZ_EINVAL
    assert lib.ozaki1_dgemm_ex_ws(8, 8, 8, 1, 8, 1, 8, 1, 8, 7, 1, 256, 16, null) == oz.OZ_ENOMEM
    assert lib.ozaki1_num_batches(0, 16, 1, ctypes.byref(ctypes.c_int())) == oz.OZ_EINVAL


def test_epilogue_wait_setting_checks_its_argument(oz):
    lib = oz._lib
    assert lib.ozaki_set_epilogue_wait_ns(-2) == oz.OZ_EINVAL
    assert lib.ozaki_set_epilogue_wait_ns(1000) == oz.OZ_OK
    assert lib.ozaki_set_epilogue_wait_ns(-1) == oz.OZ_OK  # back to the default
