"""Python binding of libozaki (argument marshalling only; every step runs in the CUDA kernels).

The functions carry the C ABI's names (``include/ozaki.h``).  Device operands are
torch CUDA tensors; matrices are column-major float64 (a tensor ``X`` of shape
(rows, cols) with ``X.stride(0) == 1``; :func:`colmajor` makes one).  Calls are
ordered on the current torch CUDA stream unless ``stream`` is given.

There is no fallback: if ``libozaki.so`` is missing or fails to load, importing
this module raises, and every call reports the library's status code as an
exception.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libozaki.so")

OZ_OK, OZ_EINVAL, OZ_ERANGE, OZ_ECUDA, OZ_ENOMEM, OZ_ETIMEOUT, OZ_ENODEV = 0, -1, -2, -3, -4, -5, -6
OZ_EXP_EMPTY = np.int32(np.uint32(0x80808080).view(np.int32))
OZ_EXP_NONFINITE = np.int32(0x7FFFFFFF)
PAD_M, PAD_N, PAD_K = 256, 256, 64
OZ_NOALLOC_SCRATCH_BYTES = 64 << 20
OZ_SCALE_UNIFORM, OZ_SCALE_FAST, OZ_SCALE_ACCU = 0, 1, 2
OZ_OZAKI1_RN, OZ_OZAKI1_EF, OZ_OZAKI1_HYBRID = 0, 1, 2
OZAKI1_VARIANTS = {"rn": OZ_OZAKI1_RN, "ef": OZ_OZAKI1_EF, "hybrid": OZ_OZAKI1_HYBRID}
SCALINGS = {"uniform": OZ_SCALE_UNIFORM, "fast": OZ_SCALE_FAST, "accu": OZ_SCALE_ACCU}


class OzakiError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {_lib.ozaki_status_string(code).decode()}")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -m fp64_gemm_emulation_gb300.build_lib`")
    lib = ctypes.CDLL(LIB_PATH)
    I, L, P, S = ctypes.c_int, ctypes.c_longlong, ctypes.c_void_p, ctypes.c_size_t
    sig = {
        "ozaki2_moduli": (I, [I, P]),
        "ozaki2_choose_k": (I, [I, L, P]),
        "ozaki2_plane_dims": (I, [I, I, I, P, P, P]),
        "ozaki2_workspace_bytes": (S, [I, I, I, I]),
        "ozaki2_exponents": (I, [I, I, I, P, I, P, I, P, P, P]),
        "ozaki2_split": (I, [I, I, I, P, I, P, I, I, P, P, P, P, P]),
        "ozaki2_residue_gemm": (I, [I, I, I, I, P, P, P, P]),
        "ozaki2_scale_split": (I, [I, I, I, P, I, P, I, I, P, P, P, P, P]),
        "ozaki2_crt": (I, [I, I, I, I, P, P, P, P, I, P]),
        "ozaki2_dgemm_ws": (I, [I, I, I, P, I, P, I, P, I, I, P, S, P]),
        "ozaki2_dgemm": (I, [I, I, I, P, I, P, I, P, I, I, P]),
        "ozaki2_dgemm_host": (I, [I, I, I, P, I, P, I, P, I, I]),
        "ozaki2_dgemm_noalloc": (I, [I, I, I, P, I, P, I, P, I, I, P]),
        "ozaki2_scaling_k": (I, [I, L, I, P]),
        "ozaki2_exponents_workspace_bytes": (S, [I, I, I, I]),
        "ozaki2_exponents_ex": (I, [I, I, I, P, I, P, I, I, I, P, P, P, S, P]),
        "ozaki2_split_ex": (I, [I, I, I, P, I, P, I, I, I, P, P, P, P, P]),
        "ozaki2_crt_ex": (I, [I, I, I, I, I, P, P, P, P, I, P]),
        "ozaki2_workspace_bytes_ex": (S, [I, I, I, I, I]),
        "ozaki2_dgemm_ex_ws": (I, [I, I, I, P, I, P, I, P, I, I, I, P, S, P]),
        "ozaki2_dgemm_ex": (I, [I, I, I, P, I, P, I, P, I, I, I, P]),
        "ozaki1_beta": (I, [L, P]),
        "ozaki1_split_scratch_bytes": (S, [I, I, I]),
        "ozaki1_workspace_bytes": (S, [I, I, I, I]),
        "ozaki1_split": (I, [I, I, I, P, I, P, I, I, P, P, P, P, P, S, P]),
        "ozaki1_slice_gemm": (I, [I, I, I, I, P, P, P, P]),
        "ozaki1_accumulate": (I, [I, I, I, I, P, P, P, P, I, P]),
        "ozaki1_dgemm_ws": (I, [I, I, I, P, I, P, I, P, I, I, P, S, P]),
        "ozaki1_dgemm": (I, [I, I, I, P, I, P, I, P, I, I, P]),
        "ozaki1_group_r": (I, [L, P]),
        "ozaki1_num_batches": (I, [I, L, I, P]),
        "ozaki1_split_scratch_bytes_ex": (S, [I, I, I, I]),
        "ozaki1_workspace_bytes_ex": (S, [I, I, I, I, I]),
        "ozaki1_split_ex": (I, [I, I, I, P, I, P, I, I, I, P, P, P, P, P, S, P]),
        "ozaki1_slice_gemm_ex": (I, [I, I, I, I, I, P, P, P, P]),
        "ozaki1_accumulate_ex": (I, [I, I, I, I, I, P, P, P, P, I, P]),
        "ozaki1_dgemm_ex_ws": (I, [I, I, I, P, I, P, I, P, I, I, I, P, S, P]),
        "ozaki1_dgemm_ex": (I, [I, I, I, P, I, P, I, P, I, I, I, P]),
        "ozaki_get_device_status": (I, [P]),
        "ozaki_status_string": (ctypes.c_char_p, [I]),
        "ozaki_set_epilogue_wait_ns": (I, [L]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def _check(rc: int, where: str) -> None:
    if rc != OZ_OK:
        raise OzakiError(rc, where)


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    return int(getattr(stream, "cuda_stream", stream))


def _ptr(t):
    return None if t is None else t.data_ptr()


def colmajor(x):
    """A column-major copy (or view) of a 2-D tensor: same shape, stride(0) == 1."""
    return x if (x.dim() == 2 and x.stride(0) == 1 and x.stride(1) >= max(1, x.shape[0])) else x.t().contiguous().t()


def _ld(x) -> int:
    assert x.dim() == 2 and x.stride(0) == 1, "operand must be column-major (stride(0) == 1)"
    return max(1, int(x.stride(1)), int(x.shape[0]))


# ------------------------------------------------------------------ host-only queries
def ozaki2_moduli(num_moduli: int) -> list[int]:
    out = (ctypes.c_int * max(1, num_moduli))()
    _check(_lib.ozaki2_moduli(num_moduli, out), "ozaki2_moduli")
    return list(out[:num_moduli])


def ozaki2_choose_k(num_moduli: int, k_inner: int) -> int:
    k = ctypes.c_int()
    _check(_lib.ozaki2_choose_k(num_moduli, k_inner, ctypes.byref(k)), "ozaki2_choose_k")
    return k.value


def ozaki2_plane_dims(m: int, n: int, k: int) -> tuple[int, int, int]:
    a, b, c = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(_lib.ozaki2_plane_dims(m, n, k, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)), "ozaki2_plane_dims")
    return a.value, b.value, c.value


def ozaki2_workspace_bytes(m: int, n: int, k: int, num_moduli: int) -> int:
    return int(_lib.ozaki2_workspace_bytes(m, n, k, num_moduli))


# ------------------------------------------------------------------ steps
def ozaki2_exponents(A, B, stream=None):
    """Step a1: (rowexp[m], colexp[n]) int32 tensors on A's device."""
    import torch

    m, k = A.shape
    n = B.shape[1]
    rowexp = torch.empty(m, dtype=torch.int32, device=A.device)
    colexp = torch.empty(n, dtype=torch.int32, device=A.device)
    _check(_lib.ozaki2_exponents(m, n, k, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(rowexp), _ptr(colexp),
                                 _stream(stream)), "ozaki2_exponents")
    return rowexp, colexp


def ozaki2_split(A, B, num_moduli: int, rowexp, colexp, stream=None):
    """Step a2: bf16-bit residue planes (uint16 views as int16 tensors) [s, Mp, Kp] and [s, Np, Kp]."""
    import torch

    m, k = A.shape
    n = B.shape[1]
    mp, np_, kp = ozaki2_plane_dims(m, n, k)
    Ap = torch.empty((num_moduli, mp, kp), dtype=torch.int16, device=A.device)
    Bp = torch.empty((num_moduli, np_, kp), dtype=torch.int16, device=A.device)
    _check(_lib.ozaki2_split(m, n, k, _ptr(A), _ld(A), _ptr(B), _ld(B), num_moduli, _ptr(rowexp), _ptr(colexp),
                             _ptr(Ap), _ptr(Bp), _stream(stream)), "ozaki2_split")
    return Ap, Bp


def ozaki2_scale_split(A, B, num_moduli: int, stream=None):
    """Steps a1 + a2 in one call: (rowexp, colexp, A_planes, B_planes); either operand may be None."""
    import torch

    dev = (A if A is not None else B).device
    k = A.shape[1] if A is not None else B.shape[0]
    m = A.shape[0] if A is not None else 0
    n = B.shape[1] if B is not None else 0
    mp, np_, kp = ozaki2_plane_dims(m, n, k)
    rowexp = torch.empty(m, dtype=torch.int32, device=dev) if A is not None else None
    colexp = torch.empty(n, dtype=torch.int32, device=dev) if B is not None else None
    Ap = torch.empty((num_moduli, mp, kp), dtype=torch.int16, device=dev) if A is not None else None
    Bp = torch.empty((num_moduli, np_, kp), dtype=torch.int16, device=dev) if B is not None else None
    _check(_lib.ozaki2_scale_split(m, n, k, _ptr(A), _ld(A) if A is not None else 1, _ptr(B),
                                   _ld(B) if B is not None else 1, num_moduli, _ptr(rowexp), _ptr(colexp),
                                   _ptr(Ap), _ptr(Bp), _stream(stream)), "ozaki2_scale_split")
    return rowexp, colexp, Ap, Bp


def ozaki2_residue_gemm(m: int, n: int, k: int, num_moduli: int, A_planes, B_planes, stream=None):
    """Steps a3+a4: C_res uint8 tensor [s, Np, Mp] with C''_t = (A'_t B'_t) mod m_t."""
    import torch

    mp, np_, kp = ozaki2_plane_dims(m, n, k)
    Cr = torch.empty((num_moduli, np_, mp), dtype=torch.uint8, device=A_planes.device)
    _check(_lib.ozaki2_residue_gemm(m, n, k, num_moduli, _ptr(A_planes), _ptr(B_planes), _ptr(Cr),
                                    _stream(stream)), "ozaki2_residue_gemm")
    return Cr


def ozaki2_crt(m: int, n: int, k: int, num_moduli: int, C_res, rowexp, colexp, C=None, stream=None):
    """Steps a5+a6: C (m x n column-major float64)."""
    import torch

    if C is None:
        C = torch.empty((n, m), dtype=torch.float64, device=C_res.device).t()
    _check(_lib.ozaki2_crt(m, n, k, num_moduli, _ptr(C_res), _ptr(rowexp), _ptr(colexp), _ptr(C), _ld(C),
                           _stream(stream)), "ozaki2_crt")
    return C


# ------------------------------------------------------------------ composed
def ozaki2_dgemm(A, B, num_moduli: int = 14, C=None, stream=None):
    """C = A B by Ozaki Scheme II (stream-ordered workspace allocation inside the library)."""
    import torch

    m, k = A.shape
    n = B.shape[1]
    if C is None:
        C = torch.empty((n, m), dtype=torch.float64, device=A.device).t()
    _check(_lib.ozaki2_dgemm(m, n, k, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C), _ld(C), num_moduli,
                             _stream(stream)), "ozaki2_dgemm")
    return C


def ozaki2_dgemm_ws(A, B, num_moduli: int, workspace, C=None, stream=None):
    """C = A B using a caller-owned device workspace (a uint8 tensor of at least
    ozaki2_workspace_bytes(m, n, k, num_moduli) bytes)."""
    import torch

    m, k = A.shape
    n = B.shape[1]
    if C is None:
        C = torch.empty((n, m), dtype=torch.float64, device=A.device).t()
    _check(_lib.ozaki2_dgemm_ws(m, n, k, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C), _ld(C), num_moduli,
                                _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
           "ozaki2_dgemm_ws")
    return C


def ozaki2_dgemm_noalloc(A, B, num_moduli: int = 14, C=None, stream=None):
    """C = A B without any device allocation: the library's fixed 64 MiB scratch buffer
    holds the workspace (for callers that cannot allocate; see include/ozaki.h)."""
    import torch

    m, k = A.shape
    n = B.shape[1]
    if C is None:
        C = torch.empty((n, m), dtype=torch.float64, device=A.device).t()
    _check(_lib.ozaki2_dgemm_noalloc(m, n, k, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C), _ld(C), num_moduli,
                                     _stream(stream)), "ozaki2_dgemm_noalloc")
    return C


def ozaki2_dgemm_host(A: np.ndarray, B: np.ndarray, num_moduli: int = 14, C: np.ndarray | None = None):
    """C = A B with HOST (numpy, column-major float64) operands; synchronous."""
    A = np.asfortranarray(A, dtype=np.float64)
    B = np.asfortranarray(B, dtype=np.float64)
    m, k = A.shape
    n = B.shape[1]
    if C is None:
        C = np.empty((m, n), dtype=np.float64, order="F")
    assert C.flags.f_contiguous and C.dtype == np.float64
    _check(_lib.ozaki2_dgemm_host(m, n, k, A.ctypes.data, max(1, m), B.ctypes.data, max(1, k), C.ctypes.data,
                                  max(1, m), num_moduli), "ozaki2_dgemm_host")
    return C


def ozaki2_dgemm_host_ptr(m, n, k, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, num_moduli):
    """Raw-pointer form of ozaki2_dgemm_host (host pointers, e.g. pinned torch tensors)."""
    _check(_lib.ozaki2_dgemm_host(m, n, k, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, num_moduli), "ozaki2_dgemm_host")


# ------------------------------------------------------------------ range estimation modes
def _scaling(scaling) -> int:
    return SCALINGS[scaling] if isinstance(scaling, str) else int(scaling)


def ozaki2_scaling_k(num_moduli: int, k_inner: int, scaling="uniform") -> int:
    k = ctypes.c_int()
    _check(_lib.ozaki2_scaling_k(num_moduli, k_inner, _scaling(scaling), ctypes.byref(k)), "ozaki2_scaling_k")
    return k.value


def ozaki2_exponents_workspace_bytes(m: int, n: int, k: int, scaling="uniform") -> int:
    return int(_lib.ozaki2_exponents_workspace_bytes(m, n, k, _scaling(scaling)))


def ozaki2_workspace_bytes_ex(m: int, n: int, k: int, num_moduli: int, scaling="uniform") -> int:
    return int(_lib.ozaki2_workspace_bytes_ex(m, n, k, num_moduli, _scaling(scaling)))


def ozaki2_exponents_ex(A, B, num_moduli: int, scaling="uniform", stream=None):
    """Step a1 in a scaling mode: (rowexp[m], colexp[n]) int32 tensors."""
    import torch

    m, k = A.shape
    n = B.shape[1]
    sc = _scaling(scaling)
    rowexp = torch.empty(m, dtype=torch.int32, device=A.device)
    colexp = torch.empty(n, dtype=torch.int32, device=A.device)
    nbytes = ozaki2_exponents_workspace_bytes(m, n, k, sc)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=A.device)
    _check(_lib.ozaki2_exponents_ex(m, n, k, _ptr(A), _ld(A), _ptr(B), _ld(B), num_moduli, sc, _ptr(rowexp),
                                    _ptr(colexp), _ptr(ws), nbytes, _stream(stream)), "ozaki2_exponents_ex")
    return rowexp, colexp


def ozaki2_split_ex(A, B, num_moduli: int, rowexp, colexp, scaling="uniform", stream=None):
    """Step a2 for exponents of a scaling mode (planes as in ozaki2_split)."""
    import torch

    m, k = A.shape
    n = B.shape[1]
    mp, np_, kp = ozaki2_plane_dims(m, n, k)
    Ap = torch.empty((num_moduli, mp, kp), dtype=torch.int16, device=A.device)
    Bp = torch.empty((num_moduli, np_, kp), dtype=torch.int16, device=A.device)
    _check(_lib.ozaki2_split_ex(m, n, k, _ptr(A), _ld(A), _ptr(B), _ld(B), num_moduli, _scaling(scaling),
                                _ptr(rowexp), _ptr(colexp), _ptr(Ap), _ptr(Bp), _stream(stream)), "ozaki2_split_ex")
    return Ap, Bp


def ozaki2_crt_ex(m: int, n: int, k: int, num_moduli: int, C_res, rowexp, colexp, scaling="uniform", C=None,
                  stream=None):
    """Steps a5+a6 for exponents of a scaling mode."""
    import torch

    if C is None:
        C = torch.empty((n, m), dtype=torch.float64, device=C_res.device).t()
    _check(_lib.ozaki2_crt_ex(m, n, k, num_moduli, _scaling(scaling), _ptr(C_res), _ptr(rowexp), _ptr(colexp),
                              _ptr(C), _ld(C), _stream(stream)), "ozaki2_crt_ex")
    return C


def ozaki2_dgemm_ex(A, B, num_moduli: int = 14, scaling="uniform", C=None, workspace=None, stream=None):
    """C = A B by Ozaki Scheme II in a scaling mode ("uniform", "fast", "accu");
    with ``workspace`` (uint8 tensor of ozaki2_workspace_bytes_ex bytes) the _ws form."""
    import torch

    m, k = A.shape
    n = B.shape[1]
    if C is None:
        C = torch.empty((n, m), dtype=torch.float64, device=A.device).t()
    sc = _scaling(scaling)
    if workspace is None:
        rc = _lib.ozaki2_dgemm_ex(m, n, k, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C), _ld(C), num_moduli, sc,
                                  _stream(stream))
    else:
        rc = _lib.ozaki2_dgemm_ex_ws(m, n, k, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C), _ld(C), num_moduli, sc,
                                     _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "ozaki2_dgemm_ex")
    return C


def ozaki2_dgemm_ex_ws(A, B, num_moduli: int, scaling, workspace, C=None, stream=None):
    """C = A B in a scaling mode with a caller-owned workspace (ozaki2_workspace_bytes_ex bytes)."""
    return ozaki2_dgemm_ex(A, B, num_moduli, scaling, C=C, workspace=workspace, stream=stream)


# ------------------------------------------------------------------ Scheme I
def ozaki1_beta(k_inner: int) -> int:
    b = ctypes.c_int()
    _check(_lib.ozaki1_beta(k_inner, ctypes.byref(b)), "ozaki1_beta")
    return b.value


def ozaki1_split_scratch_bytes(m: int, n: int, k: int) -> int:
    return int(_lib.ozaki1_split_scratch_bytes(m, n, k))


def ozaki1_workspace_bytes(m: int, n: int, k: int, num_slices: int) -> int:
    return int(_lib.ozaki1_workspace_bytes(m, n, k, num_slices))


def ozaki1_split(A, B, num_slices: int, stream=None):
    """RN split: (A_planes [s,Mp,Kp], B_planes [s,Np,Kp] as int16 bf16 bits, A_exps [s,m], B_exps [s,n])."""
    import torch

    m, k = A.shape
    n = B.shape[1]
    mp, np_, kp = ozaki2_plane_dims(m, n, k)
    Ap = torch.empty((num_slices, mp, kp), dtype=torch.int16, device=A.device)
    Bp = torch.empty((num_slices, np_, kp), dtype=torch.int16, device=A.device)
    Ae = torch.empty((num_slices, m), dtype=torch.int32, device=A.device)
    Be = torch.empty((num_slices, n), dtype=torch.int32, device=A.device)
    nbytes = ozaki1_split_scratch_bytes(m, n, k)
    scratch = torch.empty(nbytes + 256, dtype=torch.uint8, device=A.device)
    sp = (scratch.data_ptr() + 255) // 256 * 256
    _check(_lib.ozaki1_split(m, n, k, _ptr(A), _ld(A), _ptr(B), _ld(B), num_slices, _ptr(Ap), _ptr(Bp),
                             _ptr(Ae), _ptr(Be), sp, nbytes, _stream(stream)), "ozaki1_split")
    return Ap, Bp, Ae, Be


def ozaki1_slice_gemm(m: int, n: int, k: int, num_slices: int, A_planes, B_planes, stream=None):
    """Exact INT32 products [s(s+1)/2, Np, Mp] of the slice pairs (i outer, j inner)."""
    import torch

    mp, np_, kp = ozaki2_plane_dims(m, n, k)
    P = torch.empty((num_slices * (num_slices + 1) // 2, np_, mp), dtype=torch.int32, device=A_planes.device)
    _check(_lib.ozaki1_slice_gemm(m, n, k, num_slices, _ptr(A_planes), _ptr(B_planes), _ptr(P), _stream(stream)),
           "ozaki1_slice_gemm")
    return P


def ozaki1_accumulate(m: int, n: int, k: int, num_slices: int, products, A_exps, B_exps, C=None, stream=None):
    import torch

    if C is None:
        C = torch.empty((n, m), dtype=torch.float64, device=products.device).t()
    _check(_lib.ozaki1_accumulate(m, n, k, num_slices, _ptr(products), _ptr(A_exps), _ptr(B_exps), _ptr(C), _ld(C),
                                  _stream(stream)), "ozaki1_accumulate")
    return C


def ozaki1_dgemm(A, B, num_slices: int = 7, C=None, stream=None):
    """C = A B by Ozaki Scheme I (stream-ordered workspace inside the library)."""
    import torch

    m, k = A.shape
    n = B.shape[1]
    if C is None:
        C = torch.empty((n, m), dtype=torch.float64, device=A.device).t()
    _check(_lib.ozaki1_dgemm(m, n, k, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C), _ld(C), num_slices,
                             _stream(stream)), "ozaki1_dgemm")
    return C


def ozaki1_dgemm_ws(A, B, num_slices: int, workspace, C=None, stream=None):
    import torch

    m, k = A.shape
    n = B.shape[1]
    if C is None:
        C = torch.empty((n, m), dtype=torch.float64, device=A.device).t()
    _check(_lib.ozaki1_dgemm_ws(m, n, k, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C), _ld(C), num_slices,
                                _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
           "ozaki1_dgemm_ws")
    return C


# ------------------------------------------------------------------ Scheme I variants
def _variant(v) -> int:
    return OZAKI1_VARIANTS[v] if isinstance(v, str) else int(v)


def ozaki1_group_r(k_inner: int) -> int:
    r = ctypes.c_int()
    _check(_lib.ozaki1_group_r(k_inner, ctypes.byref(r)), "ozaki1_group_r")
    return r.value


def ozaki1_num_batches(num_slices: int, k_inner: int, variant="rn") -> int:
    c = ctypes.c_int()
    _check(_lib.ozaki1_num_batches(num_slices, k_inner, _variant(variant), ctypes.byref(c)), "ozaki1_num_batches")
    return c.value


def ozaki1_split_scratch_bytes_ex(m: int, n: int, k: int, variant="rn") -> int:
    return int(_lib.ozaki1_split_scratch_bytes_ex(m, n, k, _variant(variant)))


def ozaki1_workspace_bytes_ex(m: int, n: int, k: int, num_slices: int, variant="rn") -> int:
    return int(_lib.ozaki1_workspace_bytes_ex(m, n, k, num_slices, _variant(variant)))


def ozaki1_split_ex(A, B, num_slices: int, variant="rn", stream=None):
    """Split of a variant: (A_planes, B_planes, A_exps, B_exps) as ozaki1_split."""
    import torch

    m, k = A.shape
    n = B.shape[1]
    v = _variant(variant)
    mp, np_, kp = ozaki2_plane_dims(m, n, k)
    Ap = torch.empty((num_slices, mp, kp), dtype=torch.int16, device=A.device)
    Bp = torch.empty((num_slices, np_, kp), dtype=torch.int16, device=A.device)
    Ae = torch.empty((num_slices, m), dtype=torch.int32, device=A.device)
    Be = torch.empty((num_slices, n), dtype=torch.int32, device=A.device)
    nbytes = ozaki1_split_scratch_bytes_ex(m, n, k, v)
    scratch = torch.empty(nbytes + 256, dtype=torch.uint8, device=A.device)
    sp = (scratch.data_ptr() + 255) // 256 * 256
    _check(_lib.ozaki1_split_ex(m, n, k, _ptr(A), _ld(A), _ptr(B), _ld(B), num_slices, v, _ptr(Ap), _ptr(Bp),
                                _ptr(Ae), _ptr(Be), sp, nbytes, _stream(stream)), "ozaki1_split_ex")
    return Ap, Bp, Ae, Be


def ozaki1_slice_gemm_ex(m: int, n: int, k: int, num_slices: int, variant, A_planes, B_planes, stream=None):
    """Exact INT32 pair products of a variant, in its order: [s(s+1)/2, Np, Mp]."""
    import torch

    v = _variant(variant)
    mp, np_, kp = ozaki2_plane_dims(m, n, k)
    P = torch.empty((num_slices * (num_slices + 1) // 2, np_, mp), dtype=torch.int32, device=A_planes.device)
    _check(_lib.ozaki1_slice_gemm_ex(m, n, k, num_slices, v, _ptr(A_planes), _ptr(B_planes), _ptr(P),
                                     _stream(stream)), "ozaki1_slice_gemm_ex")
    return P


def ozaki1_accumulate_ex(m: int, n: int, k: int, num_slices: int, variant, products, A_exps, B_exps, C=None,
                         stream=None):
    import torch

    if C is None:
        C = torch.empty((n, m), dtype=torch.float64, device=products.device).t()
    _check(_lib.ozaki1_accumulate_ex(m, n, k, num_slices, _variant(variant), _ptr(products), _ptr(A_exps),
                                     _ptr(B_exps), _ptr(C), _ld(C), _stream(stream)), "ozaki1_accumulate_ex")
    return C


def ozaki1_dgemm_ex(A, B, num_slices: int = 7, variant="rn", C=None, workspace=None, stream=None):
    """C = A B by Scheme I in a variant ("rn", "ef", "hybrid"); with ``workspace`` the _ws form."""
    import torch

    m, k = A.shape
    n = B.shape[1]
    v = _variant(variant)
    if C is None:
        C = torch.empty((n, m), dtype=torch.float64, device=A.device).t()
    if workspace is None:
        rc = _lib.ozaki1_dgemm_ex(m, n, k, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C), _ld(C), num_slices, v,
                                  _stream(stream))
    else:
        rc = _lib.ozaki1_dgemm_ex_ws(m, n, k, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C), _ld(C), num_slices, v,
                                     _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "ozaki1_dgemm_ex")
    return C


def ozaki1_dgemm_ex_ws(A, B, num_slices: int, variant, workspace, C=None, stream=None):
    return ozaki1_dgemm_ex(A, B, num_slices, variant, C=C, workspace=workspace, stream=stream)


def ozaki_get_device_status(stream=None) -> int:
    """Status word of the current device after the work on ``stream`` (default: the current
    torch stream) has finished; cleared by the read."""
    return int(_lib.ozaki_get_device_status(_stream(stream)))


def ozaki_set_epilogue_wait_ns(ns: int) -> None:
    """Time limit of the GEMM epilogue's accumulator wait for later launches (-1: default 4 s)."""
    _check(_lib.ozaki_set_epilogue_wait_ns(int(ns)), "ozaki_set_epilogue_wait_ns")


def ozaki_status_string(code: int) -> str:
    return _lib.ozaki_status_string(code).decode()


def exported_symbols() -> list[str]:
    """Names the loaded library exports among those ``include/ozaki.h`` declares."""
    return [name for name in _declared_names() if hasattr(_lib, name)]


def _declared_names() -> list[str]:
    import re

    hdr = os.path.join(os.path.dirname(_PKG), "include", "ozaki.h")
    with open(hdr) as f:
        text = f.read()
    return re.findall(r"^(?:int|size_t|const char\*)\s+(\w+)\s*\(", text, flags=re.M)
