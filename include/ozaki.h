/*
 * ozaki.h -- C ABI of libozaki: FP64 matrix multiplication emulated on low-precision
 * tensor cores with the Ozaki scheme, for NVIDIA GB300 (sm_103a).
 *
 * Method: "Ozaki Scheme II: mapping high-precision GEMM to a few INT8 GEMMs with CRT"
 * (explainer of Ozaki, Uchino, Imamura, arXiv:2504.08009), cited below as [Ozaki II];
 * Algorithm 1 is in its section 7 (steps 1-6).  Scheme I follows the "Ozaki Scheme"
 * course notes (SplitFP / RN split / triangular products), cited as [Ozaki notes].
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Matrices are column-major with leading dimensions (BLAS / cuBLAS convention):
 *    A is m x k (lda >= max(1,m)), B is k x n (ldb >= max(1,k)), C is m x n
 *    (ldc >= max(1,m)).  The operation is C = A*B: no alpha/beta, no transposes,
 *    C is overwritten.
 *  - Unless a name ends in _host, every pointer is DEVICE memory owned by the caller;
 *    the library never frees it.  Calls are asynchronous and ordered on `stream`
 *    (0 = legacy default stream); nothing synchronises the device implicitly.
 *  - Return value: OZ_OK (0) or a negative oz_status.  Argument errors are reported
 *    synchronously before anything is launched.  A device-side failure (a bounded wait
 *    inside a kernel that expired) is recorded in a device status word that
 *    ozaki_get_device_status(stream) returns.
 *  - m, n or k equal to 0: nothing is read; for k = 0 (m, n > 0) C is set to +0.0.
 *  - Inputs holding Inf or NaN: the affected rows of C (row of A) and columns of C
 *    (column of B) are set to NaN; nothing traps.
 *
 * Scheme II workspace layout (what the step entry points read and write)
 * ----------------------------------------------------------------------
 *  Let Mp = roundup(m, 256), Np = roundup(n, 256), Kp = roundup(k, 64), s = num_moduli.
 *  - rowexp[m], colexp[n] (int32): E_i = ceil(log2 max_j |a_ij|) and
 *    F_j = ceil(log2 max_l |b_lj|); OZ_EXP_EMPTY for an all-zero row/column,
 *    OZ_EXP_NONFINITE when it holds Inf/NaN.
 *  - A_planes [s][Mp][Kp] and B_planes [s][Np][Kp]: bf16 bit patterns (uint16) holding
 *    the symmetric residues A'_t = A' mod m_t and B'_t = B' mod m_t, integers in
 *    [-128, 127] that bf16 represents exactly.  Row i of A_planes[t] is row i of A'_t
 *    (K contiguous); row j of B_planes[t] is column j of B'_t (K contiguous).  Padding
 *    rows / columns are zero.
 *  - C_res [s][Np][Mp] (uint8): C''_t = (A'_t B'_t) mod m_t in [0, m_t), column-major
 *    per modulus (element (i,j) of plane t at t*Np*Mp + j*Mp + i).
 */
#ifndef OZAKI_H
#define OZAKI_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  OZ_OK = 0,
  OZ_EINVAL = -1,   /* invalid argument (dimension, leading dimension, count, null) */
  OZ_ERANGE = -2,   /* too few moduli for this k: k_A would be < 1 */
  OZ_ECUDA = -3,    /* a CUDA runtime call or kernel launch failed */
  OZ_ENOMEM = -4,   /* workspace allocation failed or the given workspace is too small */
  OZ_ETIMEOUT = -5, /* device side: a bounded wait in a kernel expired (status word) */
  OZ_ENODEV = -6    /* no usable sm_103 device */
} oz_status;

#define OZ_MAX_MODULI 20
#define OZ_MIN_MODULI 2
#define OZ_MAX_SLICES 20
#define OZ_EXP_EMPTY ((int32_t)0x80808080)
#define OZ_EXP_NONFINITE ((int32_t)0x7fffffff)

/* ---------------------------------------------------------------- host-only queries */

/* The first num_moduli moduli of the greedy descending pairwise-coprime list starting
 * at 256 ([Ozaki II] sections 4 and 6: 2 <= m_t <= 256, pairwise coprime).  Writes
 * num_moduli ints to moduli_out (host memory).  OZ_EINVAL if num_moduli is outside
 * [1, OZ_MAX_MODULI] or moduli_out is NULL.  No GPU needed. */
int ozaki2_moduli(int num_moduli, int* moduli_out);

/* k_A = k_B of [Ozaki II] section 5: the largest integer k with
 * k_inner * 2^(2k) <= M/2 - 1, M the product of the moduli.  *k_out receives it.
 * OZ_ERANGE if no k >= 1 exists.  No GPU needed. */
int ozaki2_choose_k(int num_moduli, long long k_inner, int* k_out);

/* Padded plane dimensions Mp, Np, Kp (see the layout above).  No GPU needed. */
int ozaki2_plane_dims(int m, int n, int k, int* mp, int* np, int* kp);

/* Bytes of device workspace ozaki2_dgemm_ws needs (0 on invalid arguments). */
size_t ozaki2_workspace_bytes(int m, int n, int k, int num_moduli);

/* ---------------------------------------------------------------- Scheme II steps */

/* Step a1 ([Ozaki II] section 3 and Algorithm 1 step 2, the choice of D and E):
 * rowexp[i] = max_j ceil(log2 |a_ij|), colexp[j] = max_l ceil(log2 |b_lj|), with the
 * markers OZ_EXP_EMPTY / OZ_EXP_NONFINITE.  rowexp has m ints, colexp n ints. */
int ozaki2_exponents(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                     int32_t* rowexp, int32_t* colexp, cudaStream_t stream);

/* Step a2 (Algorithm 1 steps 2-3, left half): A' = trunc(D A) with
 * D_ii = 2^(k_A - rowexp[i]), B' = trunc(B E) likewise, then the symmetric residues
 * mod each of the first num_moduli moduli, written as bf16 planes (layout above).
 * Either operand may be skipped by passing NULL for its source and planes. */
int ozaki2_split(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                 int num_moduli, const int32_t* rowexp, const int32_t* colexp,
                 uint16_t* A_planes, uint16_t* B_planes, cudaStream_t stream);

/* Steps a1 and a2 together (Algorithm 1 steps 2-3, left half): the exponents of
 * ozaki2_exponents and the planes of ozaki2_split, same arguments, layouts and errors, in
 * fewer passes over DRAM: while Kp <= 16384 each column of B is read from DRAM once (its
 * maximum, then its residues, the second read served by L2); A, and B at larger k, take the
 * exponent pass and the split.  Everything is ordered on `stream`.  Either operand may be
 * skipped with NULL for its source, exponents and planes. */
int ozaki2_scale_split(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                       int num_moduli, int32_t* rowexp, int32_t* colexp, uint16_t* A_planes,
                       uint16_t* B_planes, cudaStream_t stream);

/* Steps a3+a4 (Algorithm 1 step 3): for every modulus t, the exact integer product
 * C'_t = A'_t B'_t on the tensor cores and C''_t = C'_t mod m_t, written to C_res.
 * Exact for every k: each run of 1024 terms of the k loop is summed exactly on the
 * tensor cores and folded mod m_t before the next starts. */
int ozaki2_residue_gemm(int m, int n, int k, int num_moduli, const uint16_t* A_planes,
                        const uint16_t* B_planes, uint8_t* C_res, cudaStream_t stream);

/* Steps a5+a6 (Algorithm 1 steps 4-6): Z = sum_t C''_t M_t y_t, C''' = Z mod M (the
 * symmetric representative), C_ij = RN(C'''_ij * 2^-(d_i + e_j)) with one rounding
 * (round-to-nearest-even, subnormals included, +-inf on overflow). */
int ozaki2_crt(int m, int n, int k, int num_moduli, const uint8_t* C_res,
               const int32_t* rowexp, const int32_t* colexp, double* C, int ldc,
               cudaStream_t stream);

/* ---------------------------------------------------------------- Scheme II, composed */

/* C = A*B by Ozaki Scheme II with num_moduli in [OZ_MIN_MODULI, OZ_MAX_MODULI] moduli,
 * using the caller's device workspace (ws_bytes >= ozaki2_workspace_bytes(...), base
 * aligned to 256 bytes).  OZ_ENOMEM if the workspace is too small. */
int ozaki2_dgemm_ws(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                    double* C, int ldc, int num_moduli, void* workspace, size_t ws_bytes,
                    cudaStream_t stream);

/* Same, with the workspace taken from and returned to the stream-ordered allocator
 * (cudaMallocAsync / cudaFreeAsync on `stream`).  On first use per device the library
 * raises the release threshold of that device's default memory pool so freed
 * workspace stays cached for the next call (a process-wide setting of that pool). */
int ozaki2_dgemm(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                 double* C, int ldc, int num_moduli, cudaStream_t stream);

/* Same with HOST pointers: copies A and B to the current device, computes, copies C
 * back and synchronises before returning (a drop-in CPU-callable DGEMM). */
int ozaki2_dgemm_host(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                      double* C, int ldc, int num_moduli);

/* ---------------------------------------------------------------- Scheme II range estimation */

/* How the scaling exponents keep the CRT result unique ([Ozaki II] sections 5 and 9):
 * every mode guarantees max_ij (|A'||B'|)_ij <= M/2 - 1 and writes exponent codes t
 * with d_i = k - t_i (row i of A) and e_j = k - t_j (column j of B), where k is the
 * value ozaki2_scaling_k returns.  OZ_EXP_EMPTY / OZ_EXP_NONFINITE keep their meaning.
 *  OZ_SCALE_UNIFORM: c_max = q 2^(k_A + k_B); t_i = ceil(log2 max_j |a_ij|), k = k_A
 *    (the mode of every entry point without _ex).
 *  OZ_SCALE_FAST (OS II-fast, Cauchy-Schwarz): 2^t_i >= ||a_i,:||_2, computed from
 *    exact integers (c_l = ceil(log2 |a_il|), G = 16, S = sum_l max(1, 4^(c_l - c_max + G)),
 *    t = c_max - G + ceil(ceil(log2 S) / 2)); k = kappa = the largest k with
 *    2^(2k) <= M/2 - 1.
 *  OZ_SCALE_ACCU (OS II-accu, a low-precision product): magnitudes rounded up to b bits
 *    of each row's range (b = the largest integer <= 7 with q 4^b <= 2^24), their
 *    exact product C^ on the tensor cores (one bf16 GEMM), rho_i = max(1, max_j C^_ij),
 *    gamma_j likewise, L = floor(log2(M/2 - 1)),
 *    t_i = kappa - floor((L - ceil(log2 rho_i)) / 2) + ceil(log2 max_j |a_ij|) - b.
 *    Needs k <= 2^24 (OZ_EINVAL otherwise). */
#define OZ_SCALE_UNIFORM 0
#define OZ_SCALE_FAST 1
#define OZ_SCALE_ACCU 2

/* k of the scaling mode for num_moduli and the inner dimension k_inner (host only).
 * OZ_ERANGE as ozaki2_choose_k; OZ_EINVAL for an unknown mode or, for OZ_SCALE_ACCU,
 * k_inner > 2^24. */
int ozaki2_scaling_k(int num_moduli, long long k_inner, int scaling, int* k_out);

/* Device scratch bytes ozaki2_exponents_ex needs: 0 (uniform), 8(m + n) (fast),
 * 2 Kp (Mp + Np) + 4 (Mp + Np) plus alignment (accu). */
size_t ozaki2_exponents_workspace_bytes(int m, int n, int k, int scaling);

/* Step a1 in a given scaling mode: writes rowexp[m] (if A) and colexp[n] (if B).
 * OZ_SCALE_ACCU needs both operands.  workspace: device memory of at least
 * ozaki2_exponents_workspace_bytes bytes, 256-byte aligned (OZ_ENOMEM otherwise; may
 * be null when that is 0).  num_moduli fixes M (unused by uniform and fast). */
int ozaki2_exponents_ex(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                        int num_moduli, int scaling, int32_t* rowexp, int32_t* colexp,
                        void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Steps a2 and a5 + a6 for exponents of a given scaling mode (same layouts and errors
 * as ozaki2_split and ozaki2_crt, which are these with OZ_SCALE_UNIFORM). */
int ozaki2_split_ex(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                    int num_moduli, int scaling, const int32_t* rowexp, const int32_t* colexp,
                    uint16_t* A_planes, uint16_t* B_planes, cudaStream_t stream);
int ozaki2_crt_ex(int m, int n, int k, int num_moduli, int scaling, const uint8_t* C_res,
                  const int32_t* rowexp, const int32_t* colexp, double* C, int ldc,
                  cudaStream_t stream);

/* The whole path in a given scaling mode: workspace bytes, caller-owned workspace,
 * stream-ordered allocation (as ozaki2_dgemm_ws / ozaki2_dgemm). */
size_t ozaki2_workspace_bytes_ex(int m, int n, int k, int num_moduli, int scaling);
int ozaki2_dgemm_ex_ws(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                       double* C, int ldc, int num_moduli, int scaling, void* workspace,
                       size_t ws_bytes, cudaStream_t stream);
int ozaki2_dgemm_ex(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                    double* C, int ldc, int num_moduli, int scaling, cudaStream_t stream);

/* ---------------------------------------------------------------- Scheme I (comparison path) */

/* Scheme I ([Ozaki notes]: RN split of Uchino et al., the triangular integer products
 * i + j <= s + 1, FP64 accumulation).  Layout of its intermediates:
 *  - A_planes [s][Mp][Kp], B_planes [s][Np][Kp]: bf16 bit patterns of the integer slices
 *    (|slice| <= 2^(beta-1) <= 64, exact in bf16), same orientation as Scheme II's planes;
 *  - A_exps [s][m], B_exps [s][n] (int32): slice p of row i of A is
 *    A_planes[p][i][:] * 2^A_exps[p][i] (0 for rows that are zero at that slice);
 *  - products [s(s+1)/2][Np][Mp] (int32, column-major per product): the exact product
 *    A'_i B'_j for the pairs (i, j) in the order i = 1..s outside, j = 1..s-i+1 inside.
 * Supported inputs: finite, with every row maximum of A and column maximum of B in
 * [2^-1000, 2^960] or zero (the rounding constants 0.75 * 2^53 * mu must be finite and mu
 * normal). */

/* beta = min(7, floor((31 - log2 k_inner) / 2)) ([Ozaki notes], RN split step 1):
 * slice width in bits.  OZ_ERANGE if beta < 1.  No GPU needed. */
int ozaki1_beta(long long k_inner, int* beta_out);

/* Device scratch ozaki1_split needs for the residuals and row maxima. */
size_t ozaki1_split_scratch_bytes(int m, int n, int k);

/* Bytes of device workspace ozaki1_dgemm_ws needs (0 on invalid arguments). */
size_t ozaki1_workspace_bytes(int m, int n, int k, int num_slices);

/* RN split of the rows of A and the columns of B into num_slices (1..OZ_MAX_SLICES)
 * integer slices each (remainder dropped): planes and slice exponents as above.  Either
 * operand may be skipped with NULL.  scratch: device memory of at least
 * ozaki1_split_scratch_bytes(m, n, k) bytes, 256-byte aligned. */
int ozaki1_split(int m, int n, int k, const double* A, int lda, const double* B, int ldb, int num_slices,
                 uint16_t* A_planes, uint16_t* B_planes, int32_t* A_exps, int32_t* B_exps,
                 void* scratch, size_t scratch_bytes, cudaStream_t stream);

/* The s(s+1)/2 exact integer products A'_i B'_j (tensor cores, INT32 output). */
int ozaki1_slice_gemm(int m, int n, int k, int num_slices, const uint16_t* A_planes,
                      const uint16_t* B_planes, int32_t* products, cudaStream_t stream);

/* C = sum over the pairs, in order, of diag(2^A_exps[i]) P_ij diag(2^B_exps[j]), every term
 * exact, accumulated with FP64 round-to-nearest additions starting from +0. */
int ozaki1_accumulate(int m, int n, int k, int num_slices, const int32_t* products,
                      const int32_t* A_exps, const int32_t* B_exps, double* C, int ldc,
                      cudaStream_t stream);

/* C = A*B by Scheme I with a caller-owned workspace / with a stream-ordered one. */
int ozaki1_dgemm_ws(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                    double* C, int ldc, int num_slices, void* workspace, size_t ws_bytes,
                    cudaStream_t stream);
int ozaki1_dgemm(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                 double* C, int ldc, int num_slices, cudaStream_t stream);
/* ---------------------------------------------------------------- Scheme I variants */

/* [Ozaki notes], "group-wise error-free accumulation" and "Hybrid":
 *  OZ_OZAKI1_RN:     the RN split and one FP64 addition per slice product (the entry points
 *                    above);
 *  OZ_OZAKI1_EF:     the bitmask split (SplitInt): with e_i = floor(log2 max_j |a_ij|),
 *                    slice p of a_ij is the p-th beta-bit field of |a_ij| below 2^(e_i + 1)
 *                    (truncation), signed, scale 2^(e_i + 1 - p beta); A_exps[p][i] holds
 *                    e_i + 1 - (p+1) beta (p 0-based), 0 for zero rows;
 *  OZ_OZAKI1_HYBRID: the RN split with the fixed grid mu''_i = 2^(ceil(log2 max_j |a_ij|)
 *                    + 1 - beta) lowered by 2^beta per slice (sigma = 0.75 2^(53 - beta p)
 *                    mu''_i for 0-based p); A_exps[p][i] = log2 of that grid.
 * EF and Hybrid accumulate group-wise: the pair products are ordered by group g = i + j
 * (g = 2..s+1, i = 1..g-1 ascending) and products[t] is pair t in that order; the pairs
 * of a group are summed exactly in INT32 in batches of r = max(1, 2^(31 - 2 beta -
 * ceil(log2 k))) (ozaki1_group_r), and C = sum over the batches, in order, of the batch
 * scaled by the power of two of its group, one FP64 round-to-nearest addition each, from +0.
 * Hybrid supports row maxima in [2^(beta s - 1022), 2^960] (every grid a normal number);
 * EF supports any finite input. */
#define OZ_OZAKI1_RN 0
#define OZ_OZAKI1_EF 1
#define OZ_OZAKI1_HYBRID 2

/* r for the inner dimension k_inner (host only; OZ_ERANGE as ozaki1_beta). */
int ozaki1_group_r(long long k_inner, int* r_out);

/* Terms of the FP64 accumulation for a variant: s(s+1)/2 pairs (RN) or the number of
 * group batches (EF, Hybrid).  Every variant's slice GEMM writes s(s+1)/2 INT32 planes. */
int ozaki1_num_batches(int num_slices, long long k_inner, int variant, int* count_out);

/* Scratch of ozaki1_split_ex and workspace of ozaki1_dgemm_ex_ws for a variant. */
size_t ozaki1_split_scratch_bytes_ex(int m, int n, int k, int variant);
size_t ozaki1_workspace_bytes_ex(int m, int n, int k, int num_slices, int variant);

/* The steps and the whole product for a variant (layouts as for the RN entry points;
 * products holds s(s+1)/2 planes [pair][Np][Mp] of int32, pairs in the variant's order). */
int ozaki1_split_ex(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                    int num_slices, int variant, uint16_t* A_planes, uint16_t* B_planes,
                    int32_t* A_exps, int32_t* B_exps, void* scratch, size_t scratch_bytes,
                    cudaStream_t stream);
int ozaki1_slice_gemm_ex(int m, int n, int k, int num_slices, int variant,
                         const uint16_t* A_planes, const uint16_t* B_planes, int32_t* products,
                         cudaStream_t stream);
int ozaki1_accumulate_ex(int m, int n, int k, int num_slices, int variant,
                         const int32_t* products, const int32_t* A_exps, const int32_t* B_exps,
                         double* C, int ldc, cudaStream_t stream);
int ozaki1_dgemm_ex_ws(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                       double* C, int ldc, int num_slices, int variant, void* workspace,
                       size_t ws_bytes, cudaStream_t stream);
int ozaki1_dgemm_ex(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                    double* C, int ldc, int num_slices, int variant, cudaStream_t stream);


/* ---------------------------------------------------------------- without allocation */

/* Size of the fixed scratch buffer ozaki2_dgemm_noalloc uses (64 MiB). */
#define OZ_NOALLOC_SCRATCH_BYTES (64u << 20)

/* C = A*B like ozaki2_dgemm, for callers that cannot allocate device memory when they
 * multiply (for example a process whose memory manager owns the whole GPU, or a loop
 * that must not allocate after start-up).  The pages have no counterpart: this is a
 * library convenience.  Nothing is allocated: the workspace is a fixed buffer of
 * OZ_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads the library
 * holds until the process exits.  Problems whose ozaki2_workspace_bytes(m, n, k,
 * num_moduli) exceeds it are rejected with OZ_ENOMEM before anything runs (at 14 moduli
 * m = n = k = 768 fits, 1024 does not).  The first call on each device looks up the
 * buffer's device address (with that device current) and keeps it for that CUDA context;
 * make that first call before any stream capture.  All calls share the one buffer, which
 * keeps the last call's contents: calls that overlap on the GPU (other streams, other
 * threads) race on it.  Arguments, ordering and errors are those of ozaki2_dgemm, checked
 * in the same order (dimensions, moduli count, null pointers, OZ_ERANGE); the size limit
 * (OZ_ENOMEM) is checked after them. */
int ozaki2_dgemm_noalloc(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                         double* C, int ldc, int num_moduli, cudaStream_t stream);

/* ---------------------------------------------------------------- status */

/* Waits for the work queued on `stream` (0 = legacy default stream), then returns the
 * device status word of the current device (OZ_OK, or OZ_ETIMEOUT if a kernel of this
 * library gave up a bounded wait) and clears it.  The word is one per device: it holds
 * what every kernel of this library on the device recorded up to the read, whatever
 * stream launched it; a kernel still running on another stream may record later.  The
 * read and the clear are ordered on `stream`.  OZ_ECUDA if a CUDA call fails. */
int ozaki_get_device_status(cudaStream_t stream);

/* Time limit, in nanoseconds, of one wait inside the tensor-core GEMM kernels launched
 * after this call: the epilogue's wait for an accumulator of exact sums.  -1 restores the
 * default of 4 s; 0 makes the wait give up as soon as it finds the accumulator not ready,
 * so that a test can drive the failure path on purpose.  On expiry the kernel records
 * OZ_ETIMEOUT in the device status word, stops both CTAs of the pair, waits for every copy
 * and MMA it issued, frees its tensor memory and returns; its outputs are then undefined.
 * A process-wide setting.  The pages have no counterpart: this is a library facility for
 * exercising failure detection.  OZ_EINVAL for ns < -1. */
int ozaki_set_epilogue_wait_ns(long long ns);

/* Human-readable name of a status code (static string). */
const char* ozaki_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* OZAKI_H */
