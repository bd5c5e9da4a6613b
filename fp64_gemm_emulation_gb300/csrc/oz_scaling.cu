// oz_scaling.cu -- the range estimation variants of [Ozaki II] section 9.
//
// The CRT result is unique while max_ij (|A'||B'|)_ij <= M/2 - 1 (section 5).  The
// uniform estimate bounds it by q 2^(k_A + k_B) (oz_exponents.cu).  The two variants
// here keep d_i = kappa - t_i, kappa the largest k with 2^(2k) <= M/2 - 1, and compute
// a per-row (per-column) exponent t_i:
//
//  OS II-fast (Cauchy-Schwarz): (|A'||B'|)_ij <= ||A'_i,:||_2 ||B'_:,j||_2 and
//    2^t_i >= ||a_i,:||_2.  With c = ceil(log2 |a_ik|) (exact, from the bits) and
//    G = 16, S_i = sum_k max(1, 4^(c - c_max + G)) is an integer sum (so the result
//    does not depend on the summation order) and t_i = c_max - G + ceil(ceil(log2 S_i)/2).
//
//  OS II-accu (a low-precision product): A^_ik = ceil(|a_ik| 2^(b - E_i)) in [0, 2^b],
//    B^ likewise per column, with q 4^b <= 2^24 so one bf16 GEMM with FP32 accumulation
//    computes C^ = A^ B^ exactly; rho_i = max(1, max_j C^_ij), gamma_j over i;
//    t_i = kappa - floor((L - ceil(log2 rho_i)) / 2) + E_i - b, L = floor(log2(M/2 - 1)).
//    Then (|A'||B'|)_ij <= 2^(x_i + y_j) C^_ij <= 2^L since C^_ij <= sqrt(rho_i gamma_j).
//
// Integer bit manipulation only; the bound product runs on the tcgen05 GEMM engine
// (oz_gemm.cu, row/column-maximum epilogue).
#include "oz_fp.cuh"
#include "oz_internal.h"

namespace oz {

constexpr int kNormGuard = 16;      // G
constexpr int kNormCols = 64;       // columns of A per thread (row-norm kernel)
constexpr int kNormRows = 1024;     // rows of B per warp (column-norm kernel)

// max(1, 4^(c - cmax + G)) for one nonzero finite element (c <= cmax), 0 otherwise.
__device__ __forceinline__ unsigned long long norm_term(double x, int cmax) {
  const int c = ceil_log2_code(x);
  if (c == OZ_EXP_EMPTY || c == OZ_EXP_NONFINITE) return 0ull;
  const int d = c - cmax + kNormGuard;
  return d >= 0 ? (1ull << (2 * d)) : 1ull;
}

// A column-major (m x k): thread = row i over a slice of kNormCols columns.
__global__ void __launch_bounds__(256) rownorm_colmajor_kernel(int m, int k, const double* __restrict__ A,
                                                               long long lda, const int32_t* __restrict__ rowexp,
                                                               unsigned long long* __restrict__ S) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= m) return;
  const int cmax = __ldg(rowexp + i);
  if (cmax == OZ_EXP_EMPTY || cmax == OZ_EXP_NONFINITE) return;
  const int j0 = blockIdx.y * kNormCols;
  const int j1 = min(k, j0 + kNormCols);
  const double* p = A + i + static_cast<long long>(j0) * lda;
  unsigned long long sum = 0;
#pragma unroll 16
  for (int j = j0; j < j1; ++j, p += lda) sum += norm_term(__ldg(p), cmax);
  if (sum) atomicAdd(S + i, sum);
}

// B column-major (k x n): warp = one column j over a slice of kNormRows rows.
__global__ void __launch_bounds__(256) colnorm_colmajor_kernel(int k, int n, const double* __restrict__ B,
                                                               long long ldb, const int32_t* __restrict__ colexp,
                                                               unsigned long long* __restrict__ S) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = blockIdx.x * 8 + warp;
  if (j >= n) return;
  const int cmax = __ldg(colexp + j);
  if (cmax == OZ_EXP_EMPTY || cmax == OZ_EXP_NONFINITE) return;
  const int r0 = blockIdx.y * kNormRows;
  const int r1 = min(k, r0 + kNormRows);
  const double* col = B + static_cast<long long>(j) * ldb;
  unsigned long long sum = 0;
#pragma unroll 16
  for (int r = r0 + lane; r < r1; r += 32) sum += norm_term(__ldg(col + r), cmax);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
  if (lane == 0 && sum) atomicAdd(S + j, sum);
}

// t = c_max - G + ceil(ceil(log2 S) / 2), in place over the maxima exponents.
__global__ void norm_finalize_kernel(int count, int32_t* __restrict__ exps, const unsigned long long* __restrict__ S) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= count) return;
  const int c = exps[i];
  if (c == OZ_EXP_EMPTY || c == OZ_EXP_NONFINITE) return;
  const unsigned long long s = S[i];  // >= 4^G: the maximum itself
  const int L = 64 - __clzll(static_cast<long long>(s - 1));
  exps[i] = c - kNormGuard + (L + 1) / 2;
}

cudaError_t launch_norm_exponents(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                                  int32_t* rowexp, int32_t* colexp, unsigned long long* Srow,
                                  unsigned long long* Scol, cudaStream_t stream) {
  cudaError_t e = launch_exponents(m, n, k, A, lda, B, ldb, rowexp, colexp, stream);
  if (e != cudaSuccess || k == 0) return e;
  if (A && m > 0) {
    if ((e = cudaMemsetAsync(Srow, 0, sizeof(unsigned long long) * m, stream)) != cudaSuccess) return e;
    dim3 grid((m + 255) / 256, (k + kNormCols - 1) / kNormCols);
    rownorm_colmajor_kernel<<<grid, 256, 0, stream>>>(m, k, A, lda, rowexp, Srow);
    norm_finalize_kernel<<<(m + 255) / 256, 256, 0, stream>>>(m, rowexp, Srow);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (B && n > 0) {
    if ((e = cudaMemsetAsync(Scol, 0, sizeof(unsigned long long) * n, stream)) != cudaSuccess) return e;
    dim3 grid((n + 7) / 8, (k + kNormRows - 1) / kNormRows);
    colnorm_colmajor_kernel<<<grid, 256, 0, stream>>>(k, n, B, ldb, colexp, Scol);
    norm_finalize_kernel<<<(n + 255) / 256, 256, 0, stream>>>(n, colexp, Scol);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// ------------------------------------------------------------------ OS II-accu
constexpr int kMagTile = 64;
constexpr int kMagThreads = 256;

// bf16 bits of ceil(|x| 2^(b - E)) (an integer in [0, 2^b], exact in bf16); 0 for rows
// without an exponent and for non-finite elements.
__device__ __forceinline__ uint16_t magnitude_bf16(double x, int E, int b) {
  if (E == OZ_EXP_EMPTY || E == OZ_EXP_NONFINITE) return 0;
  const uint64_t bits = static_cast<uint64_t>(__double_as_longlong(x));
  const int ex = static_cast<int>((bits >> 52) & 0x7FF);
  if (ex == 0x7FF) return 0;
  const uint64_t frac = bits & 0x000FFFFFFFFFFFFFull;
  uint64_t mant;
  int e2;
  if (ex == 0) {
    mant = frac;
    e2 = -1074;
  } else {
    mant = frac | (1ull << 52);
    e2 = ex - 1075;
  }
  if (mant == 0) return 0;
  const int sh = e2 + b - E;  // |x| 2^(b - E) = mant 2^sh <= 2^b
  uint32_t v;
  if (sh >= 0) {
    v = static_cast<uint32_t>(mant << sh);
  } else if (-sh >= 64) {
    v = 1;  // nonzero, far below one unit
  } else {
    const int r = -sh;
    v = static_cast<uint32_t>((mant >> r) + ((mant & ((1ull << r) - 1)) ? 1 : 0));  // ceiling
  }
  return static_cast<uint16_t>(__float_as_uint(static_cast<float>(v)) >> 16);
}

// One block = a 64 x 64 tile (rows x k) of one operand; phase 1 reads it along the
// index that is contiguous in memory, phase 2 writes 8 consecutive k (16 bytes) per
// thread into the K-contiguous plane.  Padding rows and columns are written as zero.
template <bool kRowsContiguous>
__global__ void __launch_bounds__(kMagThreads) magnitude_kernel(int rows, int K, const double* __restrict__ X,
                                                                long long rs, long long ks,
                                                                const int32_t* __restrict__ exps, int b,
                                                                uint16_t* __restrict__ plane, int kp) {
  __shared__ uint16_t tile[kMagTile][kMagTile + 2];  // [kk][r]
  const int tid = threadIdx.x;
  const int k0 = blockIdx.x * kMagTile;
  const int r0 = blockIdx.y * kMagTile;
#pragma unroll
  for (int it = 0; it < (kMagTile * kMagTile) / kMagThreads; ++it) {
    int r, kk;
    if (kRowsContiguous) {
      r = tid & 63;
      kk = (tid >> 6) + 4 * it;
    } else {
      kk = tid & 63;
      r = (tid >> 6) + 4 * it;
    }
    const int gr = r0 + r, gk = k0 + kk;
    uint16_t v = 0;
    if (gr < rows && gk < K) v = magnitude_bf16(__ldg(X + gr * rs + gk * ks), __ldg(exps + gr), b);
    tile[kk][r] = v;
  }
  __syncthreads();
#pragma unroll
  for (int it = 0; it < (kMagTile * kMagTile / 8) / kMagThreads; ++it) {
    const int item = tid + kMagThreads * it;
    const int g = item & 7, r = item >> 3;
    uint32_t w[4];
#pragma unroll
    for (int x = 0; x < 4; ++x)
      w[x] = static_cast<uint32_t>(tile[g * 8 + 2 * x][r]) | (static_cast<uint32_t>(tile[g * 8 + 2 * x + 1][r]) << 16);
    *reinterpret_cast<uint4*>(plane + static_cast<long long>(r0 + r) * kp + k0 + g * 8) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

cudaError_t launch_magnitudes(int rows, int k, const double* X, long long row_stride, long long k_stride,
                              const int32_t* exps, int b, uint16_t* plane, int rows_padded, int kp,
                              cudaStream_t stream) {
  dim3 grid(kp / kMagTile, rows_padded / kMagTile);
  if (row_stride == 1)
    magnitude_kernel<true><<<grid, kMagThreads, 0, stream>>>(rows, k, X, row_stride, k_stride, exps, b, plane, kp);
  else
    magnitude_kernel<false><<<grid, kMagThreads, 0, stream>>>(rows, k, X, row_stride, k_stride, exps, b, plane, kp);
  return cudaGetLastError();
}

// t = kappa - floor((L - ceil(log2 max(1, rho))) / 2) + E - b, in place over E.
// maxes holds the FP32 bit patterns of exact non-negative integers (<= 2^24).
__global__ void accu_finalize_kernel(int count, int32_t* __restrict__ exps, const uint32_t* __restrict__ maxes,
                                     int L, int kappa, int b) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= count) return;
  const int E = exps[i];
  if (E == OZ_EXP_EMPTY || E == OZ_EXP_NONFINITE) return;
  uint32_t rho = static_cast<uint32_t>(__uint_as_float(maxes[i]));
  rho = rho < 1u ? 1u : rho;
  const int lam = 32 - __clz(static_cast<int>(rho - 1));
  const int num = L - lam;
  const int x = num >= 0 ? num / 2 : -((1 - num) / 2);  // floor(num / 2)
  exps[i] = kappa - x + E - b;
}

cudaError_t launch_accu_finalize(int count, int32_t* exps, const uint32_t* maxes, int L, int kappa, int b,
                                 cudaStream_t stream) {
  if (count <= 0) return cudaSuccess;
  accu_finalize_kernel<<<(count + 255) / 256, 256, 0, stream>>>(count, exps, maxes, L, kappa, b);
  return cudaGetLastError();
}

}  // namespace oz
