// oz_exponents.cu -- step a1: per-row / per-column ceil(log2 max |x|) (and the floor
// variant the Scheme I bitmask split uses).
//
// [Ozaki II] section 3 scales A by D = diag(2^d_i) and B by E = diag(2^e_j); the
// exponents d_i = k_A - E_i need E_i = ceil(log2 max_j |a_ij|) = max_j ceil(log2 |a_ij|)
// (ceil(log2 .) is monotone).  The magnitude bits of an IEEE-754 double order like its
// magnitude (subnormals, infinity and NaN included), so the kernels reduce the 63-bit
// magnitude patterns with an integer max and take ceil(log2 .) (exactly, from the bit
// fields) of the maximum alone.  HBM-bound: one read of A and B.
#include "oz_fp.cuh"
#include "oz_internal.h"

namespace oz {

constexpr int kRowExpCols = 64;   // columns of A per block (row-maximum kernel)
constexpr int kColExpRows = 1024; // rows of B per warp (column-maximum kernel)

// A column-major (m x k): thread = row i, loop over a slice of columns.
template <bool kFloor>
__global__ void __launch_bounds__(256) rowexp_colmajor_kernel(int m, int k, const double* __restrict__ A,
                                                              long long lda, int32_t* __restrict__ rowexp) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= m) return;
  const int j0 = blockIdx.y * kRowExpCols;
  const int j1 = min(k, j0 + kRowExpCols);
  const double* p = A + i + static_cast<long long>(j0) * lda;
  unsigned long long mag = 0;
#pragma unroll 16
  for (int j = j0; j < j1; ++j, p += lda) mag = max(mag, magnitude_bits(__ldg(p)));
  if (mag != 0) atomicMax(&rowexp[i], log2_code<kFloor>(__longlong_as_double(static_cast<long long>(mag))));
}

// B column-major (k x n): warp = one column j and a slice of kColExpRows rows.
template <bool kFloor>
__global__ void __launch_bounds__(256) colexp_colmajor_kernel(int k, int n, const double* __restrict__ B,
                                                              long long ldb, int32_t* __restrict__ colexp) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = blockIdx.x * 8 + warp;
  if (j >= n) return;
  const int r0 = blockIdx.y * kColExpRows;
  const int r1 = min(k, r0 + kColExpRows);
  const double* col = B + static_cast<long long>(j) * ldb;
  unsigned long long mag = 0;
#pragma unroll 16
  for (int r = r0 + lane; r < r1; r += 32) mag = max(mag, magnitude_bits(__ldg(col + r)));
  int best = mag ? log2_code<kFloor>(__longlong_as_double(static_cast<long long>(mag))) : OZ_EXP_EMPTY;
  best = __reduce_max_sync(0xFFFFFFFFu, best);
  if (lane == 0 && best != OZ_EXP_EMPTY) atomicMax(&colexp[j], best);
}

template <bool kFloor>
static cudaError_t launch_exponents_t(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                                      int32_t* rowexp, int32_t* colexp, cudaStream_t stream) {
  if (A && m > 0) {
    cudaError_t e = cudaMemsetAsync(rowexp, 0x80, sizeof(int32_t) * m, stream);  // OZ_EXP_EMPTY
    if (e != cudaSuccess) return e;
    if (k > 0) {
      dim3 grid((m + 255) / 256, (k + kRowExpCols - 1) / kRowExpCols);
      rowexp_colmajor_kernel<kFloor><<<grid, 256, 0, stream>>>(m, k, A, lda, rowexp);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  if (B && n > 0) {
    cudaError_t e = cudaMemsetAsync(colexp, 0x80, sizeof(int32_t) * n, stream);
    if (e != cudaSuccess) return e;
    if (k > 0) {
      dim3 grid((n + 7) / 8, (k + kColExpRows - 1) / kColExpRows);
      colexp_colmajor_kernel<kFloor><<<grid, 256, 0, stream>>>(k, n, B, ldb, colexp);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

cudaError_t launch_exponents(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                             int32_t* rowexp, int32_t* colexp, cudaStream_t stream) {
  return launch_exponents_t<false>(m, n, k, A, lda, B, ldb, rowexp, colexp, stream);
}

cudaError_t launch_floor_exponents(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                                   int32_t* rowexp, int32_t* colexp, cudaStream_t stream) {
  return launch_exponents_t<true>(m, n, k, A, lda, B, ldb, rowexp, colexp, stream);
}

__global__ void fill_zero_kernel(int m, int n, double* C, long long ldc) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(m) * n) return;
  const int i = static_cast<int>(idx % m), j = static_cast<int>(idx / m);
  C[i + j * ldc] = 0.0;
}

cudaError_t launch_fill_zero(int m, int n, double* C, int ldc, cudaStream_t stream) {
  const long long total = static_cast<long long>(m) * n;
  if (total == 0) return cudaSuccess;
  fill_zero_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, stream>>>(m, n, C, ldc);
  return cudaGetLastError();
}

}  // namespace oz
