// oz_internal.h -- declarations shared by the host orchestration and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "ozaki.h"

namespace oz {

constexpr int kMaxModuli = OZ_MAX_MODULI;
constexpr int kLimbs = 6;        // 32-bit limbs for CRT values (M < 2^160 for 20 moduli)
constexpr int kHalfLimbs = 10;   // 16-bit limbs of the CRT constants (M < 2^160)
constexpr int kPadM = 256;       // plane row padding (A rows, C_res rows)
constexpr int kPadN = 256;       // plane row padding (B columns, C_res columns)
constexpr int kPadK = 64;        // plane K padding (one 128-byte bf16 row of a stage)

inline int64_t roundup(int64_t x, int64_t r) { return (x + r - 1) / r * r; }

// Per-modulus constants for the residue split (a2).
struct SplitConsts {
  int s;
  int kA;                       // k_A = k_B
  int mod[kMaxModuli];
  uint32_t c16[kMaxModuli];     // 2^16 mod m
  uint32_t c32[kMaxModuli];     // 2^32 mod m
  uint32_t c48[kMaxModuli];     // 2^48 mod m
  uint32_t c64[kMaxModuli];     // 2^64 mod m
  uint32_t c80[kMaxModuli];     // 2^80 mod m
  uint32_t magic[kMaxModuli];   // ceil(2^39 / m): y mod m for y < 2^30
  uint32_t offs[kMaxModuli];    // m 2^22 + floor(m/2): the offset of the single Barrett step
  uint32_t fbase[kMaxModuli];   // 0x4B000080 - floor(m/2): float bits of 2^23 + 128, shifted
  int shift_ok;                 // every modulus m has m 2^22 > 2^26 (the shifted path's bound)
  // The 13-bit limb path (a' < 2^52 as four 13-bit limbs, FP32 arithmetic):
  float f13[kMaxModuli];        // 2^13 mod m, 2^26 mod m, 2^39 mod m
  float f26[kMaxModuli];
  float f39[kMaxModuli];
  float finv[kMaxModuli];       // 1/m rounded to FP32
  float fmod[kMaxModuli];       // m
  int limb13_ok;                // m_0 = 256 and every other modulus odd, in (128, 256)
};

// Constants of the CRT reconstruction (a5, a6).
struct CrtConsts {
  int s;
  int kA;
  int mod[kMaxModuli];
  uint32_t P[kMaxModuli][kLimbs];  // M_t * y_t (< M), little-endian limbs
  int n16;                         // 16-bit limbs holding M (and every P_t < M)
  // limb l of P_{2p} in the low half and of P_{2p+1} in the high half (zero past s)
  uint32_t Pd[kMaxModuli / 2][kHalfLimbs];
  uint32_t M[kLimbs];
  uint32_t halfM[kLimbs];          // floor(M / 2)
  uint32_t Mneg[kLimbs];           // 2^(32 NL) - M for the launch's word count NL (set by launch_crt)
};

constexpr int kMaxPairs = OZ_MAX_SLICES * (OZ_MAX_SLICES + 1) / 2;  // Scheme I products

// Work description of the tcgen05 GEMM engine.  Each work unit is a (tile, product)
// pair; product p multiplies A plane a_plane[p] by B plane b_plane[p].
//   residue mode (Scheme II): product t = modulus t, planes t and t, epilogue mod m_t;
//   exact mode (Scheme I):    product p = slice pair (i, j), exact INT32 output.
// The Scheme I accumulation reads the same structure: with grouped set, its batch t is the
// sum of the pair products prod_first[t] .. prod_first[t+1]-1 (group-wise accumulation).
struct GemmConsts {
  int s;              // number of products
  int kb_per_chunk;   // k-blocks of 64 whose FP32 sum stays exact
  int kb_per_block;   // k-blocks of 64 per scheduling K-block (a multiple of kb_per_chunk)
  uint32_t launch_id; // selects this launch's pacing counter
  int grouped;        // accumulation only: the number of batches in prod_first (0: none)
  unsigned long long epi_wait_ns;  // time limit of the epilogue's wait for an accumulator
  float modf[kMaxModuli];
  float invf[kMaxModuli];
  uint8_t a_plane[kMaxPairs];
  uint8_t b_plane[kMaxPairs];
  uint8_t prod_first[kMaxPairs + 1];
};

// Host-side helpers (ozaki_host.cu).
int fill_split_consts(int s, long long k_inner, SplitConsts* out);
int fill_crt_consts(int s, long long k_inner, CrtConsts* out);
int half_range_log2(int s);  // L = floor(log2(M/2 - 1)) for the first s moduli; -1 on error

// Kernel launchers; each returns a cudaError_t from the launch.
cudaError_t launch_exponents(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                             int32_t* rowexp, int32_t* colexp, cudaStream_t stream);
cudaError_t launch_floor_exponents(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                                   int32_t* rowexp, int32_t* colexp, cudaStream_t stream);
cudaError_t launch_split(int rows, int k, const double* X, long long row_stride, long long k_stride,
                         const int32_t* exps, const SplitConsts& c, uint16_t* planes, int rows_padded,
                         int kp, cudaStream_t stream);
cudaError_t launch_split_fused_kcontig(int rows, int k, const double* X, long long ld, const SplitConsts& c,
                                       int32_t* exps, uint16_t* planes, int rows_padded, int kp,
                                       cudaStream_t stream);
int launch_residue_gemm(int mp, int np, int kp, const GemmConsts& c, const uint16_t* A_planes,
                        const uint16_t* B_planes, uint8_t* C_res, cudaStream_t stream);
int launch_slice_gemm(int mp, int np, int kp, int a_planes, int b_planes, const GemmConsts& c,
                      const uint16_t* A_planes, const uint16_t* B_planes, int32_t* out, cudaStream_t stream);
int launch_bound_gemm(int mp, int np, int kp, const uint16_t* A_plane, const uint16_t* B_plane, uint32_t* maxes,
                      cudaStream_t stream);
cudaError_t launch_norm_exponents(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                                  int32_t* rowexp, int32_t* colexp, unsigned long long* Srow,
                                  unsigned long long* Scol, cudaStream_t stream);
cudaError_t launch_magnitudes(int rows, int k, const double* X, long long row_stride, long long k_stride,
                              const int32_t* exps, int b, uint16_t* plane, int rows_padded, int kp,
                              cudaStream_t stream);
cudaError_t launch_accu_finalize(int count, int32_t* exps, const uint32_t* maxes, int L, int kappa, int b,
                                 cudaStream_t stream);
cudaError_t launch_crt(int m, int n, int mp, int np, const CrtConsts& c, const uint8_t* C_res,
                       const int32_t* rowexp, const int32_t* colexp, double* C, int ldc, cudaStream_t stream);
cudaError_t launch_fill_zero(int m, int n, double* C, int ldc, cudaStream_t stream);

// Device status word (set by kernels whose bounded waits expired).
int* device_status_ptr();

// Time limit of the GEMM epilogue's accumulator wait for the launches that follow
// (ozaki_set_epilogue_wait_ns).
unsigned long long epilogue_wait_ns();

}  // namespace oz
