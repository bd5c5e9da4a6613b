// oz_ozaki1.cu -- Ozaki Scheme I: RN split, triangular slice products, FP64 accumulation.
//
// [Ozaki notes], RN split of Uchino et al. (step 1: beta = min(7, floor((31 - log2 q)/2));
// steps 3-7 per slice: mu_i = 2^(ceil(log2 max_j |r_ij|) + 1 - beta),
// sigma_i = 0.75 * 2^53 * mu_i, S = (r + sigma) - sigma in round-to-nearest, the
// integer slice S / mu_i, r <- r - S), which is SplitFP's sigma with alpha = beta; then the
// integer matrix-multiplication algorithm: C = sum over i + j <= s + 1 of
// diag(mu_A^(i)) (A'_i B'_j) diag(mu_B^(j)), i ascending outside, j ascending inside,
// each product exact in INT32 and the sum taken in FP64 in that fixed order.
//
// GPU mapping:
//   * rn_split_pass (one launch per slice and operand): reads the residual tile,
//     rounds it to the slice grid exactly as the magic-constant double operations do
//     (round half to even, done on the integer significand so the few FP64 units are not
//     needed), writes the new residual, the slice as a bf16 plane row (K contiguous, exact:
//     |slice| <= 64) and the row maximum of the new residual for the next pass (atomicMax
//     of ceil(log2 |.|));
//   * the slice products run on the tcgen05 engine in exact mode (oz_gemm.cu);
//   * ozaki1 accumulation: one thread per output element, the s(s+1)/2 exact terms
//     added in the fixed order with double-precision round-to-nearest additions.
#include <cmath>
#include <cstring>

#include "oz_fp.cuh"
#include "oz_internal.h"

namespace oz {

constexpr int kTile = 64;
constexpr int kThreads = 256;

// (-1)^neg mag 2^e2 as a double (mag < 2^53, e2 >= -1074: always representable); +0 for mag = 0.
__device__ __forceinline__ double compose_double(bool neg, uint64_t mag, int e2) {
  if (mag == 0) return 0.0;
  const int L = 64 - __clzll(static_cast<long long>(mag));
  const int E = e2 + L - 1;  // exponent of the leading bit
  uint64_t bits = (E >= -1022) ? ((static_cast<uint64_t>(E + 1023) << 52) | ((mag << (53 - L)) & ((1ull << 52) - 1)))
                               : (mag << (e2 + 1074));  // subnormal
  if (neg) bits |= 1ull << 63;
  return __longlong_as_double(static_cast<long long>(bits));
}

// x rounded to the grid 2^ex, ties to even, as fl(x + sigma) - sigma does with
// sigma = 0.75 2^53 2^ex for |x| < 2^51 2^ex: the slice integer and the exact remainder
// x - slice 2^ex, on the integer significand (no floating-point operations).  A zero x
// keeps its sign in the remainder, as x - (+0) does.
__device__ __forceinline__ void rn_to_grid(double x, int ex, int& slice, double& rem) {
  const uint64_t b = static_cast<uint64_t>(__double_as_longlong(x));
  const int ef = static_cast<int>((b >> 52) & 0x7FF);
  uint64_t mag = (b & 0x000FFFFFFFFFFFFFull) | (ef ? (1ull << 52) : 0ull);
  if (mag == 0) {
    slice = 0;
    rem = x;
    return;
  }
  const int e2 = (ef ? ef : 1) - 1075;
  bool neg = (b >> 63) != 0;
  const int sh = ex - e2;
  uint64_t qq = 0;
  const bool sneg = neg;
  if (sh <= 0) {
    qq = (-sh < 64) ? (mag << (-sh)) : 0ull;
    mag = 0;
  } else if (sh < 64) {
    qq = mag >> sh;
    const uint64_t r = mag & ((1ull << sh) - 1), half = 1ull << (sh - 1);
    if (r > half || (r == half && (qq & 1ull))) ++qq;  // round half to even
    const uint64_t sub = qq << sh;
    if (sub > mag) {  // rounded up: the remainder changes sign
      mag = sub - mag;
      neg = !neg;
    } else {
      mag -= sub;
    }
  }
  slice = sneg ? -static_cast<int>(qq) : static_cast<int>(qq);
  rem = compose_double(neg, mag, e2);
}

template <bool kRowsContiguous>
__global__ void __launch_bounds__(kThreads) rn_split_pass_kernel(int rows, int K, const double* Rin,
                                                                 long long rs_in, long long ks_in, double* Rout,
                                                                 long long rs_out, long long ks_out,
                                                                 const int32_t* __restrict__ E, int shift, int beta,
                                                                 uint16_t* __restrict__ plane, int kp,
                                                                 int32_t* __restrict__ ex_out,
                                                                 int32_t* __restrict__ E_next) {
  __shared__ int8_t tile[kTile][kTile + 4];  // [kk][r] slice integers
  const int tid = threadIdx.x;
  const int k0 = blockIdx.x * kTile;
  const int r0 = blockIdx.y * kTile;
  int local_max = OZ_EXP_EMPTY;
#pragma unroll 4
  for (int it = 0; it < (kTile * kTile) / kThreads; ++it) {
    int r, kk;
    if (kRowsContiguous) {
      r = tid & 63;
      kk = (tid >> 6) + 4 * it;
    } else {
      kk = tid & 63;
      r = (tid >> 6) + 4 * it;
    }
    const int gr = r0 + r, gk = k0 + kk;
    int sl = 0;
    int code = OZ_EXP_EMPTY;
    if (gr < rows && gk < K) {
      const double x = Rin[gr * rs_in + gk * ks_in];
      const int Er = __ldg(E + gr);
      double rem = x;
      if (Er != OZ_EXP_EMPTY) rn_to_grid(x, Er - shift + 1 - beta, sl, rem);  // x rounded to the grid 2^ex
      if (Rout) Rout[gr * rs_out + gk * ks_out] = rem;
      code = ceil_log2_code(rem);
    }
    tile[kk][r] = static_cast<int8_t>(sl);
    if (E_next) {
      if (kRowsContiguous) {
        local_max = max(local_max, code);  // same row for all iterations
      } else {
        int wmax = __reduce_max_sync(0xFFFFFFFFu, code);  // a warp covers one row
        if ((tid & 31) == 0 && wmax != OZ_EXP_EMPTY && gr < rows) atomicMax(&E_next[gr], wmax);
      }
    }
  }
  if (E_next && kRowsContiguous && local_max != OZ_EXP_EMPTY && r0 + (tid & 63) < rows)
    atomicMax(&E_next[r0 + (tid & 63)], local_max);
  if (blockIdx.x == 0 && tid < kTile && r0 + tid < rows) {
    const int Er = E[r0 + tid];
    ex_out[r0 + tid] = (Er == OZ_EXP_EMPTY) ? 0 : Er - shift + 1 - beta;
  }
  __syncthreads();
  // bf16 plane rows, 8 consecutive k per thread (16-byte stores)
#pragma unroll 1
  for (int it = 0; it < (kTile * kTile / 8) / kThreads; ++it) {
    const int item = tid + kThreads * it;
    const int g = item & 7, r = item >> 3;
    uint32_t w[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const float lo = __int_as_float(0x4B000080 + tile[g * 8 + 2 * x][r]) - 8388736.0f;
      const float hi = __int_as_float(0x4B000080 + tile[g * 8 + 2 * x + 1][r]) - 8388736.0f;
      w[x] = __byte_perm(__float_as_uint(lo), __float_as_uint(hi), 0x7632);
    }
    *reinterpret_cast<uint4*>(plane + static_cast<long long>(r0 + r) * kp + k0 + g * 8) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Bits [lo, lo + beta) of N = mant 2^sh (mant < 2^53; bits below 2^0 of N are dropped,
// i.e. N is the truncation), as a non-negative field.
__device__ __forceinline__ int bit_field(uint64_t mant, int sh, int lo, int beta) {
  const int d = lo - sh;  // bit d of mant is bit lo of N
  uint64_t v = 0;
  if (d >= 0 && d < 64)
    v = mant >> d;
  else if (d < 0 && d > -64)
    v = mant << (-d);
  return static_cast<int>(v & ((1ull << beta) - 1));
}

// EF split ([Ozaki notes], SplitInt): with e the row's floor(log2 max |x|), N =
// trunc(|x| 2^(s beta - e - 1)) < 2^(s beta) and slice p (1-based) is the beta-bit field
// of N at bit (s - p) beta, with the sign of x; its scale is 2^(e + 1 - p beta).  Every
// slice is a bit field of x, so one pass writes all s planes (64 x 64 tiles through shared
// memory, 16-byte stores of 8 consecutive k per plane row).  exps[p][row] receives
// e + 1 - (p + 1) beta (0 for zero rows).
template <bool kRowsContiguous>
__global__ void __launch_bounds__(kThreads) bitmask_split_kernel(int rows, int K, const double* __restrict__ X,
                                                                 long long rs, long long ks,
                                                                 const int32_t* __restrict__ E, int ns, int beta,
                                                                 uint16_t* __restrict__ planes, int rows_padded,
                                                                 int kp, int32_t* __restrict__ exps) {
  __shared__ uint64_t tile[kTile][kTile + 1];  // [kk][r] bits of x
  const int tid = threadIdx.x;
  const int k0 = blockIdx.x * kTile;
  const int r0 = blockIdx.y * kTile;
#pragma unroll 4
  for (int it = 0; it < (kTile * kTile) / kThreads; ++it) {
    int r, kk;
    if (kRowsContiguous) {
      r = tid & 63;
      kk = (tid >> 6) + 4 * it;
    } else {
      kk = tid & 63;
      r = (tid >> 6) + 4 * it;
    }
    const int gr = r0 + r, gk = k0 + kk;
    tile[kk][r] = (gr < rows && gk < K) ? static_cast<uint64_t>(__double_as_longlong(X[gr * rs + gk * ks])) : 0ull;
  }
  if (blockIdx.x == 0 && tid < kTile && r0 + tid < rows) {
    const int e = E[r0 + tid];
    const bool zero = (e == OZ_EXP_EMPTY || e == OZ_EXP_NONFINITE);
    for (int p = 0; p < ns; ++p) exps[static_cast<long long>(p) * rows + r0 + tid] = zero ? 0 : e + 1 - (p + 1) * beta;
  }
  __syncthreads();
  const long long plane_elems = static_cast<long long>(rows_padded) * kp;
#pragma unroll 1
  for (int it = 0; it < (kTile * kTile / 8) / kThreads; ++it) {
    const int item = tid + kThreads * it;
    const int g = item & 7, r = item >> 3;
    const int e = (r0 + r < rows) ? E[r0 + r] : OZ_EXP_EMPTY;
    const bool zero = (e == OZ_EXP_EMPTY || e == OZ_EXP_NONFINITE);
    uint64_t mant[8];
    int sh[8];
    bool neg[8];
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      const uint64_t b = tile[g * 8 + x][r];
      const int ef = static_cast<int>((b >> 52) & 0x7FF);
      const bool ok = !zero && ef != 0x7FF && (b & 0x7FFFFFFFFFFFFFFFull) != 0;
      mant[x] = ok ? ((b & 0x000FFFFFFFFFFFFFull) | (ef ? (1ull << 52) : 0ull)) : 0ull;
      const int e2 = (ef ? ef : 1) - 1075;  // |x| = mant 2^e2
      sh[x] = e2 + ns * beta - e - 1;
      neg[x] = (b >> 63) != 0;
    }
    uint16_t* dst = planes + static_cast<long long>(r0 + r) * kp + k0 + g * 8;
#pragma unroll 1
    for (int p = 0; p < ns; ++p) {
      const int lo = (ns - 1 - p) * beta;
      uint32_t w[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        int v0 = bit_field(mant[2 * x], sh[2 * x], lo, beta);
        int v1 = bit_field(mant[2 * x + 1], sh[2 * x + 1], lo, beta);
        v0 = neg[2 * x] ? -v0 : v0;
        v1 = neg[2 * x + 1] ? -v1 : v1;
        const float f0 = __int_as_float(0x4B000080 + v0) - 8388736.0f;  // exact: |v| < 2^7
        const float f1 = __int_as_float(0x4B000080 + v1) - 8388736.0f;
        w[x] = __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x7632);
      }
      *reinterpret_cast<uint4*>(dst + p * plane_elems) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// Hybrid split in one pass ([Ozaki notes], Hybrid split): the grids mu''_i 2^(-beta (p-1))
// are fixed by the input's row maximum (E = ceil(log2 max |x|), grid exponent E + 1 - beta p),
// so every slice of an element follows from the element alone.  fl(r + sigma) - sigma with
// sigma = 0.75 2^53 grid is round-half-to-even of r / grid, so it is done here exactly on the
// integers: x = M 2^e2 (|M| < 2^53); slice p is q = RNE(M / 2^(ex - e2)) and M -= q 2^(ex - e2),
// the same slices and residuals the double operations produce (every grid a normal number).
template <bool kRowsContiguous>
__global__ void __launch_bounds__(kThreads) hybrid_split_kernel(int rows, int K, const double* __restrict__ X,
                                                                long long rs, long long ks,
                                                                const int32_t* __restrict__ E, int ns, int beta,
                                                                uint16_t* __restrict__ planes, int rows_padded,
                                                                int kp, int32_t* __restrict__ exps) {
  __shared__ uint64_t tile[kTile][kTile + 1];  // [kk][r] bits of x
  const int tid = threadIdx.x;
  const int k0 = blockIdx.x * kTile;
  const int r0 = blockIdx.y * kTile;
#pragma unroll 4
  for (int it = 0; it < (kTile * kTile) / kThreads; ++it) {
    int r, kk;
    if (kRowsContiguous) {
      r = tid & 63;
      kk = (tid >> 6) + 4 * it;
    } else {
      kk = tid & 63;
      r = (tid >> 6) + 4 * it;
    }
    const int gr = r0 + r, gk = k0 + kk;
    tile[kk][r] = (gr < rows && gk < K) ? static_cast<uint64_t>(__double_as_longlong(X[gr * rs + gk * ks])) : 0ull;
  }
  if (blockIdx.x == 0 && tid < kTile && r0 + tid < rows) {
    const int e = E[r0 + tid];
    const bool zero = (e == OZ_EXP_EMPTY || e == OZ_EXP_NONFINITE);
    for (int p = 0; p < ns; ++p) exps[static_cast<long long>(p) * rows + r0 + tid] = zero ? 0 : e + 1 - (p + 1) * beta;
  }
  __syncthreads();
  const long long plane_elems = static_cast<long long>(rows_padded) * kp;
#pragma unroll 1
  for (int it = 0; it < (kTile * kTile / 8) / kThreads; ++it) {
    const int item = tid + kThreads * it;
    const int g = item & 7, r = item >> 3;
    const int e = (r0 + r < rows) ? E[r0 + r] : OZ_EXP_EMPTY;
    const bool zero = (e == OZ_EXP_EMPTY || e == OZ_EXP_NONFINITE);
    uint64_t mag[8];  // |residual| / 2^e2
    int e2[8];
    bool neg[8];
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      const uint64_t b = tile[g * 8 + x][r];
      const int ef = static_cast<int>((b >> 52) & 0x7FF);
      const bool ok = !zero && ef != 0x7FF && (b & 0x7FFFFFFFFFFFFFFFull) != 0;
      mag[x] = ok ? ((b & 0x000FFFFFFFFFFFFFull) | (ef ? (1ull << 52) : 0ull)) : 0ull;
      e2[x] = (ef ? ef : 1) - 1075;
      neg[x] = (b >> 63) != 0;
    }
    uint16_t* dst = planes + static_cast<long long>(r0 + r) * kp + k0 + g * 8;
#pragma unroll 1
    for (int p = 0; p < ns; ++p) {
      const int ex = e + 1 - (p + 1) * beta;  // grid exponent of slice p
      uint32_t w[4];
#pragma unroll
      for (int x2 = 0; x2 < 4; ++x2) {
        int v[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int x = 2 * x2 + h;
          // residual r = (-1)^neg mag 2^e2; slice = sign(r) RNE(mag / 2^sh); r -= slice 2^ex
          const int sh = ex - e2[x];
          if (sh <= 0) {  // the grid is as fine as the element's last bit: the rest is the slice
            const uint64_t qq = (-sh < 64) ? (mag[x] << (-sh)) : 0ull;
            v[h] = neg[x] ? -static_cast<int>(qq) : static_cast<int>(qq);
            mag[x] = 0;
          } else if (sh >= 64) {
            v[h] = 0;
          } else {
            const uint64_t a = mag[x];
            uint64_t qq = a >> sh;
            const uint64_t rem = a & ((1ull << sh) - 1), half = 1ull << (sh - 1);
            if (rem > half || (rem == half && (qq & 1ull))) ++qq;  // round half to even
            v[h] = neg[x] ? -static_cast<int>(qq) : static_cast<int>(qq);
            const uint64_t sub = qq << sh;
            if (sub > a) {  // rounded up: the residual changes sign
              mag[x] = sub - a;
              neg[x] = !neg[x];
            } else {
              mag[x] = a - sub;
            }
          }
        }
        const float f0 = __int_as_float(0x4B000080 + v[0]) - 8388736.0f;  // exact: |v| <= 2^(beta-1)
        const float f1 = __int_as_float(0x4B000080 + v[1]) - 8388736.0f;
        w[x2] = __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x7632);
      }
      *reinterpret_cast<uint4*>(dst + p * plane_elems) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// v 2^e as a double, equal to ldexp(double(v), e): for a normal result the bits are built
// with integer operations (|v| < 2^32 fits the 53-bit significand exactly); results in the
// subnormal or overflow range take ldexp itself.  Keeps the FP64 units for the additions.
__device__ __forceinline__ double scaled_int(int v, int e) {
  if (v == 0) return 0.0;
  const uint32_t a = v < 0 ? 0u - static_cast<uint32_t>(v) : static_cast<uint32_t>(v);
  const int L = 32 - __clz(static_cast<int>(a));  // a in [2^(L-1), 2^L)
  const int E = L - 1 + e;                        // exponent of the leading bit
  if (E < -1022 || E > 1023) return ldexp(static_cast<double>(v), e);
  const uint64_t frac = (static_cast<uint64_t>(a) << (53 - L)) & ((1ull << 52) - 1);
  const uint64_t bits = (static_cast<uint64_t>(E + 1023) << 52) | frac | (v < 0 ? (1ull << 63) : 0ull);
  return __longlong_as_double(static_cast<long long>(bits));
}

// C_ij = sum, in order, over the terms -- single pair products (RN), or batches of the
// pair products of one group summed in INT32 (EF, Hybrid) -- of ldexp(term, exA[ip][i] +
// exB[jp][j]), (ip, jp) the term's (first) pair: one FP64 addition per term.
__global__ void __launch_bounds__(256) ozaki1_accumulate_kernel(int m, int n, int mp, int np, int nterms,
                                                                const GemmConsts c,
                                                                const int32_t* __restrict__ prod,
                                                                const int32_t* __restrict__ exA,
                                                                const int32_t* __restrict__ exB,
                                                                double* __restrict__ C, long long ldc) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= m) return;
  const long long plane = static_cast<long long>(np) * mp;
  for (int j = blockIdx.y; j < n; j += gridDim.y) {
    double acc = 0.0;
    const int32_t* p = prod + static_cast<long long>(j) * mp + i;
#pragma unroll 4
    for (int q = 0; q < nterms; ++q) {
      const int first = c.grouped ? c.prod_first[q] : q;
      const int last = c.grouped ? c.prod_first[q + 1] : q + 1;
      int v = 0;  // a batch's INT32 sum is exact (at most r products)
      for (int t = first; t < last; ++t) v += __ldg(p + t * plane);
      const int e = __ldg(exA + c.a_plane[first] * m + i) + __ldg(exB + c.b_plane[first] * n + j);
      acc = __dadd_rn(acc, scaled_int(v, e));
    }
    C[i + j * ldc] = acc;
  }
}

}  // namespace oz

using namespace oz;

namespace {

int beta_for(long long k) {
  // largest b with k * 4^b <= 2^31, capped at 7 (= min(7, floor((31 - log2 k) / 2)))
  if (k < 1) return -1;
  int b = 0;
  while (b < 7 && (static_cast<unsigned long long>(k) << (2 * (b + 1))) <= (1ull << 31)) ++b;
  if ((static_cast<unsigned long long>(k)) > (1ull << 31)) return -1;
  return b;
}

bool valid_variant(int v) { return v == OZ_OZAKI1_RN || v == OZ_OZAKI1_EF || v == OZ_OZAKI1_HYBRID; }

// r = max(1, 2^(31 - 2 beta - ceil(log2 k))): products whose INT32 sum stays exact.
int group_r(long long k, int beta) {
  int c = 0;
  while ((1ll << c) < k) ++c;  // ceil(log2 k)
  const int e = 31 - 2 * beta - c;
  return e > 0 ? (1 << e) : 1;
}

// The pair products the slice GEMM computes, in accumulation order: RN = i outer, j inner
// over the triangle; EF / Hybrid = group g = i + j ascending, i ascending inside, with the
// batches of at most r consecutive pairs of one group in prod_first (grouped = 1, read by
// the accumulation only).
GemmConsts product_consts(int s, int beta, int variant, long long k) {
  GemmConsts g;
  std::memset(&g, 0, sizeof(g));
  int q = 0;
  if (variant == OZ_OZAKI1_RN) {
    for (int i = 0; i < s; ++i)
      for (int j = 0; j + i < s; ++j) {  // (i+1) + (j+1) <= s + 1
        g.a_plane[q] = static_cast<uint8_t>(i);
        g.b_plane[q] = static_cast<uint8_t>(j);
        ++q;
      }
  } else {
    const int r = group_r(k, beta);
    int t = 0;
    for (int grp = 2; grp <= s + 1; ++grp) {
      for (int i = 1; i <= grp - 1; ++i) {
        if ((i - 1) % r == 0) g.prod_first[t++] = static_cast<uint8_t>(q);
        g.a_plane[q] = static_cast<uint8_t>(i - 1);
        g.b_plane[q] = static_cast<uint8_t>(grp - i - 1);
        ++q;
      }
    }
    g.prod_first[t] = static_cast<uint8_t>(q);
    g.grouped = t;  // the number of batches (nonzero)
  }
  g.s = q;
  // |slice| <= 2^(beta - 1) (RN, Hybrid) or < 2^beta (EF): 2^(26 - 2 beta) or 2^(24 - 2 beta)
  // products per chunk keep the FP32 sums below 2^24, exact
  const long long chunk_k = 1ll << ((variant == OZ_OZAKI1_EF ? 24 : 26) - 2 * beta);
  g.kb_per_chunk = static_cast<int>(chunk_k / 64 > 0 ? chunk_k / 64 : 1);
  g.kb_per_block = g.kb_per_chunk * ((1 << 24) / g.kb_per_chunk);  // whole k range per unit
  return g;
}

// Terms of the FP64 accumulation: pairs (RN) or batches (EF, Hybrid).
int accumulation_terms(const GemmConsts& g) { return g.grouped ? g.grouped : g.s; }

struct Layout1 {
  int mp, np, kp, nprod;
  size_t off_RA, off_RB, off_EA, off_EB, scratch_total;  // scratch of the split step
  size_t off_planesA, off_planesB, off_exA, off_exB, off_prod, off_scratch, total;
};

size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

Layout1 layout1(int m, int n, int k, int s, int variant) {
  Layout1 L;
  L.mp = static_cast<int>(roundup(m, kPadM));
  L.np = static_cast<int>(roundup(n, kPadN));
  L.kp = static_cast<int>(roundup(k, kPadK));
  L.nprod = s * (s + 1) / 2;  // one INT32 plane per pair product
  size_t off = 0;
  L.off_RA = off;  // residuals (RN only: the EF and Hybrid splits take one pass)
  if (variant == OZ_OZAKI1_RN) off = a256(off + 8ull * m * k);
  L.off_RB = off;
  if (variant == OZ_OZAKI1_RN) off = a256(off + 8ull * k * n);
  L.off_EA = off;  // two row-maximum arrays per operand (current, next)
  off = a256(off + 8ull * m);
  L.off_EB = off;
  off = a256(off + 8ull * n);
  L.scratch_total = off;
  off = 0;
  L.off_planesA = off;
  off = a256(off + 2ull * s * L.mp * L.kp);
  L.off_planesB = off;
  off = a256(off + 2ull * s * L.np * L.kp);
  L.off_exA = off;
  off = a256(off + 4ull * s * m);
  L.off_exB = off;
  off = a256(off + 4ull * s * n);
  L.off_prod = off;
  off = a256(off + 4ull * L.nprod * L.np * L.mp);
  L.off_scratch = off;
  off = a256(off + L.scratch_total);
  L.total = off;
  return L;
}

cudaError_t launch_pass(bool rows_contig, int rows, int k, const double* Rin, long long rs_in, long long ks_in,
                        double* Rout, long long rs_out, long long ks_out, const int32_t* E, int shift, int beta,
                        uint16_t* plane, int rows_padded, int kp, int32_t* ex_out, int32_t* E_next,
                        cudaStream_t st) {
  dim3 grid(kp / kTile, rows_padded / kTile);
  if (rows_contig)
    rn_split_pass_kernel<true><<<grid, kThreads, 0, st>>>(rows, k, Rin, rs_in, ks_in, Rout, rs_out, ks_out, E, shift,
                                                          beta, plane, kp, ex_out, E_next);
  else
    rn_split_pass_kernel<false><<<grid, kThreads, 0, st>>>(rows, k, Rin, rs_in, ks_in, Rout, rs_out, ks_out, E,
                                                           shift, beta, plane, kp, ex_out, E_next);
  return cudaGetLastError();
}

cudaError_t launch_hybrid(bool rows_contig, int rows, int k, const double* X, long long rs, long long ks,
                          const int32_t* E, int s, int beta, uint16_t* planes, int rows_padded, int kp,
                          int32_t* exps, cudaStream_t st) {
  dim3 grid(kp / kTile, rows_padded / kTile);
  if (rows_contig)
    hybrid_split_kernel<true><<<grid, kThreads, 0, st>>>(rows, k, X, rs, ks, E, s, beta, planes, rows_padded, kp,
                                                         exps);
  else
    hybrid_split_kernel<false><<<grid, kThreads, 0, st>>>(rows, k, X, rs, ks, E, s, beta, planes, rows_padded, kp,
                                                          exps);
  return cudaGetLastError();
}

cudaError_t launch_bitmask(bool rows_contig, int rows, int k, const double* X, long long rs, long long ks,
                           const int32_t* E, int s, int beta, uint16_t* planes, int rows_padded, int kp,
                           int32_t* exps, cudaStream_t st) {
  dim3 grid(kp / kTile, rows_padded / kTile);
  if (rows_contig)
    bitmask_split_kernel<true><<<grid, kThreads, 0, st>>>(rows, k, X, rs, ks, E, s, beta, planes, rows_padded, kp,
                                                          exps);
  else
    bitmask_split_kernel<false><<<grid, kThreads, 0, st>>>(rows, k, X, rs, ks, E, s, beta, planes, rows_padded, kp,
                                                           exps);
  return cudaGetLastError();
}

}  // namespace

extern "C" {

int ozaki1_beta(long long k_inner, int* beta_out) {
  if (!beta_out || k_inner < 1) return OZ_EINVAL;
  const int b = beta_for(k_inner);
  if (b < 1) return OZ_ERANGE;
  *beta_out = b;
  return OZ_OK;
}

int ozaki1_group_r(long long k_inner, int* r_out) {
  int beta;
  const int rc = ozaki1_beta(k_inner, &beta);
  if (rc) return rc;
  if (!r_out) return OZ_EINVAL;
  *r_out = group_r(k_inner, beta);
  return OZ_OK;
}

int ozaki1_num_batches(int num_slices, long long k_inner, int variant, int* count_out) {
  if (!count_out || num_slices < 1 || num_slices > OZ_MAX_SLICES || !valid_variant(variant)) return OZ_EINVAL;
  int beta;
  const int rc = ozaki1_beta(k_inner, &beta);
  if (rc) return rc;
  *count_out = accumulation_terms(product_consts(num_slices, beta, variant, k_inner));
  return OZ_OK;
}

size_t ozaki1_split_scratch_bytes_ex(int m, int n, int k, int variant) {
  if (m < 0 || n < 0 || k < 0 || !valid_variant(variant)) return 0;
  return layout1(m, n, k, 1, variant).scratch_total;
}

size_t ozaki1_split_scratch_bytes(int m, int n, int k) {
  return ozaki1_split_scratch_bytes_ex(m, n, k, OZ_OZAKI1_RN);
}

size_t ozaki1_workspace_bytes_ex(int m, int n, int k, int num_slices, int variant) {
  if (m < 0 || n < 0 || k < 0 || num_slices < 1 || num_slices > OZ_MAX_SLICES || !valid_variant(variant)) return 0;
  if (k > 0 && beta_for(k) < 1) return 0;
  return layout1(m, n, k, num_slices, variant).total;
}

size_t ozaki1_workspace_bytes(int m, int n, int k, int num_slices) {
  return ozaki1_workspace_bytes_ex(m, n, k, num_slices, OZ_OZAKI1_RN);
}

int ozaki1_split_ex(int m, int n, int k, const double* A, int lda, const double* B, int ldb, int num_slices,
                    int variant, uint16_t* A_planes, uint16_t* B_planes, int32_t* A_exps, int32_t* B_exps,
                    void* scratch, size_t scratch_bytes, cudaStream_t stream) {
  if (m < 0 || n < 0 || k < 1 || num_slices < 1 || num_slices > OZ_MAX_SLICES || !valid_variant(variant))
    return OZ_EINVAL;
  if ((A && (lda < (m > 1 ? m : 1) || !A_planes || !A_exps)) || (B && (ldb < (k > 1 ? k : 1) || !B_planes || !B_exps)))
    return OZ_EINVAL;
  int beta;
  int rc = ozaki1_beta(k, &beta);
  if (rc) return rc;
  const Layout1 L = layout1(m, n, k, num_slices, variant);
  if (!scratch || scratch_bytes < L.scratch_total || (reinterpret_cast<uintptr_t>(scratch) & 255)) return OZ_ENOMEM;
  uint8_t* ws = static_cast<uint8_t*>(scratch);
  double* RA = reinterpret_cast<double*>(ws + L.off_RA);
  double* RB = reinterpret_cast<double*>(ws + L.off_RB);
  int32_t* EA[2] = {reinterpret_cast<int32_t*>(ws + L.off_EA), reinterpret_cast<int32_t*>(ws + L.off_EA) + m};
  int32_t* EB[2] = {reinterpret_cast<int32_t*>(ws + L.off_EB), reinterpret_cast<int32_t*>(ws + L.off_EB) + n};
  if (variant == OZ_OZAKI1_EF) {
    // all s bit fields in one pass, from each row's floor(log2 max |x|)
    if (launch_floor_exponents(m, n, k, A, lda, B, ldb, EA[0], EB[0], stream) != cudaSuccess) return OZ_ECUDA;
    if (A && m > 0 &&
        launch_bitmask(true, m, k, A, 1, lda, EA[0], num_slices, beta, A_planes, L.mp, L.kp, A_exps, stream) !=
            cudaSuccess)
      return OZ_ECUDA;
    if (B && n > 0 &&
        launch_bitmask(false, n, k, B, ldb, 1, EB[0], num_slices, beta, B_planes, L.np, L.kp, B_exps, stream) !=
            cudaSuccess)
      return OZ_ECUDA;
    return OZ_OK;
  }
  if (launch_exponents(m, n, k, A, lda, B, ldb, EA[0], EB[0], stream) != cudaSuccess) return OZ_ECUDA;
  if (variant == OZ_OZAKI1_HYBRID) {
    // fixed grids from the input's row maxima: all s slices in one pass
    if (A && m > 0 &&
        launch_hybrid(true, m, k, A, 1, lda, EA[0], num_slices, beta, A_planes, L.mp, L.kp, A_exps, stream) !=
            cudaSuccess)
      return OZ_ECUDA;
    if (B && n > 0 &&
        launch_hybrid(false, n, k, B, ldb, 1, EB[0], num_slices, beta, B_planes, L.np, L.kp, B_exps, stream) !=
            cudaSuccess)
      return OZ_ECUDA;
    return OZ_OK;
  }
  // RN: one rounding pass per slice, each slice's grid from the current residual's row maximum
  const bool hybrid = false;
  for (int p = 0; p < num_slices; ++p) {
    const bool last = (p == num_slices - 1);
    const int cur = hybrid ? 0 : (p & 1), nxt = cur ^ 1;
    const int shift = hybrid ? beta * p : 0;
    const bool want_next = !last && !hybrid;
    if (A && m > 0) {
      if (want_next && cudaMemsetAsync(EA[nxt], 0x80, 4ull * m, stream) != cudaSuccess) return OZ_ECUDA;
      const double* Rin = p == 0 ? A : RA;
      const long long ks_in = p == 0 ? lda : m;
      if (launch_pass(true, m, k, Rin, 1, ks_in, last ? nullptr : RA, 1, m, EA[cur], shift, beta,
                      A_planes + static_cast<long long>(p) * L.mp * L.kp, L.mp, L.kp, A_exps + static_cast<long long>(p) * m,
                      want_next ? EA[nxt] : nullptr, stream) != cudaSuccess)
        return OZ_ECUDA;
    }
    if (B && n > 0) {
      if (want_next && cudaMemsetAsync(EB[nxt], 0x80, 4ull * n, stream) != cudaSuccess) return OZ_ECUDA;
      const double* Rin = p == 0 ? B : RB;
      const long long rs_in = p == 0 ? ldb : k;
      if (launch_pass(false, n, k, Rin, rs_in, 1, last ? nullptr : RB, k, 1, EB[cur], shift, beta,
                      B_planes + static_cast<long long>(p) * L.np * L.kp, L.np, L.kp, B_exps + static_cast<long long>(p) * n,
                      want_next ? EB[nxt] : nullptr, stream) != cudaSuccess)
        return OZ_ECUDA;
    }
  }
  return OZ_OK;
}

int ozaki1_split(int m, int n, int k, const double* A, int lda, const double* B, int ldb, int num_slices,
                 uint16_t* A_planes, uint16_t* B_planes, int32_t* A_exps, int32_t* B_exps, void* scratch,
                 size_t scratch_bytes, cudaStream_t stream) {
  return ozaki1_split_ex(m, n, k, A, lda, B, ldb, num_slices, OZ_OZAKI1_RN, A_planes, B_planes, A_exps, B_exps,
                         scratch, scratch_bytes, stream);
}

int ozaki1_slice_gemm_ex(int m, int n, int k, int num_slices, int variant, const uint16_t* A_planes,
                         const uint16_t* B_planes, int32_t* products, cudaStream_t stream) {
  if (m < 0 || n < 0 || k < 1 || num_slices < 1 || num_slices > OZ_MAX_SLICES || !valid_variant(variant) ||
      !A_planes || !B_planes || !products)
    return OZ_EINVAL;
  if (m == 0 || n == 0) return OZ_OK;
  int beta;
  const int rc = ozaki1_beta(k, &beta);
  if (rc) return rc;
  const Layout1 L = layout1(m, n, k, num_slices, variant);
  return launch_slice_gemm(L.mp, L.np, L.kp, num_slices, num_slices, product_consts(num_slices, beta, variant, k),
                           A_planes, B_planes, products, stream);
}

int ozaki1_slice_gemm(int m, int n, int k, int num_slices, const uint16_t* A_planes, const uint16_t* B_planes,
                      int32_t* products, cudaStream_t stream) {
  return ozaki1_slice_gemm_ex(m, n, k, num_slices, OZ_OZAKI1_RN, A_planes, B_planes, products, stream);
}

int ozaki1_accumulate_ex(int m, int n, int k, int num_slices, int variant, const int32_t* products,
                         const int32_t* A_exps, const int32_t* B_exps, double* C, int ldc, cudaStream_t stream) {
  if (m < 0 || n < 0 || k < 1 || num_slices < 1 || num_slices > OZ_MAX_SLICES || !valid_variant(variant) ||
      !products || !A_exps || !B_exps || !C || ldc < (m > 1 ? m : 1))
    return OZ_EINVAL;
  if (m == 0 || n == 0) return OZ_OK;
  int beta;
  const int rc = ozaki1_beta(k, &beta);
  if (rc) return rc;
  const Layout1 L = layout1(m, n, k, num_slices, variant);
  const GemmConsts g = product_consts(num_slices, beta, variant, k);
  dim3 grid((m + 255) / 256, n < 65535 ? n : 65535);
  ozaki1_accumulate_kernel<<<grid, 256, 0, stream>>>(m, n, L.mp, L.np, accumulation_terms(g), g, products, A_exps,
                                                      B_exps, C, ldc);
  return cudaGetLastError() == cudaSuccess ? OZ_OK : OZ_ECUDA;
}

int ozaki1_accumulate(int m, int n, int k, int num_slices, const int32_t* products, const int32_t* A_exps,
                      const int32_t* B_exps, double* C, int ldc, cudaStream_t stream) {
  return ozaki1_accumulate_ex(m, n, k, num_slices, OZ_OZAKI1_RN, products, A_exps, B_exps, C, ldc, stream);
}

int ozaki1_dgemm_ex_ws(int m, int n, int k, const double* A, int lda, const double* B, int ldb, double* C, int ldc,
                       int num_slices, int variant, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (m < 0 || n < 0 || k < 0 || lda < (m > 1 ? m : 1) || ldb < (k > 1 ? k : 1) || ldc < (m > 1 ? m : 1))
    return OZ_EINVAL;
  if (num_slices < 1 || num_slices > OZ_MAX_SLICES || !valid_variant(variant)) return OZ_EINVAL;
  if (m == 0 || n == 0) return OZ_OK;
  if (!C) return OZ_EINVAL;
  if (k == 0) return launch_fill_zero(m, n, C, ldc, stream) == cudaSuccess ? OZ_OK : OZ_ECUDA;
  if (!A || !B) return OZ_EINVAL;
  int beta;
  int rc = ozaki1_beta(k, &beta);
  if (rc) return rc;
  const Layout1 L = layout1(m, n, k, num_slices, variant);
  if (!workspace || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255)) return OZ_ENOMEM;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint16_t* Ap = reinterpret_cast<uint16_t*>(ws + L.off_planesA);
  uint16_t* Bp = reinterpret_cast<uint16_t*>(ws + L.off_planesB);
  int32_t* exA = reinterpret_cast<int32_t*>(ws + L.off_exA);
  int32_t* exB = reinterpret_cast<int32_t*>(ws + L.off_exB);
  int32_t* prod = reinterpret_cast<int32_t*>(ws + L.off_prod);
  if ((rc = ozaki1_split_ex(m, n, k, A, lda, B, ldb, num_slices, variant, Ap, Bp, exA, exB, ws + L.off_scratch,
                            L.scratch_total, stream)))
    return rc;
  if ((rc = ozaki1_slice_gemm_ex(m, n, k, num_slices, variant, Ap, Bp, prod, stream))) return rc;
  return ozaki1_accumulate_ex(m, n, k, num_slices, variant, prod, exA, exB, C, ldc, stream);
}

int ozaki1_dgemm_ws(int m, int n, int k, const double* A, int lda, const double* B, int ldb, double* C, int ldc,
                    int num_slices, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  return ozaki1_dgemm_ex_ws(m, n, k, A, lda, B, ldb, C, ldc, num_slices, OZ_OZAKI1_RN, workspace, ws_bytes, stream);
}

int ozaki1_dgemm_ex(int m, int n, int k, const double* A, int lda, const double* B, int ldb, double* C, int ldc,
                    int num_slices, int variant, cudaStream_t stream) {
  if (m < 0 || n < 0 || k < 0 || lda < (m > 1 ? m : 1) || ldb < (k > 1 ? k : 1) || ldc < (m > 1 ? m : 1))
    return OZ_EINVAL;
  if (num_slices < 1 || num_slices > OZ_MAX_SLICES || !valid_variant(variant)) return OZ_EINVAL;
  if (m == 0 || n == 0) return OZ_OK;
  if (k == 0) return C ? (launch_fill_zero(m, n, C, ldc, stream) == cudaSuccess ? OZ_OK : OZ_ECUDA) : OZ_EINVAL;
  if (!A || !B || !C) return OZ_EINVAL;  // argument errors before any allocation
  int beta;
  int rc = ozaki1_beta(k, &beta);
  if (rc) return rc;
  const size_t bytes = ozaki1_workspace_bytes_ex(m, n, k, num_slices, variant);
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, bytes, stream) != cudaSuccess) {
    cudaGetLastError();
    return OZ_ENOMEM;
  }
  rc = ozaki1_dgemm_ex_ws(m, n, k, A, lda, B, ldb, C, ldc, num_slices, variant, ws, bytes, stream);
  const cudaError_t e = cudaFreeAsync(ws, stream);
  if (rc == OZ_OK && e != cudaSuccess) rc = OZ_ECUDA;
  return rc;
}

int ozaki1_dgemm(int m, int n, int k, const double* A, int lda, const double* B, int ldb, double* C, int ldc,
                 int num_slices, cudaStream_t stream) {
  return ozaki1_dgemm_ex(m, n, k, A, lda, B, ldb, C, ldc, num_slices, OZ_OZAKI1_RN, stream);
}

}  // extern "C"
