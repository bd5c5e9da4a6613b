// oz_crt.cu -- steps a5 + a6: CRT accumulation, range reduction, one rounding.
//
// [Ozaki II] Algorithm 1, steps 4-6.  Per output element, with residues
// c_t = C''_t in [0, m_t) and P_t = M_t y_t (< M, so P_t / M = y_t / m_t):
//   Z    = sum_t c_t P_t                      exact: 16-bit limb sums (dot products), then up to six words
//   Q    = round(Z / M) or one less            from the top limbs of Z in FP32
//   X    = Z - Q M, then one correction by M  symmetric representative, |X| < M/2
//   C    = RN(X 2^-(d_i + e_j))               one rounding, subnormals included
// The quotient estimate is biased down by 2^-8, more than its error, so it is never
// too large and at most one too small; one correction then restores the unique
// representative ([Ozaki II] section 5: the true product lies in (-M/2, M/2) because
// 2 c_max < M).  The estimate can only be one too small when its fractional part is
// within 3 * 2^-9 of the next integer, so the comparison with M/2 that detects it runs
// for those elements alone (X near +-M/2; none for typical products, whose |X| is far
// below M/2).  The remainder and the rounding are exact integer arithmetic.
#include <cmath>

#include "oz_internal.h"

namespace oz {

// Bits [pos, pos + 64) of a 6-limb little-endian integer (zero beyond the top).
__device__ __forceinline__ uint64_t window64(const uint32_t (&x)[kLimbs], int pos) {
  const int li = pos >> 5, sh = pos & 31;
  uint32_t a0 = 0, a1 = 0, a2 = 0;
#pragma unroll
  for (int l = 0; l < kLimbs; ++l) {
    a0 = (l == li) ? x[l] : a0;
    a1 = (l == li + 1) ? x[l] : a1;
    a2 = (l == li + 2) ? x[l] : a2;
  }
  const uint64_t lo = (static_cast<uint64_t>(a1) << 32) | a0;
  return sh ? ((lo >> sh) | (static_cast<uint64_t>(a2) << (64 - sh))) : lo;
}

// True if any bit below position pos (pos >= 0) is set.
__device__ __forceinline__ bool any_below(const uint32_t (&x)[kLimbs], int pos) {
  bool any = false;
#pragma unroll
  for (int l = 0; l < kLimbs; ++l) {
    const int lo = 32 * l;
    if (lo + 32 <= pos)
      any |= (x[l] != 0);
    else if (lo < pos)
      any |= (x[l] & ((1u << (pos - lo)) - 1u)) != 0;
  }
  return any;
}

// RN-even of (-1)^neg * mag * 2^-D as IEEE-754 binary64 bits (mag: 6 limbs, any above
// the caller's limb count zero).
__device__ __forceinline__ uint64_t round_scaled_bits(const uint32_t (&mag)[kLimbs], bool neg, int D) {
  int L = 0;  // bit length of mag
#pragma unroll
  for (int l = 0; l < kLimbs; ++l)
    if (mag[l] != 0) L = 32 * l + (32 - __clz(mag[l]));
  if (L == 0) return 0;  // exact zero: +0.0
  const int drop = max(L - 53, D - 1074);  // bits of mag below the result's last place
  uint64_t mant;
  if (drop <= 0) {
    const uint64_t v = (static_cast<uint64_t>(mag[1]) << 32) | mag[0];  // L <= 53 here
    mant = v << (-drop);
  } else {
    mant = window64(mag, drop);
    const bool round = (window64(mag, drop - 1) & 1u) != 0;
    const bool sticky = any_below(mag, drop - 1);
    if (round && (sticky || (mant & 1u))) ++mant;
  }
  int e = drop - D;  // value = mant * 2^e
  if (mant >= (1ull << 53)) {
    mant >>= 1;
    ++e;
  }
  uint64_t bits;
  if (mant == 0) {
    bits = 0;
  } else if (mant >= (1ull << 52)) {
    const int biased = e + 52 + 1023;
    bits = (biased >= 2047) ? 0x7FF0000000000000ull
                            : ((static_cast<uint64_t>(biased) << 52) | (mant & ((1ull << 52) - 1)));
  } else {
    bits = mant;  // subnormal: e == -1074
  }
  return bits | (neg ? 0x8000000000000000ull : 0ull);
}

// RN-even of (-1)^neg * x * 2^-D (x: NL limbs) for results that are normal numbers or
// overflow, from 64-bit words: the word holding the leading one and the word below it
// give the 64-bit window, anything lower only the sticky bit.  Returns false for results
// in the subnormal range (the general routine above handles them).
template <int NL>
__device__ __forceinline__ bool round_normal_words(const uint32_t (&x)[kLimbs], bool neg, int D, uint64_t& out) {
  constexpr int NW = (NL + 1) / 2;
  uint64_t w[NW];
#pragma unroll
  for (int i = 0; i < NW; ++i)
    w[i] = static_cast<uint64_t>(x[2 * i]) | ((2 * i + 1 < NL) ? static_cast<uint64_t>(x[2 * i + 1]) << 32 : 0ull);
  // the highest non-zero word w[h] (h = 0 if all above w[0] are zero), the word below it, and
  // whether any word further down is non-zero
  uint64_t hi = w[0], lo = 0, below = 0;
  int base = 0;
#pragma unroll
  for (int i = 1; i < NW; ++i) {
    if (w[i] != 0) {
      hi = w[i];
      lo = w[i - 1];
      base = 64 * i;
      below = 0;
#pragma unroll
      for (int b = 0; b + 1 < i; ++b) below |= w[b];
    }
  }
  bool sticky = below != 0;
  if (hi == 0) {
    out = 0;  // exact zero: +0.0
    return true;
  }
  const int lz = __clzll(static_cast<long long>(hi));
  const uint64_t win = lz ? (hi << lz) | (lo >> (64 - lz)) : hi;
  sticky = sticky || ((lz ? (lo << lz) : lo) != 0);
  const int e_unb = base + 63 - lz - D;  // exponent of the leading one in the result
  if (e_unb < -1022) return false;
  const uint64_t sgn = neg ? 0x8000000000000000ull : 0ull;
  if (e_unb > 1023) {
    out = 0x7FF0000000000000ull | sgn;
    return true;
  }
  uint64_t mant = win >> 11;
  const bool rb = (win >> 10) & 1u;
  sticky = sticky || ((win & 0x3FFu) != 0);
  if (rb && (sticky || (mant & 1u))) ++mant;  // may carry into 2^53: exponent + 1 below
  out = ((static_cast<uint64_t>(e_unb + 1022) << 52) + mant) | sgn;
  return true;
}

// One thread = 4 consecutive rows i of one column j (a 4-byte load per modulus).
// NL = 32-bit words needed for Z = sum_t c_t P_t (< 255 s M).  The sum runs on N16
// limbs of 16 bits of P_t, one 32-bit accumulator per limb, with two-way dot products
// (dp2a: two 16-bit limbs of a pair of moduli times the pair's two residue bytes, plus
// the accumulator): every term is below 255 2^16 and s of them stay below 2^32, so the
// sums are exact, at one instruction per two moduli and limb.  The residues of four
// moduli for one element come from a 4 x 4 byte transpose of the four elements' words.
// The limbs are then carried into NL words.
template <int NL, int N16>
__global__ void __launch_bounds__(256) crt_kernel(int m, int n, int mp, int np, const CrtConsts c, float inv_m_top,
                                                  const uint8_t* __restrict__ C_res,
                                                  const int32_t* __restrict__ rowexp,
                                                  const int32_t* __restrict__ colexp, double* __restrict__ C,
                                                  long long ldc) {
  static_assert(N16 >= 1 && N16 <= kHalfLimbs && N16 <= 2 * NL && kMaxModuli % 4 == 0, "CRT limb class");
  const int i0 = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i0 >= m) return;
  const long long plane = static_cast<long long>(np) * mp;
  int E[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) E[e] = (i0 + e < m) ? __ldg(rowexp + i0 + e) : OZ_EXP_EMPTY;
  for (int j = blockIdx.y; j < n; j += gridDim.y) {
    const int F = __ldg(colexp + j);
    // all residues of the 4 elements first: s independent 4-byte loads in flight
    uint32_t res[kMaxModuli];
    const uint8_t* base = C_res + static_cast<long long>(j) * mp + i0;
#pragma unroll
    for (int t = 0; t < kMaxModuli; ++t)
      res[t] = (t < c.s) ? __ldg(reinterpret_cast<const uint32_t*>(base + t * plane)) : 0u;
    double* out = C + i0 + j * ldc;
    // Z = sum_t c_t P_t for the 4 elements at once, on 16-bit limbs (carries later)
    uint32_t acc[4][N16];
#pragma unroll
    for (int e = 0; e < 4; ++e)
#pragma unroll
      for (int l = 0; l < N16; ++l) acc[e][l] = 0;
#pragma unroll
    for (int g = 0; g < kMaxModuli / 4; ++g) {
      if (4 * g >= c.s) break;
      // R[e] = residue bytes of moduli 4g .. 4g+3 for element e (res[t] holds modulus t
      // for the 4 elements)
      const uint32_t t0 = __byte_perm(res[4 * g], res[4 * g + 1], 0x5140u);
      const uint32_t t1 = __byte_perm(res[4 * g], res[4 * g + 1], 0x7362u);
      const uint32_t t2 = __byte_perm(res[4 * g + 2], res[4 * g + 3], 0x5140u);
      const uint32_t t3 = __byte_perm(res[4 * g + 2], res[4 * g + 3], 0x7362u);
      const uint32_t R[4] = {__byte_perm(t0, t2, 0x5410u), __byte_perm(t0, t2, 0x7632u),
                             __byte_perm(t1, t3, 0x5410u), __byte_perm(t1, t3, 0x7632u)};
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int l = 0; l < N16; ++l) acc[e][l] = __dp2a_lo(c.Pd[2 * g][l], R[e], acc[e][l]);
      if (4 * g + 2 < c.s) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int l = 0; l < N16; ++l) acc[e][l] = __dp2a_hi(c.Pd[2 * g + 1][l], R[e], acc[e][l]);
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (i0 + e >= m) break;
      if (E[e] == OZ_EXP_NONFINITE || F == OZ_EXP_NONFINITE) {
        out[e] = __longlong_as_double(0x7FF8000000000000ll);
        continue;
      }
      if (E[e] == OZ_EXP_EMPTY || F == OZ_EXP_EMPTY) {
        out[e] = 0.0;
        continue;
      }
      // Z into NL words: word w holds limbs 2w and 2w + 1; run < 2^29 + 2^45 + 2^32.
      uint32_t x[kLimbs];
      uint64_t run = 0;
#pragma unroll
      for (int w = 0; w < NL; ++w) {
        if (2 * w < N16) run += acc[e][2 * w];
        if (2 * w + 1 < N16) run += static_cast<uint64_t>(acc[e][2 * w + 1]) << 16;
        x[w] = static_cast<uint32_t>(run);
        run >>= 32;
      }
      // Q = floor(Z/M + 1/2 - 2^-8) from the top three limbs in FP32 (error < 2^-9):
      // round(Z/M) or one less, never more, so X = Z - Q M is the representative or
      // the representative plus M.  It is one less only if the estimate h lies within
      // 2^-9 + 2^-8 of the next integer, so below a fractional part of 1 - 2^-7 it is
      // exactly round(Z/M) and X needs no correction.
      float zs = __uint2float_rn(x[NL - 1]);
      zs = fmaf(__uint2float_rn(x[NL - 2]), 2.3283064365386963e-10f, zs);
      zs = fmaf(__uint2float_rn(x[NL - 3]), 5.421010862427522e-20f, zs);
      const float h = fmaf(zs, inv_m_top, 0.49609375f);
      const float hq = floorf(h);
      const bool near = (h - hq) >= 0.9921875f;  // exact difference: h < 2^13
      const uint32_t Q = static_cast<uint32_t>(hq);
      uint64_t qc = 0;
      uint32_t borrow = 0;
#pragma unroll
      for (int l = 0; l < NL; ++l) {
        const uint64_t qm = static_cast<uint64_t>(Q) * c.M[l] + qc;
        qc = qm >> 32;
        const uint64_t d = static_cast<uint64_t>(x[l]) - static_cast<uint32_t>(qm) - borrow;
        x[l] = static_cast<uint32_t>(d);
        borrow = static_cast<uint32_t>(d >> 63);
      }
      bool neg = (x[NL - 1] >> 31) != 0;
      {  // magnitude: X for X >= 0, two's complement negation otherwise
        const uint32_t flip = neg ? 0xFFFFFFFFu : 0u;
        uint32_t cy = neg ? 1u : 0u;
#pragma unroll
        for (int l = 0; l < NL; ++l) {
          const uint64_t v = static_cast<uint64_t>(x[l] ^ flip) + cy;
          x[l] = static_cast<uint32_t>(v);
          cy = static_cast<uint32_t>(v >> 32);
        }
      }
      if (near && !neg) {  // X > M/2 means X = representative + M, representative < 0: magnitude M - X
        bool gt = false, decided = false;
#pragma unroll
        for (int l = NL - 1; l >= 0; --l) {
          if (!decided && x[l] != c.halfM[l]) {
            gt = x[l] > c.halfM[l];
            decided = true;
          }
        }
        if (gt) {
          uint32_t b = 0;
#pragma unroll
          for (int l = 0; l < NL; ++l) {
            const uint64_t d = static_cast<uint64_t>(c.M[l]) - x[l] - b;
            x[l] = static_cast<uint32_t>(d);
            b = static_cast<uint32_t>(d >> 63);
          }
          neg = true;
        }
      }
#pragma unroll
      for (int l = NL; l < kLimbs; ++l) x[l] = 0;
      const int D = 2 * c.kA - E[e] - F;  // d_i + e_j
      uint64_t bits;
      if (!round_normal_words<NL>(x, neg, D, bits)) bits = round_scaled_bits(x, neg, D);
      out[e] = __longlong_as_double(static_cast<long long>(bits));
    }
  }
}

// Limbs needed for Z < 255 s M (host side: bit length of M plus log2(255 s)).
static int crt_limbs(const CrtConsts& c) {
  int top = kLimbs - 1;
  while (top > 0 && c.M[top] == 0) --top;
  int bits = 32 * top;
  for (uint32_t v = c.M[top]; v; v >>= 1) ++bits;
  bits += 13;  // 255 * 20 < 2^13
  return (bits + 31) / 32;
}

cudaError_t launch_crt(int m, int n, int mp, int np, const CrtConsts& c, const uint8_t* C_res,
                       const int32_t* rowexp, const int32_t* colexp, double* C, int ldc, cudaStream_t stream) {
  if (m == 0 || n == 0) return cudaSuccess;
  dim3 grid((m + 1023) / 1024, n < 1024 ? n : 1024);  // each block loops over n / 1024 columns
  const int nl = crt_limbs(c) < 3 ? 3 : crt_limbs(c);
  // 2^(32 (nl - 1)) / M: the quotient estimate reads the top limb in units of 2^(32 (nl - 1))
  double Md = 0.0;
  for (int l = kLimbs - 1; l >= 0; --l) Md = Md * 4294967296.0 + c.M[l];
  const float inv_m_top = static_cast<float>(std::ldexp(1.0, 32 * (nl - 1)) / Md);
  // (NL, N16) for each moduli count: the words of Z and the 16-bit limbs of M
#define OZ_CRT_LAUNCH(NLv, N16v) \
  crt_kernel<NLv, N16v><<<grid, 256, 0, stream>>>(m, n, mp, np, c, inv_m_top, C_res, rowexp, colexp, C, ldc)
  switch (nl * 16 + c.n16) {
    case 3 * 16 + 1: OZ_CRT_LAUNCH(3, 1); break;
    case 3 * 16 + 2: OZ_CRT_LAUNCH(3, 2); break;
    case 3 * 16 + 3: OZ_CRT_LAUNCH(3, 3); break;
    case 3 * 16 + 4: OZ_CRT_LAUNCH(3, 4); break;
    case 3 * 16 + 5: OZ_CRT_LAUNCH(3, 5); break;
    case 4 * 16 + 6: OZ_CRT_LAUNCH(4, 6); break;
    case 4 * 16 + 7: OZ_CRT_LAUNCH(4, 7); break;
    case 5 * 16 + 8: OZ_CRT_LAUNCH(5, 8); break;
    case 5 * 16 + 9: OZ_CRT_LAUNCH(5, 9); break;
    case 6 * 16 + 10: OZ_CRT_LAUNCH(6, 10); break;
    default: return cudaErrorInvalidValue;  // no class for this moduli count (cannot happen for 2..20 moduli <= 256)
  }
#undef OZ_CRT_LAUNCH
  return cudaGetLastError();
}

}  // namespace oz
