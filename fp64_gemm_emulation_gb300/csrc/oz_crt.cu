// oz_crt.cu -- steps a5 + a6: CRT accumulation, range reduction, one rounding.
//
// [Ozaki II] Algorithm 1, steps 4-6.  Per output element, with residues
// c_t = C''_t in [0, m_t) and P_t = M_t y_t (< M, so P_t / M = y_t / m_t):
//   Z    = sum_t c_t P_t                      exact: 16-bit limb sums (dot products), then up to six words
//   Q    = round(Z / M) or one less            from the top words of Z in FP32
//   X    = Z - Q M, then one correction by M  symmetric representative, |X| < M/2
//   C    = RN(X 2^-(d_i + e_j))               one rounding, subnormals included
// The quotient is rounded from Z/M - 2^-8, a bias larger than the estimate's error, so it
// is never too large and at most one too small; one correction then restores the unique
// representative ([Ozaki II] section 5: the true product lies in (-M/2, M/2) because
// 2 c_max < M).  It can only be one too small when the biased estimate lies within
// 2^-8 + 2^-10 below a half-integer, so the comparison with M/2 that detects it runs for
// those elements alone (X near +-M/2; none for typical products, whose |X| is far below
// M/2).  The remainder and the rounding are exact integer arithmetic.
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

// Multi-word arithmetic on NL little-endian 32-bit words with the carry flag (one asm
// block per operation, so that no other instruction comes between the links of a chain).

// x = a + b (mod 2^(32 NL)).
template <int NL>
__device__ __forceinline__ void add_words(uint32_t (&x)[kLimbs], const uint32_t (&a)[kLimbs],
                                          const uint32_t (&b)[kLimbs]) {
  if constexpr (NL == 3) {
    asm("add.cc.u32 %0, %3, %6;\n\t"
        "addc.cc.u32 %1, %4, %7;\n\t"
        "addc.u32 %2, %5, %8;"
        : "=r"(x[0]), "=r"(x[1]), "=r"(x[2])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(b[0]), "r"(b[1]), "r"(b[2]));
  } else if constexpr (NL == 4) {
    asm("add.cc.u32 %0, %4, %8;\n\t"
        "addc.cc.u32 %1, %5, %9;\n\t"
        "addc.cc.u32 %2, %6, %10;\n\t"
        "addc.u32 %3, %7, %11;"
        : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]), "r"(b[2]), "r"(b[3]));
  } else if constexpr (NL == 5) {
    asm("add.cc.u32 %0, %5, %10;\n\t"
        "addc.cc.u32 %1, %6, %11;\n\t"
        "addc.cc.u32 %2, %7, %12;\n\t"
        "addc.cc.u32 %3, %8, %13;\n\t"
        "addc.u32 %4, %9, %14;"
        : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(b[0]), "r"(b[1]), "r"(b[2]), "r"(b[3]), "r"(b[4]));
  } else if constexpr (NL == 6) {
    asm("add.cc.u32 %0, %6, %12;\n\t"
        "addc.cc.u32 %1, %7, %13;\n\t"
        "addc.cc.u32 %2, %8, %14;\n\t"
        "addc.cc.u32 %3, %9, %15;\n\t"
        "addc.cc.u32 %4, %10, %16;\n\t"
        "addc.u32 %5, %11, %17;"
        : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(b[0]), "r"(b[1]), "r"(b[2]), "r"(b[3]), "r"(b[4]), "r"(b[5]));
  }
}

// x = x + cy (mod 2^(32 NL)), cy in {0, 1}.
template <int NL>
__device__ __forceinline__ void inc_words(uint32_t (&x)[kLimbs], uint32_t cy) {
  if constexpr (NL == 3) {
    asm("add.cc.u32 %0, %0, %3;\n\t"
        "addc.cc.u32 %1, %1, 0;\n\t"
        "addc.u32 %2, %2, 0;"
        : "+r"(x[0]), "+r"(x[1]), "+r"(x[2])
        : "r"(cy));
  } else if constexpr (NL == 4) {
    asm("add.cc.u32 %0, %0, %4;\n\t"
        "addc.cc.u32 %1, %1, 0;\n\t"
        "addc.cc.u32 %2, %2, 0;\n\t"
        "addc.u32 %3, %3, 0;"
        : "+r"(x[0]), "+r"(x[1]), "+r"(x[2]), "+r"(x[3])
        : "r"(cy));
  } else if constexpr (NL == 5) {
    asm("add.cc.u32 %0, %0, %5;\n\t"
        "addc.cc.u32 %1, %1, 0;\n\t"
        "addc.cc.u32 %2, %2, 0;\n\t"
        "addc.cc.u32 %3, %3, 0;\n\t"
        "addc.u32 %4, %4, 0;"
        : "+r"(x[0]), "+r"(x[1]), "+r"(x[2]), "+r"(x[3]), "+r"(x[4])
        : "r"(cy));
  } else if constexpr (NL == 6) {
    asm("add.cc.u32 %0, %0, %6;\n\t"
        "addc.cc.u32 %1, %1, 0;\n\t"
        "addc.cc.u32 %2, %2, 0;\n\t"
        "addc.cc.u32 %3, %3, 0;\n\t"
        "addc.cc.u32 %4, %4, 0;\n\t"
        "addc.u32 %5, %5, 0;"
        : "+r"(x[0]), "+r"(x[1]), "+r"(x[2]), "+r"(x[3]), "+r"(x[4]), "+r"(x[5])
        : "r"(cy));
  }
}

// x = x + Q Mn (mod 2^(32 NL)): the products' low words in one carry chain, their high
// words (one word up) in a second.
template <int NL>
__device__ __forceinline__ void mad_words(uint32_t (&x)[kLimbs], uint32_t Q, const uint32_t (&Mn)[kLimbs]) {
  if constexpr (NL == 3) {
    asm("mad.lo.cc.u32 %0, %3, %4, %0;\n\t"
        "madc.lo.cc.u32 %1, %3, %5, %1;\n\t"
        "madc.lo.u32 %2, %3, %6, %2;\n\t"
        "mad.hi.cc.u32 %1, %3, %4, %1;\n\t"
        "madc.hi.u32 %2, %3, %5, %2;"
        : "+r"(x[0]), "+r"(x[1]), "+r"(x[2])
        : "r"(Q), "r"(Mn[0]), "r"(Mn[1]), "r"(Mn[2]));
  } else if constexpr (NL == 4) {
    asm("mad.lo.cc.u32 %0, %4, %5, %0;\n\t"
        "madc.lo.cc.u32 %1, %4, %6, %1;\n\t"
        "madc.lo.cc.u32 %2, %4, %7, %2;\n\t"
        "madc.lo.u32 %3, %4, %8, %3;\n\t"
        "mad.hi.cc.u32 %1, %4, %5, %1;\n\t"
        "madc.hi.cc.u32 %2, %4, %6, %2;\n\t"
        "madc.hi.u32 %3, %4, %7, %3;"
        : "+r"(x[0]), "+r"(x[1]), "+r"(x[2]), "+r"(x[3])
        : "r"(Q), "r"(Mn[0]), "r"(Mn[1]), "r"(Mn[2]), "r"(Mn[3]));
  } else if constexpr (NL == 5) {
    asm("mad.lo.cc.u32 %0, %5, %6, %0;\n\t"
        "madc.lo.cc.u32 %1, %5, %7, %1;\n\t"
        "madc.lo.cc.u32 %2, %5, %8, %2;\n\t"
        "madc.lo.cc.u32 %3, %5, %9, %3;\n\t"
        "madc.lo.u32 %4, %5, %10, %4;\n\t"
        "mad.hi.cc.u32 %1, %5, %6, %1;\n\t"
        "madc.hi.cc.u32 %2, %5, %7, %2;\n\t"
        "madc.hi.cc.u32 %3, %5, %8, %3;\n\t"
        "madc.hi.u32 %4, %5, %9, %4;"
        : "+r"(x[0]), "+r"(x[1]), "+r"(x[2]), "+r"(x[3]), "+r"(x[4])
        : "r"(Q), "r"(Mn[0]), "r"(Mn[1]), "r"(Mn[2]), "r"(Mn[3]), "r"(Mn[4]));
  } else if constexpr (NL == 6) {
    asm("mad.lo.cc.u32 %0, %6, %7, %0;\n\t"
        "madc.lo.cc.u32 %1, %6, %8, %1;\n\t"
        "madc.lo.cc.u32 %2, %6, %9, %2;\n\t"
        "madc.lo.cc.u32 %3, %6, %10, %3;\n\t"
        "madc.lo.cc.u32 %4, %6, %11, %4;\n\t"
        "madc.lo.u32 %5, %6, %12, %5;\n\t"
        "mad.hi.cc.u32 %1, %6, %7, %1;\n\t"
        "madc.hi.cc.u32 %2, %6, %8, %2;\n\t"
        "madc.hi.cc.u32 %3, %6, %9, %3;\n\t"
        "madc.hi.cc.u32 %4, %6, %10, %4;\n\t"
        "madc.hi.u32 %5, %6, %11, %5;"
        : "+r"(x[0]), "+r"(x[1]), "+r"(x[2]), "+r"(x[3]), "+r"(x[4]), "+r"(x[5])
        : "r"(Q), "r"(Mn[0]), "r"(Mn[1]), "r"(Mn[2]), "r"(Mn[3]), "r"(Mn[4]), "r"(Mn[5]));
  }
}

struct Words6 {
  uint32_t w[kLimbs];
};

// The rare results in the subnormal range, out of line so that the common path keeps its
// words in registers.
__device__ __noinline__ uint64_t round_subnormal(Words6 v, bool neg, int D) {
  return round_scaled_bits(v.w, neg, D);
}

// The CRT sum, range reduction and rounding of one element from its exact sum
// Z = x[0..NL-1] (32-bit words, little-endian): returns the bits of C_ij.  All on 32-bit
// words: the quotient estimate, X = Z - Q M (as Z + Q (2^(32 NL) - M) in two carry
// chains), the magnitude, and the rounding from a 64-bit window cut out of the three words
// from the leading one down (funnel shifts), the words below only as sticky.
template <int NL>
__device__ __forceinline__ uint64_t crt_finish(uint32_t (&x)[kLimbs], int E, int F, const CrtConsts& c,
                                               float inv_m_top) {
  if (E == OZ_EXP_NONFINITE || F == OZ_EXP_NONFINITE) return 0x7FF8000000000000ull;
  if (E == OZ_EXP_EMPTY || F == OZ_EXP_EMPTY) return 0;
  // z = Z/M - 2^-8 in FP32 from the top two words, all three when NL = 3 (error below
  // 2^-10: Z/M < 255 s < 2^13, a few roundings of relative size 2^-24 and one of 2^-13; for
  // NL >= 4, M > 2^83 and the words left out are worth less than 2^-18).  Q = round(z) is
  // round(Z/M) or one less, never more, so X = Z - Q M is the representative or the
  // representative plus M.  It is one less only if Z/M lies just above a half-integer,
  // where z lies within 2^-8 + 2^-10 below it: every such element has |z - Q| > 0.4921875,
  // and only those elements compare X with M/2.
  float zs = fmaf(__uint2float_rn(x[NL - 2]), 2.3283064365386963e-10f, __uint2float_rn(x[NL - 1]));
  if constexpr (NL == 3) zs = fmaf(__uint2float_rn(x[0]), 5.421010862427522e-20f, zs);
  const float z = fmaf(zs, inv_m_top, -0.00390625f);
  const float t = z + 8388608.0f;  // 2^23 + round(z), as -0.5 < z < 2^13
  const uint32_t Q = __float_as_uint(t) - 0x4B000000u;
  const bool near = fabsf(z - (t - 8388608.0f)) > 0.4921875f;  // exact difference
  mad_words<NL>(x, Q, c.Mneg);                                   // X = Z - Q M (mod 2^(32 NL))
  bool neg = (x[NL - 1] >> 31) != 0;
  {  // magnitude: X for X >= 0, two's complement negation otherwise
    const uint32_t flip = neg ? 0xFFFFFFFFu : 0u;
#pragma unroll
    for (int l = 0; l < NL; ++l) x[l] ^= flip;
    inc_words<NL>(x, flip & 1u);
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
        b = static_cast<uint32_t>(d >> 32) & 1u;
      }
      neg = true;
    }
  }
  const int D = 2 * c.kA - E - F;  // d_i + e_j
  // leading word a = x[hi], then b, c below it; any word further down only as sticky
  int hw = 0;
  uint32_t a = x[0], b = 0, cw = 0, below = 0;
#pragma unroll
  for (int l = 1; l < NL; ++l) {
    if (x[l] != 0) {
      hw = l;
      a = x[l];
      b = x[l - 1];
      cw = (l >= 2) ? x[l - 2] : 0u;
      below = 0;
#pragma unroll
      for (int q = 0; q + 2 < l; ++q) below |= x[q];
    }
  }
  if (a == 0) return 0;  // exact zero: +0.0
  const int lz = __clz(a);
  const uint32_t w1 = __funnelshift_l(b, a, lz);   // window bits 63..32 (leading one at bit 63)
  const uint32_t w0 = __funnelshift_l(cw, b, lz);  // window bits 31..0
  const bool sticky = ((cw << lz) | below | (w0 & 0x3FFu)) != 0;
  const int e_unb = 32 * hw + 31 - lz - D;  // exponent of the leading one in the result
  if (e_unb < -1022) {  // subnormal range: the general routine
#pragma unroll
    for (int l = NL; l < kLimbs; ++l) x[l] = 0;
    return round_subnormal(Words6{x[0], x[1], x[2], x[3], x[4], x[5]}, neg, D);
  }
  const uint32_t sgn = neg ? 0x80000000u : 0u;
  if (e_unb > 1023) return static_cast<uint64_t>(0x7FF00000u | sgn) << 32;
  uint32_t mlo = __funnelshift_r(w0, w1, 11), mhi = w1 >> 11;  // 53-bit significand
  const uint32_t inc = ((w0 >> 10) & 1u) & ((sticky ? 1u : 0u) | (mlo & 1u));
  const uint64_t m = ((static_cast<uint64_t>(mhi) << 32) | mlo) + inc;  // may carry into 2^53: exponent + 1
  const uint64_t bits = (static_cast<uint64_t>(e_unb + 1022) << 52) + m;
  return bits | (static_cast<uint64_t>(sgn) << 32);
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
__global__ void __launch_bounds__(256, 3) crt_kernel(int m, int n, int mp, int np, const CrtConsts c, float inv_m_top,
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
      // Z into NL words: word w = limb 2w + limb 2w+1 shifted up by 16 (its low half; the
      // high half of limb 2w-1 joins it) in one carry chain.  Z < 2^(32 NL), so the top
      // limb is below 2^16 and no carry leaves the top word.
      uint32_t x[kLimbs], ev[kLimbs], od[kLimbs];
#pragma unroll
      for (int w = 0; w < kLimbs; ++w) {
        const uint32_t below = (w >= 1 && 2 * w - 1 < N16) ? acc[e][w >= 1 ? 2 * w - 1 : 0] : 0u;
        const uint32_t above = (2 * w + 1 < N16) ? acc[e][2 * w + 1] : 0u;
        ev[w] = (2 * w < N16) ? acc[e][2 * w] : 0u;
        od[w] = __byte_perm(below, above, 0x5432);  // below >> 16 | (above & 0xFFFF) << 16
        x[w] = 0;
      }
      add_words<NL>(x, ev, od);
      out[e] = __longlong_as_double(static_cast<long long>(crt_finish<NL>(x, E[e], F, c, inv_m_top)));
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
  CrtConsts cc = c;  // with 2^(32 nl) - M for the quotient's subtraction
  uint32_t borrow = 0;
  for (int l = 0; l < kLimbs; ++l) {
    const uint64_t d = (l < nl) ? 0ull - static_cast<uint64_t>(c.M[l]) - borrow : 0ull;
    cc.Mneg[l] = (l < nl) ? static_cast<uint32_t>(d) : 0u;
    borrow = (l < nl) ? static_cast<uint32_t>(d >> 63) : 0u;
  }
  // (NL, N16) for each moduli count: the words of Z and the 16-bit limbs of M
#define OZ_CRT_LAUNCH(NLv, N16v) \
  crt_kernel<NLv, N16v><<<grid, 256, 0, stream>>>(m, n, mp, np, cc, inv_m_top, C_res, rowexp, colexp, C, ldc)
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
