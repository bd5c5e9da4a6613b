// oz_split.cu -- step a2: scale, truncate and take the symmetric residues.
//
// [Ozaki II] Algorithm 1, step 2 (A' = trunc(DA)) and the left half of step 3
// (A'_t = A' mod m_t, symmetric, signed 8-bit) for every modulus t, in one pass over
// the FP64 operand, without the FP64 units.  In the common case (a' < 2^52, no
// power-of-two factor) a' is cut into four 13-bit limbs held as exact FP32 values and
// each residue takes a few FP32 FMAs; otherwise a' = trunc(|a| 2^d) is kept as u * 2^p
// with u < 2^53, and a' mod m is (u mod m)(2^p mod m) mod m with u split into 16-bit
// limbs and one integer Barrett step.
//
// For a row-contiguous operand one block handles a 64 x 64 tile (rows x k): phase 1 reads
// the tile with coalesced loads along the rows and stores the FP64 patterns in shared
// memory; phase 2 reads them along k and writes 16-byte vectors of 8 bf16 residues per
// modulus, so the K-contiguous planes are written in full 128-byte rows.
#include "oz_fp.cuh"
#include "oz_internal.h"

namespace oz {

constexpr int kSplitTile = 64;
constexpr int kSplitThreads = 256;

// Packs trunc(|x| 2^(kA - E)) as sign<<63 | p<<53 | u, value u 2^p (u < 2^53).
__device__ __forceinline__ uint64_t pack_scaled(double x, int E, int kA) {
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
  const int sh = e2 + (kA - E);  // |x| 2^d = mant 2^sh
  uint64_t u;
  uint32_t p;
  if (sh >= 0) {
    u = mant;
    p = static_cast<uint32_t>(sh);
  } else {
    u = (-sh >= 64) ? 0 : (mant >> (-sh));  // truncation toward zero
    p = 0;
  }
  if (u == 0) return 0;
  return (bits & 0x8000000000000000ull) | (static_cast<uint64_t>(p) << 53) | u;
}

// y mod m for y < 2^30 and 2 <= m <= 256, with magic = ceil(2^39 / m).
__device__ __forceinline__ uint32_t mod_small(uint32_t y, uint32_t m, uint32_t magic) {
  return y - (__umulhi(y, magic) >> 7) * m;
}

// bf16 bit pattern of the symmetric residue of the packed integer modulo m.
//   r = |a'| mod m                      (16-bit limbs of u, one Barrett step)
//   w = r, or m - r for a negative a'    (the residue of a' itself, in [1, m])
//   v = w - m if w >= ceil(m/2) else w   (symmetric representative, [-(m/2), (m-1)/2])
// and bf16(v) from the float 2^23 + 128 + v (exact), minus 2^23 + 128, top 16 bits:
// no integer-to-float conversion instruction.
__device__ __forceinline__ uint32_t residue_bf16(uint32_t x0, uint32_t x1, uint32_t x2, uint32_t p, bool neg,
                                                 uint32_t m, uint32_t c16, uint32_t c32, uint32_t magic) {
  uint32_t r = mod_small(x2 * c32 + x1 * c16 + x0, m, magic);
  if (p != 0) {
    uint32_t w = 1;
    for (uint32_t i = 0; i < p && w != 0; ++i) {
      w <<= 1;
      if (w >= m) w -= m;
    }
    r = mod_small(r * w, m, magic);
  }
  const int h = static_cast<int>((m + 1) >> 1);
  int w = neg ? static_cast<int>(m - r) : static_cast<int>(r);
  if (w >= h) w -= static_cast<int>(m);
  const float f = __int_as_float(0x4B000080 + w) - 8388736.0f;  // exactly w
  return __float_as_uint(f) >> 16;
}

// Integer path with p == 0 (a' = sign * u, u up to 2^53; the FP32 limb path below takes
// u < 2^52): the symmetric residue of a' modulo m, as a float.
//   ys = sign * (x2 c32 + x1 c16 + x0) + BIG + floor(m/2)   (BIG = m 2^22)
//   q  = floor(ys / m)                                      (one Barrett step)
//   ys - q m = v + floor(m/2) with v the symmetric representative in
//   [-floor(m/2), ceil(m/2) - 1]; the float 2^23 + 128 + v is built directly from the
//   bits (the per-modulus constant absorbs floor(m/2)) and 2^23 + 128 subtracted.
// BIG is a multiple of m above |y| < (m - 1)(2^21 + 2^16) + 2^16, added whatever the sign,
// so ys > 0 and ys < m 2^22 + m 2^21.05 + m < 2^31 <= 2^39 / m keeps the quotient exact.
// sx* are the sign-applied 16-bit limbs of u; offs = BIG + floor(m/2).
__device__ __forceinline__ float residue_fast(int sx0, int sx1, int sx2, uint32_t m, uint32_t c16, uint32_t c32,
                                              uint32_t magic, uint32_t offs, uint32_t fbase) {
  const uint32_t y = static_cast<uint32_t>(sx2 * static_cast<int>(c32) + sx1 * static_cast<int>(c16) + sx0);
  const uint32_t ys = y + offs;
  const uint32_t q = __umulhi(ys, magic) >> 7;
  return __int_as_float(static_cast<int>(fbase + (ys - q * m))) - 8388736.0f;
}

// Shifted path (0 < p <= kShiftMax for some element, e.g. k_A > 53): a' = u 2^p < 2^63 as
// four 16-bit limbs, y = x3 c48 + x2 c32 + x1 c16 + x0 with |y| < 2^26, then the same single
// Barrett step as the fast path: BIG = m 2^22 exceeds |y| when every modulus is above 16
// (SplitConsts::shift_ok), so ys = y + BIG + floor(m/2) > 0, and ys < 2^30 + 2^26 + m < 2^31
// <= 2^39 / m keeps the quotient exact.
constexpr uint32_t kShiftMax = 10;

// Wide path (kShiftMax < p <= kWideMax for some element: k_A above 62, e.g. 17 or more
// moduli, or 16 moduli with a small k): a' = u 2^p < 2^96 as six signed 16-bit limbs.  Each
// constant 2^(16 i) mod m is below m, so |y| < 6 2^16 m < BIG = m 2^22 and
// ys < m 2^23 <= 2^31: the single Barrett step stays exact for every modulus.  Every a' the
// scalings produce is below 2^(k_A + 1) <= 2^86 for 20 moduli, so p never exceeds kWideMax.
constexpr uint32_t kWideMax = 43;

__device__ __forceinline__ float residue_wide(uint64_t packed, uint32_t m, const uint32_t (&cw)[6], uint32_t magic,
                                              uint32_t big, uint32_t halfm, uint32_t fbase) {
  // the limbs are rebuilt for every modulus: this path is rare, and holding them for all
  // eight values would raise the register count of the common paths
  const uint64_t u = packed & ((1ull << 53) - 1);
  const uint32_t p = static_cast<uint32_t>(packed >> 53) & 0x3FFu;
  const uint64_t lo = u << p;                                            // bits 0..63
  const uint32_t hi = p ? static_cast<uint32_t>(u >> (64 - p)) : 0u;     // bits 64..95
  int acc = static_cast<int>(static_cast<uint32_t>(lo) & 0xFFFFu);
  acc += static_cast<int>(static_cast<uint32_t>(lo) >> 16) * static_cast<int>(cw[1]);
  acc += static_cast<int>(static_cast<uint32_t>(lo >> 32) & 0xFFFFu) * static_cast<int>(cw[2]);
  acc += static_cast<int>(static_cast<uint32_t>(lo >> 48)) * static_cast<int>(cw[3]);
  acc += static_cast<int>(hi & 0xFFFFu) * static_cast<int>(cw[4]);
  acc += static_cast<int>(hi >> 16) * static_cast<int>(cw[5]);
  const bool neg = (packed >> 63) != 0;
  const uint32_t ys = (neg ? big - static_cast<uint32_t>(acc) : static_cast<uint32_t>(acc)) + halfm;
  const uint32_t q = __umulhi(ys, magic) >> 7;
  return __int_as_float(static_cast<int>(fbase + (ys - q * m))) - 8388736.0f;
}

__device__ __forceinline__ float residue_shifted(int sx0, int sx1, int sx2, int sx3, uint32_t m, uint32_t c16,
                                                 uint32_t c32, uint32_t c48, uint32_t magic, uint32_t offs,
                                                 uint32_t fbase) {
  const uint32_t y = static_cast<uint32_t>(sx3 * static_cast<int>(c48) + sx2 * static_cast<int>(c32) +
                                           sx1 * static_cast<int>(c16) + sx0);
  const uint32_t ys = y + offs;
  const uint32_t q = __umulhi(ys, magic) >> 7;
  return __int_as_float(static_cast<int>(fbase + (ys - q * m))) - 8388736.0f;
}

// The integer paths: residues of the 8 packed values of one thread modulo every modulus,
// written as 8 bf16 (16 bytes) per plane at dst + t * plane_elems, for warps the FP32 limb
// path does not take.  Every lane of the warp must call it (the p tests are warp-uniform);
// lanes with dst == nullptr compute but do not store.
__device__ __forceinline__ void residues_to_planes(const uint64_t (&v)[8], const SplitConsts& c, uint16_t* dst,
                                                 long long plane_elems) {
  // per element: 16-bit limbs of u, the shift p and the sign, shared by all moduli
  uint32_t x0[8], x1[8], x2[8], pp[8];
  bool ng[8];
#pragma unroll
  for (int x = 0; x < 8; ++x) {
    const uint64_t u = v[x] & ((1ull << 53) - 1);
    x0[x] = static_cast<uint32_t>(u) & 0xFFFFu;
    x1[x] = static_cast<uint32_t>(u) >> 16;
    x2[x] = static_cast<uint32_t>(u >> 32);
    pp[x] = static_cast<uint32_t>(v[x] >> 53) & 0x3FFu;
    ng[x] = (v[x] >> 63) != 0;
  }
  uint32_t pmax = 0;
#pragma unroll
  for (int x = 0; x < 8; ++x) pmax = max(pmax, pp[x]);
  pmax = __reduce_max_sync(0xFFFFFFFFu, pmax);
  const bool warp_any_p = pmax != 0;
  if (warp_any_p && pmax <= kShiftMax && c.shift_ok) {
    // every a' of the warp is u 2^p with p <= kShiftMax: four signed 16-bit limbs of u 2^p
    int sx0[8], sx1[8], sx2[8], sx3[8];
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      const uint64_t a = (v[x] & ((1ull << 53) - 1)) << pp[x];  // < 2^63
      const int sg = ng[x] ? -1 : 1;
      sx0[x] = sg * static_cast<int>(static_cast<uint32_t>(a) & 0xFFFFu);
      sx1[x] = sg * static_cast<int>(static_cast<uint32_t>(a) >> 16);
      sx2[x] = sg * static_cast<int>(static_cast<uint32_t>(a >> 32) & 0xFFFFu);
      sx3[x] = sg * static_cast<int>(static_cast<uint32_t>(a >> 48));
    }
#pragma unroll 1
    for (int t = 0; t < c.s; ++t) {
      const uint32_t m = static_cast<uint32_t>(c.mod[t]), c16 = c.c16[t], c32 = c.c32[t], c48 = c.c48[t],
                     mg = c.magic[t];
      const uint32_t halfm = m >> 1, offs = (m << 22) + halfm, fbase = 0x4B000080u - halfm;
      uint32_t w[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const float lo = residue_shifted(sx0[2 * x], sx1[2 * x], sx2[2 * x], sx3[2 * x], m, c16, c32, c48, mg, offs,
                                         fbase);
        const float hi = residue_shifted(sx0[2 * x + 1], sx1[2 * x + 1], sx2[2 * x + 1], sx3[2 * x + 1], m, c16, c32,
                                         c48, mg, offs, fbase);
        w[x] = __byte_perm(__float_as_uint(lo), __float_as_uint(hi), 0x7632);  // two bf16
      }
      if (dst) *reinterpret_cast<uint4*>(dst + t * plane_elems) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else if (warp_any_p && pmax <= kWideMax) {
    // some a' of the warp is u 2^p with kShiftMax < p <= kWideMax: six 16-bit limbs
#pragma unroll 1
    for (int t = 0; t < c.s; ++t) {
      const uint32_t m = static_cast<uint32_t>(c.mod[t]), mg = c.magic[t];
      const uint32_t cw[6] = {1u, c.c16[t], c.c32[t], c.c48[t], c.c64[t], c.c80[t]};
      const uint32_t big = m << 22, halfm = m >> 1, fbase = 0x4B000080u - halfm;
      uint32_t w[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const float lo = residue_wide(v[2 * x], m, cw, mg, big, halfm, fbase);
        const float hi = residue_wide(v[2 * x + 1], m, cw, mg, big, halfm, fbase);
        w[x] = __byte_perm(__float_as_uint(lo), __float_as_uint(hi), 0x7632);  // two bf16
      }
      if (dst) *reinterpret_cast<uint4*>(dst + t * plane_elems) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else if (!warp_any_p) {
    // every a' of the warp is u itself (no power-of-two factor), some u >= 2^52
    int sx0[8], sx1[8], sx2[8];
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      const int sg = ng[x] ? -1 : 1;
      sx0[x] = sg * static_cast<int>(x0[x]);
      sx1[x] = sg * static_cast<int>(x1[x]);
      sx2[x] = sg * static_cast<int>(x2[x]);
    }
    // moduli unrolled: every constant is an operand at a fixed place of the parameter bank
#pragma unroll
    for (int t = 0; t < kMaxModuli; ++t) {
      if (t >= c.s) break;
      const uint32_t m = static_cast<uint32_t>(c.mod[t]), c16 = c.c16[t], c32 = c.c32[t], mg = c.magic[t];
      const uint32_t offs = c.offs[t], fbase = c.fbase[t];
      uint32_t w[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const float lo = residue_fast(sx0[2 * x], sx1[2 * x], sx2[2 * x], m, c16, c32, mg, offs, fbase);
        const float hi = residue_fast(sx0[2 * x + 1], sx1[2 * x + 1], sx2[2 * x + 1], m, c16, c32, mg, offs, fbase);
        w[x] = __byte_perm(__float_as_uint(lo), __float_as_uint(hi), 0x7632);  // two bf16
      }
      if (dst) *reinterpret_cast<uint4*>(dst + t * plane_elems) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
#pragma unroll 1
    for (int t = 0; t < c.s; ++t) {
      const uint32_t m = static_cast<uint32_t>(c.mod[t]), c16 = c.c16[t], c32 = c.c32[t], mg = c.magic[t];
      uint32_t w[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const uint32_t lo =
            residue_bf16(x0[2 * x], x1[2 * x], x2[2 * x], pp[2 * x], ng[2 * x], m, c16, c32, mg);
        const uint32_t hi = residue_bf16(x0[2 * x + 1], x1[2 * x + 1], x2[2 * x + 1], pp[2 * x + 1],
                                         ng[2 * x + 1], m, c16, c32, mg);
        w[x] = lo | (hi << 16);
      }
      if (dst) *reinterpret_cast<uint4*>(dst + t * plane_elems) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// ---------------------------------------------------------------- 13-bit limb path
// The common case: every a' of the warp is u < 2^52 with no power-of-two factor (for
// E = ceil(log2 max|a|) this holds whenever k_A <= 51, e.g. 14 moduli at every k >= 256).
// Then a' = sign * (x0 + x1 2^13 + x2 2^26 + x3 2^39) with 13-bit limbs x_l, and for an odd
// modulus 128 < m < 256
//   y = sign * (x0 + x1 (2^13 mod m) + x2 (2^26 mod m) + x3 (2^39 mod m)) ≡ a' (mod m),
// |y| <= 8191 (1 + 3 * 254) < 2^23, so y and every partial sum are exact in FP32.
// q = round(y/m) from one FMA with 1/m rounded to FP32 (error |y| |1/m - fl(1/m)| < 2^23 2^-32
// = 2^-9, below the distance 1/(2m) > 2^-9 from y/m to a half-integer, which holds for odd
// m), and r = y - q m (exact) is the symmetric representative in [-(m-1)/2, (m-1)/2].
// For m_0 = 256, y = sign * x0 (2^13 ≡ 0) and q = round((y + 1/4) / 256) (exact, never a
// tie) takes r into [-128, 127].  Every step is an FP32 FMA or add: no integer multiply.
// A zero limb, sum or remainder is +0 (an exact zero sum rounds to +0), so r's bf16 bits
// are those of the integer residue.

// Right shift that takes the 53-bit significand of x (exponent field raised to 1 for
// zeros and subnormals) to trunc(|x| 2^(k_A - E)); rb = 1075 + E - k_A for the row.
__device__ __forceinline__ int limb_shift(uint64_t raw, int rb) {
  const int ex = static_cast<int>(static_cast<uint32_t>(raw >> 52) & 0x7FFu);
  return rb - max(ex, 1);
}

// The row's rb: a row without finite nonzero entries (or a padding row) gets a shift that
// clears every value, as the residues of such rows are zero.
__device__ __forceinline__ int row_shift_base(int E, int kA) {
  return (E == OZ_EXP_EMPTY || E == OZ_EXP_NONFINITE) ? 4096 : 1075 + E - kA;
}

// The four signed limbs of one value as exact floats (rs >= 1, so u < 2^52).
__device__ __forceinline__ void limbs13(uint64_t raw, int rs, float (&x)[4]) {
  const uint32_t lo = static_cast<uint32_t>(raw), hi = static_cast<uint32_t>(raw >> 32);
  const uint32_t ex = (hi >> 20) & 0x7FFu;
  const uint32_t hm = (hi & 0xFFFFFu) | (ex != 0 ? 0x100000u : 0u);  // significand bits 32..52
  const int sh = min(rs, 63);
  const bool low = sh < 32;
  const uint32_t ul = low ? __funnelshift_r(lo, hm, sh) : (hm >> (sh & 31));
  const uint32_t uh = low ? (hm >> sh) : 0u;
  // sign * (2^23 + x) -/+ 2^23: exactly sign * x, and +0 for x = 0
  const uint32_t sbit = hi & 0x80000000u;
  const float sg = __uint_as_float(sbit | 0x3F800000u);
  const float nb = __uint_as_float(sbit ^ 0xCB000000u);
  x[0] = fmaf(__uint_as_float((ul & 0x1FFFu) | 0x4B000000u), sg, nb);
  x[1] = fmaf(__uint_as_float(((ul >> 13) & 0x1FFFu) | 0x4B000000u), sg, nb);
  x[2] = fmaf(__uint_as_float((__funnelshift_r(ul, uh, 26) & 0x1FFFu) | 0x4B000000u), sg, nb);
  x[3] = fmaf(__uint_as_float((uh >> 7) | 0x4B000000u), sg, nb);
}

// Residues of 8 values (raw FP64 patterns of one row, rb its shift base) modulo every
// modulus, 8 bf16 per plane at dst + t * plane_elems.  Every lane of the warp calls it;
// returns false, having written nothing, unless every value of the warp has rs >= 1 (the
// caller then takes the general path).  Lanes with dst == nullptr compute but do not store.
__device__ __forceinline__ bool residues13_to_planes(const uint64_t (&raw)[8], int rb, const SplitConsts& c,
                                                   uint16_t* dst, long long plane_elems) {
  int rs[8];
  int rmin = 1 << 30;
#pragma unroll
  for (int x = 0; x < 8; ++x) {
    rs[x] = limb_shift(raw[x], rb);
    rmin = min(rmin, rs[x]);
  }
  if (!__all_sync(0xFFFFFFFFu, rmin >= 1)) return false;
  float xl[8][4];
#pragma unroll
  for (int x = 0; x < 8; ++x) limbs13(raw[x], rs[x], xl[x]);
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23: adding it rounds |v| < 2^22 to an integer
#pragma unroll
  for (int t = 0; t < kMaxModuli; ++t) {
    if (t >= c.s) break;
    float r[8];
    if (t == 0) {  // m = 256
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const float q = fmaf(xl[x][0] + 0.25f, 0.00390625f, kMagic) - kMagic;
        r[x] = fmaf(-q, 256.0f, xl[x][0]);
      }
    } else {
      const float c1 = c.f13[t], c2 = c.f26[t], c3 = c.f39[t], iv = c.finv[t], mf = c.fmod[t];
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const float y = fmaf(xl[x][3], c3, fmaf(xl[x][2], c2, fmaf(xl[x][1], c1, xl[x][0])));
        const float q = fmaf(y, iv, kMagic) - kMagic;
        r[x] = fmaf(-q, mf, y);
      }
    }
    uint32_t w[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) w[x] = __byte_perm(__float_as_uint(r[2 * x]), __float_as_uint(r[2 * x + 1]), 0x7632);
    if (dst) *reinterpret_cast<uint4*>(dst + t * plane_elems) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  return true;
}

// 8 values of one row: the 13-bit limb path when it applies, the general path otherwise.
__device__ __forceinline__ void split8(const uint64_t (&raw)[8], int E, const SplitConsts& c, uint16_t* dst,
                                       long long plane_elems) {
  if (c.limb13_ok && residues13_to_planes(raw, row_shift_base(E, c.kA), c, dst, plane_elems)) return;
  uint64_t v[8];
#pragma unroll
  for (int x = 0; x < 8; ++x) v[x] = pack_scaled(__longlong_as_double(static_cast<long long>(raw[x])), E, c.kA);
  residues_to_planes(v, c, dst, plane_elems);
}

template <bool kRowsContiguous>
__global__ void __launch_bounds__(kSplitThreads, 4) split_kernel(int rows, int K, const double* __restrict__ X,
                                                              long long rs, long long ks,
                                                              const int32_t* __restrict__ exps,
                                                              const SplitConsts c, uint16_t* __restrict__ planes,
                                                              int rows_padded, int kp) {
  __shared__ uint64_t tile[kSplitTile][kSplitTile + 1];  // [kk][r]
  const int tid = threadIdx.x;
  const int k0 = blockIdx.x * kSplitTile;
  const int r0 = blockIdx.y * kSplitTile;

#pragma unroll
  for (int it = 0; it < (kSplitTile * kSplitTile) / kSplitThreads; ++it) {
    int r, kk;
    if (kRowsContiguous) {
      r = tid & 63;
      kk = (tid >> 6) + 4 * it;
    } else {
      kk = tid & 63;
      r = (tid >> 6) + 4 * it;
    }
    const int gr = r0 + r, gk = k0 + kk;
    tile[kk][r] = (gr < rows && gk < K) ? static_cast<uint64_t>(__double_as_longlong(__ldg(X + gr * rs + gk * ks)))
                                        : 0ull;  // +0.0 outside the operand
  }
  __syncthreads();

  const long long plane_elems = static_cast<long long>(rows_padded) * kp;
#pragma unroll 1
  for (int it = 0; it < (kSplitTile * kSplitTile / 8) / kSplitThreads; ++it) {
    const int item = tid + kSplitThreads * it;
    const int g = item & 7;   // group of 8 consecutive k
    const int r = item >> 3;  // row within the tile
    uint64_t v[8];
#pragma unroll
    for (int x = 0; x < 8; ++x) v[x] = tile[g * 8 + x][r];
    const int E = (r0 + r < rows) ? __ldg(exps + r0 + r) : OZ_EXP_EMPTY;
    uint16_t* dst = planes + static_cast<long long>(r0 + r) * kp + k0 + g * 8;
    split8(v, E, c, dst, plane_elems);
  }
}

// K-contiguous operand (B, column j = k contiguous): no transpose needed.  One thread
// takes 8 consecutive k of one row: 64 contiguous bytes in, 16 contiguous bytes out per
// modulus; a warp covers 256 consecutive k (2 KB read, 512 B written per plane).
__global__ void __launch_bounds__(256, 4) split_kcontig_kernel(int rows, int K, const double* __restrict__ X,
                                                            long long ld, const int32_t* __restrict__ exps,
                                                            const SplitConsts c, uint16_t* __restrict__ planes,
                                                            int rows_padded, int kp) {
  const int groups = kp >> 3;  // 8-k groups per row
  const long long item = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const bool valid = item < static_cast<long long>(rows_padded) * groups;  // all lanes stay for the vote
  const int r = valid ? static_cast<int>(item / groups) : 0;
  const int k0 = valid ? static_cast<int>(item - static_cast<long long>(r) * groups) * 8 : 0;
  uint64_t v[8];
  int E = OZ_EXP_EMPTY;
  if (valid && r < rows) {
    E = __ldg(exps + r);
    const double* src = X + static_cast<long long>(r) * ld + k0;
#pragma unroll
    for (int x = 0; x < 8; ++x) v[x] = (k0 + x < K) ? static_cast<uint64_t>(__double_as_longlong(__ldg(src + x))) : 0ull;
  } else {
#pragma unroll
    for (int x = 0; x < 8; ++x) v[x] = 0;
  }
  split8(v, E, c, valid ? planes + static_cast<long long>(r) * kp + k0 : nullptr,
         static_cast<long long>(rows_padded) * kp);
}

// Steps a1 + a2 for a K-contiguous operand (B: column j is k contiguous) with one DRAM read
// of each column: one block per row of the operand (a column of B) takes the row's largest
// magnitude (the same integer maximum of the 63-bit patterns as the exponent kernels),
// writes F_j = ceil(log2 max), then splits the row, whose second read comes from L2 (a few
// blocks per SM keep about 40 MB of rows in flight, well inside the 129 MB L2).  Padding rows
// (r >= rows) write zero planes.
constexpr int kFusedThreads = 256;

__global__ void __launch_bounds__(kFusedThreads, 3)
    split_kcontig_fused_kernel(int rows, int K, const double* __restrict__ X, long long ld, const SplitConsts c,
                               int32_t* __restrict__ exps, uint16_t* __restrict__ planes, int rows_padded, int kp) {
  __shared__ unsigned long long warp_max[kFusedThreads / 32];
  const int r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int groups = kp >> 3;
  const double* src = X + static_cast<long long>(r) * ld;
  unsigned long long mag = 0;
  if (r < rows) {
#pragma unroll 8
    for (int kk = tid; kk < K; kk += kFusedThreads) mag = max(mag, magnitude_bits(__ldg(src + kk)));
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) mag = max(mag, __shfl_xor_sync(0xFFFFFFFFu, mag, off));
  if (lane == 0) warp_max[warp] = mag;
  __syncthreads();
  mag = warp_max[0];
#pragma unroll
  for (int w = 1; w < kFusedThreads / 32; ++w) mag = max(mag, warp_max[w]);
  const int E = mag ? ceil_log2_code(__longlong_as_double(static_cast<long long>(mag))) : OZ_EXP_EMPTY;
  if (tid == 0 && r < rows) exps[r] = E;
  const long long plane_elems = static_cast<long long>(rows_padded) * kp;
  for (int g0 = 0; g0 < groups; g0 += kFusedThreads) {  // block-uniform trip count
    const int g = g0 + tid;
    const int k0 = 8 * g;
    uint64_t v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
      v[e] = (r < rows && g < groups && k0 + e < K) ? static_cast<uint64_t>(__double_as_longlong(__ldg(src + k0 + e)))
                                                    : 0ull;
    split8(v, r < rows ? E : OZ_EXP_EMPTY, c, g < groups ? planes + static_cast<long long>(r) * kp + k0 : nullptr,
           plane_elems);
  }
}

cudaError_t launch_split_fused_kcontig(int rows, int k, const double* X, long long ld, const SplitConsts& c,
                                       int32_t* exps, uint16_t* planes, int rows_padded, int kp,
                                       cudaStream_t stream) {
  split_kcontig_fused_kernel<<<rows_padded, kFusedThreads, 0, stream>>>(rows, k, X, ld, c, exps, planes, rows_padded,
                                                                        kp);
  return cudaGetLastError();
}

cudaError_t launch_split(int rows, int k, const double* X, long long row_stride, long long k_stride,
                         const int32_t* exps, const SplitConsts& c, uint16_t* planes, int rows_padded, int kp,
                         cudaStream_t stream) {
  if (row_stride == 1) {  // A: rows contiguous, transpose through shared memory
    dim3 grid(kp / kSplitTile, rows_padded / kSplitTile);
    split_kernel<true><<<grid, kSplitThreads, 0, stream>>>(rows, k, X, row_stride, k_stride, exps, c, planes,
                                                           rows_padded, kp);
  } else if (k_stride == 1) {  // B: K contiguous, direct
    const long long items = static_cast<long long>(rows_padded) * (kp / 8);
    split_kcontig_kernel<<<static_cast<unsigned>((items + 255) / 256), 256, 0, stream>>>(rows, k, X, row_stride,
                                                                                        exps, c, planes,
                                                                                        rows_padded, kp);
  } else {
    dim3 grid(kp / kSplitTile, rows_padded / kSplitTile);
    split_kernel<false><<<grid, kSplitThreads, 0, stream>>>(rows, k, X, row_stride, k_stride, exps, c, planes,
                                                            rows_padded, kp);
  }
  return cudaGetLastError();
}

}  // namespace oz
