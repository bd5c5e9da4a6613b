// oz_fp.cuh -- exact IEEE-754 binary64 field helpers shared by the kernels.
#pragma once

#include <cstdint>

#include "oz_internal.h"

namespace oz {

// |x| as its 63-bit pattern: for x, y not NaN, |x| < |y| iff the patterns compare the same
// way, and every NaN pattern lies above infinity's.
__device__ __forceinline__ unsigned long long magnitude_bits(double x) {
  return static_cast<unsigned long long>(__double_as_longlong(x)) & 0x7FFFFFFFFFFFFFFFull;
}

// ceil(log2 |x|) from the IEEE-754 fields; OZ_EXP_EMPTY for 0, OZ_EXP_NONFINITE for Inf/NaN.
__device__ __forceinline__ int ceil_log2_code(double x) {
  const uint64_t b = static_cast<uint64_t>(__double_as_longlong(x)) & 0x7FFFFFFFFFFFFFFFull;
  if (b == 0) return OZ_EXP_EMPTY;
  const int ex = static_cast<int>(b >> 52);
  const uint64_t f = b & 0x000FFFFFFFFFFFFFull;
  if (ex == 0x7FF) return OZ_EXP_NONFINITE;
  if (ex == 0) {  // subnormal: |x| = f * 2^-1074, f in [2^(L-1), 2^L)
    const int L = 64 - __clzll(static_cast<long long>(f));
    return -1074 + ((f & (f - 1)) ? L : L - 1);
  }
  return (ex - 1023) + (f != 0 ? 1 : 0);
}

// floor(log2 |x|) from the IEEE-754 fields; OZ_EXP_EMPTY for 0, OZ_EXP_NONFINITE for Inf/NaN.
__device__ __forceinline__ int floor_log2_code(double x) {
  const uint64_t b = static_cast<uint64_t>(__double_as_longlong(x)) & 0x7FFFFFFFFFFFFFFFull;
  if (b == 0) return OZ_EXP_EMPTY;
  const int ex = static_cast<int>(b >> 52);
  if (ex == 0x7FF) return OZ_EXP_NONFINITE;
  if (ex == 0) return -1075 + (64 - __clzll(static_cast<long long>(b)));  // subnormal: f 2^-1074
  return ex - 1023;
}

template <bool kFloor>
__device__ __forceinline__ int log2_code(double x) {
  return kFloor ? floor_log2_code(x) : ceil_log2_code(x);
}

}  // namespace oz
