// Order-preserving keys and coarse radix digits of fp32 scores, shared by the select
// kernels ("Serving GLM5.2 NVFP4 Agentic Workload with SGLang", "Kernel Optimization >
// TopK-V2", Fig. 3: scores are binned by an order-preserving unsigned key), and the
// warp-level inclusive scan both kernels build their block scans from.
#pragma once

#include <cstdint>

namespace topk {
namespace {

// Order-preserving 32-bit key: larger key <=> larger score. -0.0 is folded onto
// +0.0; every NaN maps to 0, below -inf (0x007FFFFF).
__device__ __forceinline__ uint32_t f2key(float x) {
  const uint32_t u = __float_as_uint(x);
  const uint32_t a = u & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return 0u;
  if (a == 0u) return 0x80000000u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Coarse 12-bit digit, monotone non-decreasing in the score: sign, a 5-bit exponent
// window (|x| in [2^-15, 2^17)) and 6 mantissa bits, clamped at both ends. Equal
// scores share a digit (-0 is folded onto +0 by adding +0); NaN is first mapped to
// -inf, which together with every score at or below -2^17 lands in bin 0.
__device__ __forceinline__ uint32_t coarse_digit(float x) {
  const float xc = __fadd_rn(fmaxf(x, __int_as_float(0xFF800000)), 0.0f);
  const float ax = fminf(fmaxf(fabsf(xc), 3.0517578125e-05f), 131071.99f);
  const uint32_t m = (__float_as_uint(ax) >> 17) - 7168u;  // in [0, 2047]
  const uint32_t s = (uint32_t)((int32_t)__float_as_uint(xc) >> 31);
  return ((m ^ s) ^ 0x800u) & 0xFFFu;
}

// A float t such that x < t implies coarse_digit(x) < b (a conservative filter used
// to skip vectors without computing digits). NaN never satisfies x < t.
__device__ __forceinline__ float skip_below(uint32_t b) {
  if (b == 0u) return __uint_as_float(0xFF800000u);  // -inf: nothing is skipped
  if (b < 2048u) {
    const uint32_t j = 2048u - b;  // (2047 - b) + 1, in [1, 2047]
    return -__uint_as_float((j + 7168u) << 17);
  }
  if (b == 2048u) return 0.0f;
  return __uint_as_float(((b - 2048u) + 7168u) << 17);
}

__device__ __forceinline__ int warp_incl_scan(int x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

}  // namespace
}  // namespace topk
