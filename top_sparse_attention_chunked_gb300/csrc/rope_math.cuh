// The fp32 arithmetic of RMSNorm + rotary embedding for one head vector held
// by a warp (E = D / 32 consecutive elements a lane), shared by the kernels
// that apply it so that they give the same bits. Every operation is an
// explicit round-to-nearest intrinsic, which the compiler never contracts
// into a fused multiply-add.
#pragma once

#include <cstdint>

namespace dsa {

// y = x * g / sqrt(mean(x^2) + eps) for the warp's vector, 1/sqrt taken in one
// correctly rounded step. When the fp32 sum of squares leaves [2^-100, 2^100]
// (or is zero) the vector is first scaled by 2^-+64 (exact, chosen from its
// absmax) so that the sum neither overflows nor vanishes; the scale cancels in
// y, and eps takes its square (in two steps: 2^128 is not an fp32 value). x is
// overwritten by the scaled copy.
template <int E, int D>
__device__ __forceinline__ void rms_normalize(float* x, const float* g, float eps_in, float* y) {
  float ss = 0.0f;
#pragma unroll
  for (int e = 0; e < E; ++e) ss = __fmaf_rn(x[e], x[e], ss);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
  float eps = eps_in;
  if (!(ss >= 0x1p-100f && ss <= 0x1p100f)) {
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    float sc = 1.0f;
    if (amax > 0x1p60f) {
      sc = 0x1p-64f;
      eps = __fmul_rn(__fmul_rn(eps_in, 0x1p-64f), 0x1p-64f);
    } else if (amax > 0.0f && amax < 0x1p-60f) {
      sc = 0x1p64f;
      eps = __fmul_rn(__fmul_rn(eps_in, 0x1p64f), 0x1p64f);
    }
    ss = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      x[e] = __fmul_rn(x[e], sc);
      ss = __fmaf_rn(x[e], x[e], ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
  }
  const float inv = __frsqrt_rn(__fadd_rn(__fmul_rn(ss, 1.0f / D), eps));   // one rounding
#pragma unroll
  for (int e = 0; e < E; ++e) y[e] = __fmul_rn(__fmul_rn(x[e], inv), g[e]);
}

// One rotated element: the first half of a pair (i < r/2) gives
// v c - partner s, the second half v c + partner s.
__device__ __forceinline__ float rope_rotate(float v, float partner, float c, float s, bool first) {
  const float a = __fmul_rn(v, c), b = __fmul_rn(partner, s);
  return first ? __fsub_rn(a, b) : __fadd_rn(a, b);
}

}  // namespace dsa
