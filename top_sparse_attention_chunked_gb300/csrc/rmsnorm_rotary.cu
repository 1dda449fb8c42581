// RMSNorm + rotary embedding in fp32, the step that produces the query and
// key vectors (q, k, index query qI, index key kI) the attention step reads.
//
// PR #33997 ("[CUDA] Support FP16 KV cache and FP16 query/key in
// DynamicSparseAttention<BFloat16> and FP32 rotary cache / FP16 output in
// RMSNormRotary"), Description item 1: RMSNorm and RoPE computed in fp32 with
// no intermediate BF16 rounding, from a BF16 or FP32 cos/sin cache, rounded
// once to a BF16 or FP16 output.
//
// Per head vector x of D elements at position p:
//   y = x * gamma / sqrt(mean(x^2) + eps)
//   out_i       = y_i cos[p,i] - y_{i+r/2} sin[p,i]     (i < r/2)
//   out_{i+r/2} = y_{i+r/2} cos[p,i] + y_i sin[p,i]
//   out_i       = y_i                                   (i >= r)
//
// One warp per token and group of up to four heads (D/32 elements a lane);
// the token's cos / sin values are loaded once per group. The per-vector
// arithmetic (rope_math.cuh) is a shuffle-butterfly sum of squares in fp32,
// the IEEE square root and division, and an exact 2^-+64 rescale when that
// sum leaves [2^-100, 2^100], all in explicit round-to-nearest operations. The normalised
// vector is staged in shared memory so that each lane can read its rotation
// partner for any even rotary width.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstdio>

#include "dsa_internal.h"
#include "rope_math.cuh"

namespace dsa {

int report_error(int status, const char* msg);   // sets dsa_last_error_string()

namespace {

constexpr int kRopeWarps = 8;

struct RopeParams {
  const void* x;
  const float* gamma;
  const void* cos_cache;
  const void* sin_cache;
  const int32_t* positions;
  void* y;
  long long rows;        // tokens * heads
  int heads, rotary_dim, max_pos;
  float eps;
  int x_dtype, cos_dtype, y_dtype;
};

__device__ __forceinline__ float load_half(const void* base, long long i, bool fp16) {
  const uint16_t u = static_cast<const uint16_t*>(base)[i];
  if (fp16) return __half2float(__ushort_as_half(u));
  return __uint_as_float(static_cast<uint32_t>(u) << 16);
}

__device__ __forceinline__ uint16_t to_out(float v, bool fp16) {
  if (fp16) return __half_as_ushort(__float2half_rn(v));
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// N consecutive 16-bit values (N = 2 or 4) in one vector load.
template <int N>
__device__ __forceinline__ uint2 load16_raw(const void* base, long long i) {
  const uint16_t* q = static_cast<const uint16_t*>(base) + i;
  if constexpr (N == 4) return *reinterpret_cast<const uint2*>(q);
  return make_uint2(*reinterpret_cast<const uint32_t*>(q), 0u);
}

template <int N>
__device__ __forceinline__ void to_floats(uint2 u, bool fp16, float* v) {
  const uint32_t w[2] = {u.x, u.y};
#pragma unroll
  for (int k = 0; k < N / 2; ++k) {
    if (fp16) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
      v[2 * k] = f.x;
      v[2 * k + 1] = f.y;
    } else {
      v[2 * k] = __uint_as_float(w[k] << 16);
      v[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  }
}

template <int N>
__device__ __forceinline__ void load16(const void* base, long long i, bool fp16, float* v) {
  to_floats<N>(load16_raw<N>(base, i), fp16, v);
}

// One warp per (token, group of up to kHeadsPerWarp heads): the token's
// cos / sin values are loaded once for the group. `vec_cs`: a lane's angle
// indices are consecutive (rotary_dim / 2 a multiple of D / 32) and the caches
// are aligned for vector loads.
constexpr int kHeadsPerWarp = 4;

// FULL: the rotary width is the head dim and the caches take vector loads
// (the common case). Every element then rotates, element i's partner i +- D/2
// sits in lane ^ 16 (D/2 / E = 16 for either head dim) and the first half of
// each pair is lanes 0-15, so the per-element width checks and the general
// partner lookup drop out; the arithmetic is the same.
template <int D, bool FULL>
__global__ void __launch_bounds__(kRopeWarps * 32) rmsnorm_rotary_kernel(const RopeParams p,
                                                                         long long units,
                                                                         int groups, bool vec_cs) {
  constexpr int E = D / 32;   // elements per lane
  __shared__ float s_y[kRopeWarps][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool xf16 = p.x_dtype == DSA_FP16, yf16 = p.y_dtype == DSA_FP16;
  const bool cf32 = p.cos_dtype == DSA_FP32;
  const int h = p.rotary_dim >> 1;
  const int i0 = lane * E;                       // this lane's first element
  const bool rot = FULL || i0 < p.rotary_dim;   // all E elements rotate (vec_cs) or check each
  float g[E];
#pragma unroll
  for (int e = 0; e < E; ++e) g[e] = __ldg(p.gamma + i0 + e);
  for (long long u = static_cast<long long>(blockIdx.x) * kRopeWarps + warp; u < units;
       u += static_cast<long long>(gridDim.x) * kRopeWarps) {
    // 32-bit division whenever the unit count allows it
    const long long tok = units < (1LL << 31) ? static_cast<long long>(static_cast<int>(u) / groups)
                                              : u / groups;
    const int h0 = static_cast<int>(u - tok * groups) * kHeadsPerWarp;
    const int nh = min(kHeadsPerWarp, p.heads - h0);
    // the token's angles for this lane's elements
    float c[E], sn[E];
    if (FULL || h > 0) {
      int pos = __ldg(p.positions + tok);
      pos = pos < 0 ? 0 : (pos >= p.max_pos ? p.max_pos - 1 : pos);   // clamped to the cache
      const long long row = static_cast<long long>(pos) * h;
      if (FULL || (vec_cs && rot)) {
        const long long j0 = row + (i0 < h ? i0 : i0 - h);
        if (cf32) {
          if constexpr (E == 4) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.cos_cache) + j0));
            const float4 b = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.sin_cache) + j0));
            c[0] = a.x; c[1] = a.y; c[2] = a.z; c[3] = a.w;
            sn[0] = b.x; sn[1] = b.y; sn[2] = b.z; sn[3] = b.w;
          } else {
            const float2 a = __ldg(reinterpret_cast<const float2*>(static_cast<const float*>(p.cos_cache) + j0));
            const float2 b = __ldg(reinterpret_cast<const float2*>(static_cast<const float*>(p.sin_cache) + j0));
            c[0] = a.x; c[1] = a.y;
            sn[0] = b.x; sn[1] = b.y;
          }
        } else {
          load16<E>(p.cos_cache, j0, false, c);
          load16<E>(p.sin_cache, j0, false, sn);
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int i = i0 + e;
          c[e] = 1.0f;
          sn[e] = 0.0f;
          if (i < p.rotary_dim) {
            const long long ci = row + (i < h ? i : i - h);
            c[e] = cf32 ? __ldg(static_cast<const float*>(p.cos_cache) + ci) : load_half(p.cos_cache, ci, false);
            sn[e] = cf32 ? __ldg(static_cast<const float*>(p.sin_cache) + ci) : load_half(p.sin_cache, ci, false);
          }
        }
      }
    }
    // every head's loads in flight before the first is used
    uint2 raw[kHeadsPerWarp];
    const long long base0 = (tok * p.heads + h0) * D + i0;
#pragma unroll
    for (int hh = 0; hh < kHeadsPerWarp; ++hh)
      raw[hh] = hh < nh ? load16_raw<E>(p.x, base0 + static_cast<long long>(hh) * D) : make_uint2(0, 0);
#pragma unroll
    for (int hh = 0; hh < kHeadsPerWarp; ++hh) {
      if (hh >= nh) break;
      const long long base = base0 + static_cast<long long>(hh) * D;
      float x[E];
      to_floats<E>(raw[hh], xf16, x);
      float y[E];
      rms_normalize<E, D>(x, g, p.eps, y);
      float partner[E];
      if constexpr (FULL) {
#pragma unroll
        for (int e = 0; e < E; ++e) partner[e] = __shfl_xor_sync(0xffffffffu, y[e], 16);
      } else if (vec_cs) {
        // r/2 is a multiple of E: element i's partner i +- r/2 sits in lane
        // lane +- r/(2E) at the same slot, one shuffle away
        const int src = !rot ? lane : (i0 < h ? lane + h / E : lane - h / E);
#pragma unroll
        for (int e = 0; e < E; ++e) partner[e] = __shfl_sync(0xffffffffu, y[e], src);
      } else if (h > 0) {
#pragma unroll
        for (int e = 0; e < E; ++e) s_y[warp][i0 + e] = y[e];
        __syncwarp();
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int i = i0 + e;
          partner[e] = i < p.rotary_dim ? s_y[warp][i < h ? i + h : i - h] : 0.0f;
        }
        __syncwarp();   // partner reads done before the next vector's writes
      }
      uint16_t o[E];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int i = i0 + e;
        float v = y[e];
        if constexpr (FULL) v = rope_rotate(v, partner[e], c[e], sn[e], lane < 16);
        else if (i < p.rotary_dim) v = rope_rotate(v, partner[e], c[e], sn[e], i < h);
        o[e] = to_out(v, yf16);
      }
      uint16_t* out = static_cast<uint16_t*>(p.y) + base;
      if constexpr (E == 4) {
        *reinterpret_cast<uint2*>(out) =
            make_uint2(o[0] | (static_cast<uint32_t>(o[1]) << 16), o[2] | (static_cast<uint32_t>(o[3]) << 16));
      } else {
        *reinterpret_cast<uint32_t*>(out) = o[0] | (static_cast<uint32_t>(o[1]) << 16);
      }
    }
  }
}

bool aligned_to(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" int dsa_rmsnorm_rotary(const dsa_rope_problem* rp, const void* x, const float* gamma,
                                  const void* cos_cache, const void* sin_cache,
                                  const int32_t* positions, void* y, void* stream) {
  reset_launches();
  if (!rp) return report_error(DSA_ERR_INVALID_ARG, "rope problem is NULL");
  const int D = rp->head_dim, r = rp->rotary_dim;
  if (rp->tokens < 0) return report_error(DSA_ERR_INVALID_ARG, "tokens must be >= 0");
  if (rp->heads < 1) return report_error(DSA_ERR_INVALID_ARG, "heads must be >= 1");
  if (D != 64 && D != 128) return report_error(DSA_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (r < 0 || r > D || (r & 1)) return report_error(DSA_ERR_INVALID_ARG, "rotary_dim must be even and in 0..head_dim");
  if (r > 0 && rp->max_pos < 1) return report_error(DSA_ERR_INVALID_ARG, "max_pos must be >= 1");
  if (!(rp->eps >= 0.0f) || std::isinf(rp->eps)) return report_error(DSA_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if ((rp->x_dtype != DSA_BF16 && rp->x_dtype != DSA_FP16) ||
      (rp->y_dtype != DSA_BF16 && rp->y_dtype != DSA_FP16))
    return report_error(DSA_ERR_UNSUPPORTED, "x and y must be BF16 or FP16");
  if (r > 0 && rp->cos_dtype != DSA_FP32 && rp->cos_dtype != DSA_BF16)
    return report_error(DSA_ERR_UNSUPPORTED, "the cos / sin caches must be FP32 or BF16");
  if (!x || !gamma || !y) return report_error(DSA_ERR_INVALID_ARG, "x, gamma and y are required");
  if (r > 0 && (!cos_cache || !sin_cache || !positions))
    return report_error(DSA_ERR_INVALID_ARG, "cos_cache, sin_cache and positions are required when rotary_dim > 0");
  const size_t ca = rp->cos_dtype == DSA_FP32 ? 4 : 2;
  if (!aligned_to(x, 16) || !aligned_to(y, 16) || !aligned_to(gamma, 4) ||
      (r > 0 && (!aligned_to(cos_cache, ca) || !aligned_to(sin_cache, ca) || !aligned_to(positions, 4))))
    return report_error(DSA_ERR_MISALIGNED, "x and y must be 16-byte aligned; gamma, positions and the caches element-aligned");
  const long long rows = rp->tokens * rp->heads;
  const long long bytes = rows * D * 2;
  const uintptr_t x0 = reinterpret_cast<uintptr_t>(x), y0 = reinterpret_cast<uintptr_t>(y);
  if (x0 != y0 && x0 < y0 + static_cast<uintptr_t>(bytes) && y0 < x0 + static_cast<uintptr_t>(bytes))
    return report_error(DSA_ERR_INVALID_ARG, "y overlaps x without being the same array");
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
    cudaGetLastError();
    return report_error(DSA_ERR_NO_DEVICE, "no usable CUDA device");
  }
  if (rows == 0) return DSA_OK;
  RopeParams p;
  p.x = x;
  p.gamma = gamma;
  p.cos_cache = cos_cache;
  p.sin_cache = sin_cache;
  p.positions = positions;
  p.y = y;
  p.rows = rows;
  p.heads = rp->heads;
  p.rotary_dim = r;
  p.max_pos = rp->max_pos;
  p.eps = rp->eps;
  p.x_dtype = rp->x_dtype;
  p.cos_dtype = rp->cos_dtype;
  p.y_dtype = rp->y_dtype;
  const int groups = (rp->heads + kHeadsPerWarp - 1) / kHeadsPerWarp;
  const long long units = rp->tokens * groups;
  long long blocks = (units + kRopeWarps - 1) / kRopeWarps;
  const long long most = static_cast<long long>(sms) * 64;
  if (blocks > most) blocks = most;
  // vector loads of a lane's cos / sin values: its E angle indices are
  // consecutive when r/2 is a multiple of E, and the row starts then stay
  // aligned to E elements if the caches are
  const int E = D / 32;
  const size_t cs_vec = static_cast<size_t>(E) * (rp->cos_dtype == DSA_FP32 ? 4 : 2);
  const bool vec_cs = r > 0 && ((r / 2) % E) == 0 && aligned_to(cos_cache, cs_vec) &&
                      aligned_to(sin_cache, cs_vec);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool full = vec_cs && r == D;
  const dim3 grid(static_cast<unsigned>(blocks)), block(kRopeWarps * 32);
  const cudaError_t e =
      D == 128 ? (full ? launch_kernel("rmsnorm_rotary_kernel", rmsnorm_rotary_kernel<128, true>, grid, block, 0,
                                       st, false, p, units, groups, vec_cs)
                       : launch_kernel("rmsnorm_rotary_kernel", rmsnorm_rotary_kernel<128, false>, grid, block,
                                       0, st, false, p, units, groups, vec_cs))
               : (full ? launch_kernel("rmsnorm_rotary_kernel", rmsnorm_rotary_kernel<64, true>, grid, block, 0,
                                       st, false, p, units, groups, vec_cs)
                       : launch_kernel("rmsnorm_rotary_kernel", rmsnorm_rotary_kernel<64, false>, grid, block,
                                       0, st, false, p, units, groups, vec_cs));
  if (e != cudaSuccess) {
    char buf[160];
    snprintf(buf, sizeof(buf), "rmsnorm_rotary launch: %s", cudaGetErrorString(e));
    return report_error(DSA_ERR_CUDA, buf);
  }
  return DSA_OK;
}
