// Cache append: write the S new tokens of every sequence into the index-key
// and K/V caches, quantising to INT8 on the way in when the cache is INT8.
//
// PR #33997 ("[CUDA] Support FP16 KV cache and FP16 query/key in
// DynamicSparseAttention<BFloat16> ..."), Files changed: the implementation
// file holds the cache writes next to the attention kernels; its description
// names the quantized cache. The new tokens are the last S rows of a sequence
// whose cache holds T_b rows, so token s lands in row T_b - S + s.
//
// INT8: per token and KV head, scale = absmax / 127 and code = the nearest
// integer to x / scale (ties to even), clamped to +-127; an all-zero row gets
// scale 0 and codes 0. Both divisions are IEEE fp32 (round to nearest), so the
// codes are a deterministic function of the input. A 16-bit cache of the other
// 16-bit type takes the value rounded to nearest even.
//
// K/V tiles are staged in shared memory, then eight lanes take each
// 128-element row (16 elements a lane); index-key rows are copied in 16-byte
// pieces. The work is a pure stream (each input byte read once, each output
// byte written once), so the kernel is sized for bytes in flight, not
// arithmetic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dsa_internal.h"
#include "sm100_ptx.cuh"

namespace dsa {
namespace {

constexpr int kAppThreads = 256;

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// 8 packed 16-bit values -> floats (exact)
__device__ __forceinline__ void unpack8(uint4 u, bool fp16, float* x) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (fp16) {
      const __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      const float2 f = __half22float2(h);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    } else {
      // bf16 -> fp32 is a 16-bit shift
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf162(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// The code of x is rint(RN(x / scale)) with ties to even. Multiplying by
// inv = RN(1 / scale) instead gives q with |q - x/scale| <= |x/scale| * 2^-23
// (two roundings of relative size at most 2^-24; |x/scale| <= 128, so at most
// 2^-16), and RN(x/scale) lies within half an fp32 ulp (at most 2^-18 below
// 128) of x/scale. Half-integers are exact fp32 values, so when q is farther
// than kTieBand (2^-12, well above both) from every half-integer, q, x/scale
// and RN(x/scale) all lie strictly between the same two half-integers and
// round to the same integer. Only inputs inside the band take the IEEE
// division. inv must be finite and normal (scale >= 2^-126 and at most
// FLT_MAX/127 keep it so); below 2^-126 every element is divided.
constexpr float kTieBand = 1.0f / 4096.0f;
constexpr float kMinNormal = 1.17549435e-38f;   // 2^-126
// Adding 1.5 * 2^23 to |q| < 2^22 lands in [2^23, 2^24), where fp32 steps by
// 1, so the sum is q rounded to the nearest integer, ties to even; the
// integer sits in the low mantissa bits (bits minus kRoundBits), so its low
// byte is the int8 code's two's-complement byte.
constexpr float kRound = 12582912.0f;            // 1.5 * 2^23
constexpr uint32_t kRoundBits = 0x4B400000u;     // bit pattern of kRound

// Codes of one lane's 16 elements, packed into four words. Every lane of the
// warp must call it (the fallback is taken by the whole warp, so that the
// common case issues no division at all). With a normal scale no clamp is
// needed: |x| <= absmax and scale >= (absmax/127)(1 - 2^-24) bound |x/scale|
// and |q| below 127.5, so every code is within +-127.
__device__ __forceinline__ uint4 quantize16(const float* x, float scale) {
  uint32_t t[16];
  uint32_t slow = 0;          // elements whose code needs the IEEE quotient
  if (scale >= kMinNormal) {
    const float inv = __frcp_rn(scale);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float q = x[e] * inv;
      const float sum = q + kRound;
      const float r = sum - kRound;                // q rounded, exact
      t[e] = __float_as_uint(sum);
      if (fabsf(fabsf(q - r) - 0.5f) <= kTieBand) slow |= 1u << e;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 16; ++e) t[e] = kRoundBits;   // code 0
    if (scale > 0.0f) slow = 0xffffu;   // tiny scale: 1/scale may overflow
  }
  if (__any_sync(0xffffffffu, slow != 0)) {
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      if ((slow >> e) & 1u) {
        const float c = fminf(fmaxf(rintf(__fdiv_rn(x[e], scale)), -127.0f), 127.0f);
        t[e] = kRoundBits + static_cast<uint32_t>(static_cast<int>(c));
      }
    }
  }
  // byte 0 of each word, four to a word
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    w[k] = __byte_perm(__byte_perm(t[4 * k], t[4 * k + 1], 0x0040),
                       __byte_perm(t[4 * k + 2], t[4 * k + 3], 0x0040), 0x5410);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ void unpack16(const uint4* u, bool fp16, float* x) {
  unpack8(u[0], fp16, x);
  unpack8(u[1], fp16, x + 8);
}

__device__ __forceinline__ uint4 convert8(uint4 u, bool src_fp16) {
  float x[8];
  unpack8(u, src_fp16, x);
  if (src_fp16)   // FP16 -> BF16
    return make_uint4(pack_bf162(x[0], x[1]), pack_bf162(x[2], x[3]), pack_bf162(x[4], x[5]),
                      pack_bf162(x[6], x[7]));
  return make_uint4(pack_half2(x[0], x[1]), pack_half2(x[2], x[3]), pack_half2(x[4], x[5]),
                    pack_half2(x[6], x[7]));
}

// Grid: z = the sequence b, y = 0 (index keys), 1 (K) or 2 (V), x = tiles of
// rows. For one sequence the new K (or V) rows of all heads are one
// contiguous span of q_len * Hkv rows, and in a dense cache so are the rows
// they go to (rows (T_b - q_len) * Hkv ...), whatever the head; a tile is
// kAppRowsK of them. In a paged cache each row's destination goes through the
// block table, and a row whose entry lies outside the pool is not written. The tile is staged in shared memory with cp.async (eight 16-byte
// copies per thread in flight, no registers held), then eight lanes take a
// row: lane l reads bytes 16l and 128 + 16l of it (elements 8l..8l+7 and
// 64+8l..64+8l+7), so each 8-lane phase of a shared load covers 128
// consecutive bytes. Index keys are copied through registers.
constexpr int kAppRowsK = 128;                               // K/V rows per tile
constexpr int kAppSmem = kAppRowsK * DSA_HEAD_DIM * 2;        // 32 KB (no opt-in needed)
constexpr int kAppRowsI = 2 * kAppThreads / 8;               // index-key rows per tile (64)

template <bool PAGED>
__global__ void __launch_bounds__(kAppThreads) cache_append_kernel(const AppendParams p) {
  extern __shared__ __align__(16) uint8_t tile[];
  const int b = blockIdx.z;
  const int kind = blockIdx.y;
  const long long tok0 = static_cast<long long>(b) * p.S;                  // first source token
  const long long dst0 = static_cast<long long>(b) * p.cap + (p.lens.T[b] - p.S);  // its row
  if (kind == 0) {
    // index keys are BF16 on both sides: a plain copy, 8 pieces per row
    const uint16_t* src = static_cast<const uint16_t*>(p.kI_new);
    uint16_t* dst = static_cast<uint16_t*>(p.kI);
    const long long r0 = static_cast<long long>(blockIdx.x) * kAppRowsI;
    if (r0 >= p.S) return;
    uint4 u[2];
    long long r[2];
    int part[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int piece = i * kAppThreads + threadIdx.x;
      r[i] = r0 + (piece >> 3);
      part[i] = piece & 7;
      u[i] = make_uint4(0, 0, 0, 0);
      if (r[i] < p.S) u[i] = ld_stream(src + (tok0 + r[i]) * DSA_IDX_DIM + part[i] * 8);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if (r[i] >= p.S) continue;
      long long row = dst0 + r[i];
      if constexpr (PAGED) {
        bool bad = false;
        row = cache_row(p.pg, b, p.cap, p.lens.T[b] - p.S + static_cast<int>(r[i]), &bad);
        if (bad) continue;   // never write through an entry outside the pool
      }
      *reinterpret_cast<uint4*>(dst + row * DSA_IDX_DIM + part[i] * 8) = u[i];
    }
    return;
  }
  const bool is_k = (kind == 1);
  const long long nrows = static_cast<long long>(p.S) * p.Hkv;
  const long long r0 = static_cast<long long>(blockIdx.x) * kAppRowsK;
  if (r0 >= nrows) return;
  const int rows = static_cast<int>(nrows - r0 < kAppRowsK ? nrows - r0 : kAppRowsK);
  const uint8_t* src = static_cast<const uint8_t*>(is_k ? p.k_new : p.v_new) +
                       (tok0 * p.Hkv + r0) * (DSA_HEAD_DIM * 2);
  // stage the tile: rows * 256 bytes in 16-byte pieces
  for (int c = threadIdx.x; c < kAppRowsK * 16; c += kAppThreads) {
    const bool in = (c >> 4) < rows;
    cp_async16(tile + c * 16, in ? src + c * 16 : src, in);
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  const int grp = threadIdx.x >> 3;                  // 32 groups of 8 lanes
  const int l8 = threadIdx.x & 7;
  const bool src16 = (p.q_dtype == DSA_FP16);
  const long long drow0 = dst0 * p.Hkv + r0;         // first cache row of the tile
#pragma unroll 1
  for (int rr = grp; rr < kAppRowsK; rr += kAppThreads / 8) {
    const bool valid = rr < rows;
    const uint8_t* row = tile + rr * (DSA_HEAD_DIM * 2);
    uint4 u[2];
    u[0] = *reinterpret_cast<const uint4*>(row + l8 * 16);
    u[1] = *reinterpret_cast<const uint4*>(row + 128 + l8 * 16);
    long long drow = drow0 + rr;
    bool bad = false;
    if constexpr (PAGED) {
      if (valid) {   // (no early exit: every lane takes part in the INT8 warp vote)
        const int rs = static_cast<int>(r0) + rr;    // row within the sequence's span
        const int tok = rs / p.Hkv;
        drow = cache_row(p.pg, b, p.cap, p.lens.T[b] - p.S + tok, &bad) * p.Hkv + (rs - tok * p.Hkv);
      }
    }
    if (p.kv_dtype == DSA_INT8) {
      float x[16];
      unpack16(u, src16, x);
      float amax = 0.0f;
#pragma unroll
      for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(x[e]));
      // absmax over the group's 128 elements (xor offsets below 8 stay in
      // it; every lane of the warp takes part). Rows past the tile's end
      // were zero-filled by the copy.
#pragma unroll
      for (int off = 4; off > 0; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      const float scale = __fdiv_rn(amax, 127.0f);   // 0 for an all-zero row
      const uint4 codes = quantize16(x, scale);
      if (!valid || bad) continue;
      int8_t* dst = static_cast<int8_t*>(is_k ? p.k : p.v) + drow * DSA_HEAD_DIM;
      *reinterpret_cast<uint2*>(dst + l8 * 8) = make_uint2(codes.x, codes.y);
      *reinterpret_cast<uint2*>(dst + 64 + l8 * 8) = make_uint2(codes.z, codes.w);
      if (l8 == 0) (is_k ? p.k_scale : p.v_scale)[drow] = scale;
    } else {
      if (!valid || bad) continue;
      uint4 o0 = u[0], o1 = u[1];   // same 16-bit type: a copy
      if (p.kv_dtype != p.q_dtype) {
        o0 = convert8(o0, src16);
        o1 = convert8(o1, src16);
      }
      uint16_t* dst = static_cast<uint16_t*>(is_k ? p.k : p.v) + drow * DSA_HEAD_DIM;
      *reinterpret_cast<uint4*>(dst + l8 * 8) = o0;
      *reinterpret_cast<uint4*>(dst + 64 + l8 * 8) = o1;
    }
  }
}

}  // namespace

cudaError_t launch_cache_append(const AppendParams& p, int sms, cudaStream_t stream) {
  (void)sms;
  const long long kv_tiles = (static_cast<long long>(p.S) * p.Hkv + kAppRowsK - 1) / kAppRowsK;
  const long long kI_tiles = (static_cast<long long>(p.S) + kAppRowsI - 1) / kAppRowsI;
  const long long tiles = kv_tiles > kI_tiles ? kv_tiles : kI_tiles;
  if (tiles > 0x7fffffffll) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(tiles), 3, p.B);
  if (p.pg.table != nullptr)
    return launch_kernel("cache_append_kernel", cache_append_kernel<true>, grid, dim3(kAppThreads),
                         kAppSmem, stream, false, p);
  return launch_kernel("cache_append_kernel", cache_append_kernel<false>, grid, dim3(kAppThreads),
                       kAppSmem, stream, false, p);
}

}  // namespace dsa
