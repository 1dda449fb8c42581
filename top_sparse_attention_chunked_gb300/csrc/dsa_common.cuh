// Device helpers shared by the kernels.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace dsa {

// Order-preserving image of an fp32 score as an unsigned key: a larger float
// gives a larger key; -0.0 maps to the key of +0.0 (equal scores tie).
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Keys visible to query s of a sequence with T cache rows whose S new tokens
// are the last S rows: positions 0 .. T-S+s.
__device__ __forceinline__ int visible_len(int T, int S, int s) { return T - S + s + 1; }

// x * 2^e for e <= 0 (or -inf) without an underflowing intermediate factor:
// when 2^e itself would be subnormal, the power is split into an exact
// power-of-two scaling and a normal fractional factor, so a huge x times a
// tiny weight keeps full precision (the follow-up PR #33847 flush).
__device__ __forceinline__ float mul_exp2(float x, float e) {
  if (e >= -125.0f) return x * exp2f(e);
  if (!(e > -1.0e30f)) return 0.0f * x;   // -inf (or absurdly small): weight 0
  float n = floorf(e);
  return ldexpf(x * exp2f(e - n), static_cast<int>(n));
}

// ----------------------------------------------------------- block scans
// Exclusive prefix sum over a block of NT threads (NT multiple of 32, <= 1024).
// `warp_tot` is shared scratch of 32 words. Returns the exclusive prefix and
// writes the block total to *total.
template <int NT>
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_tot,
                                                         uint32_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[wid] = x;
  __syncthreads();
  if (wid == 0) {
    uint32_t t = (lane < NT / 32) ? warp_tot[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    warp_tot[lane] = t;   // inclusive over warps
  }
  __syncthreads();
  uint32_t base = (wid > 0) ? warp_tot[wid - 1] : 0u;
  *total = warp_tot[NT / 32 - 1];
  __syncthreads();   // warp_tot may be reused right after
  return base + x - v;
}

// Given a histogram h[0..nb) in shared memory, find the digit d such that
// (number of entries in bins above d) < need <= that number + h[d], scanning
// from the top bin down. Writes d, the count above it and h[d] to the out
// pointers (shared). Whole block must call; NT threads; nb <= 2 * 1024.
template <int NT>
__device__ __forceinline__ void find_threshold_digit(const uint32_t* h, int nb, uint32_t need,
                                                     uint32_t* warp_tot, int* d_out,
                                                     uint32_t* above_out, uint32_t* cnt_out) {
  // each thread owns a run of bins counted from the top: bins
  // nb-1-(tid*per) down to nb-(tid+1)*per
  constexpr int kMaxPer = (2048 + NT - 1) / NT;
  const int per = (nb + NT - 1) / NT;
  uint32_t local = 0;
  uint32_t hv[kMaxPer];
#pragma unroll
  for (int j = 0; j < kMaxPer; ++j) {
    int bin = nb - 1 - (static_cast<int>(threadIdx.x) * per + j);
    hv[j] = (j < per && bin >= 0) ? h[bin] : 0u;
    local += hv[j];
  }
  uint32_t total;
  uint32_t before = block_exclusive_scan<NT>(local, warp_tot, &total);
  // the thread whose run crosses `need` reports
  if (before < need && need <= before + local) {
    uint32_t acc = before;
#pragma unroll
    for (int j = 0; j < kMaxPer; ++j) {
      if (j < per && acc < need && need <= acc + hv[j]) {
        *d_out = nb - 1 - (static_cast<int>(threadIdx.x) * per + j);
        *above_out = acc;
        *cnt_out = hv[j];
      }
      acc += hv[j];
    }
  }
  __syncthreads();
}

// ----------------------------------------------------------- phase stamps
// For latency studies only, compiled with -DDSA_TRACE: a kernel keeps per CTA
// the latest %globaltimer reading at up to 16 points (DSA_TS, from any
// thread, into shared memory) and at its end thread 0 writes them to
// buf[((kid * 4096) + cta) * 16 + i], where buf is the device pointer stored
// at byte 8 of the workspace's status block (null: nothing is written).
// Nothing reaches global memory before the kernel's end, so the stamps do not
// delay its barriers. Without the define all three expand to nothing.
#ifdef DSA_TRACE
__device__ __forceinline__ unsigned long long trace_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
#define DSA_TS_DECL                                   \
  __shared__ unsigned long long dsa_ts[16];           \
  if (threadIdx.x == 0)                               \
    for (int i_ = 0; i_ < 16; ++i_) dsa_ts[i_] = 0ull
#define DSA_TS(i) atomicMax(&dsa_ts[i], ::dsa::trace_now())
#define DSA_TS_FLUSH(status, kid)                                                               \
  do {                                                                                          \
    if (threadIdx.x == 0 && (status)) {                                                         \
      unsigned long long* b_ = *reinterpret_cast<unsigned long long* const*>(                   \
          reinterpret_cast<const uint8_t*>(status) + 8);                                        \
      const unsigned c_ = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);       \
      if (b_ && c_ < 4096u)                                                                     \
        for (int i_ = 0; i_ < 16; ++i_) b_[((kid) * 4096u + c_) * 16u + i_] = dsa_ts[i_];     \
    }                                                                                           \
  } while (0)
#else
#define DSA_TS_DECL ((void)0)
#define DSA_TS(i) ((void)0)
#define DSA_TS_FLUSH(status, kid) ((void)0)
#endif

}  // namespace dsa
