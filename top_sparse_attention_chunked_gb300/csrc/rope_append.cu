// RMSNorm + rotary embedding of a step's new vectors and the cache append in
// one launch: the work that precedes the indexer in a decoding layer.
//
// Equal, bit for bit, to dsa_rmsnorm_rotary on q (q dtype, in place), qI
// (BF16, in place), k_new (into the q dtype) and kI_new (into BF16), all at
// positions T_b - S + s, followed by dsa_cache_append of the rotated kI, k and
// the given v: the same rounding sequence (rope_math.cuh), the same
// conversions, and INT8 codes rint(x / scale) from the IEEE quotient, which
// the append's reciprocal path is proven to reproduce. PR #33997 ("[CUDA]
// Support FP16 KV cache and FP16 query/key in DynamicSparseAttention<BFloat16>
// and FP32 rotary cache / FP16 output in RMSNormRotary"): Description item 1
// (RMSNormRotary in exact fp32) and its Files changed table (cache writes
// beside the attention kernels).
//
// One warp per head vector; warps walk five ranges of units in turn: q rows,
// qI rows, k rows, kI rows, v rows (D = 128 for q, k, v; 64 for qI, kI).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstdio>

#include "dsa_internal.h"
#include "rope_math.cuh"

namespace dsa {

int report_error(int status, const char* msg);   // sets dsa_last_error_string()

namespace {

constexpr int kRaWarps = 8;

struct RopeAppendParams {
  void* q;                 // [B, S, Hq, 128] q dtype, rotated in place
  void* qI;                // [B, S, 16, 64] bf16, rotated in place
  const void* k_new;       // [B, S, Hkv, 128] q dtype
  const void* kI_new;      // [B, S, 64] bf16
  const void* v_new;       // [B, S, Hkv, 128] q dtype
  void* kI;                // [B, cap, 64] bf16
  void* k;                 // [B, cap, Hkv, 128] kv dtype
  void* v;
  float* k_scale;          // [B, cap, Hkv] (INT8 only)
  float* v_scale;
  const float* g_q;        // [128]
  const float* g_k;        // [128]
  const float* g_qI;       // [64]
  const float* g_kI;       // [64]
  const void* cos;         // [max_pos, rot / 2]
  const void* sin;
  const void* cos_i;       // [max_pos, rot_i / 2]
  const void* sin_i;
  long long n_q, n_qi, n_k, n_ki, n_v;   // rows of each range
  int B, S, Hq, Hkv, cap;
  int q_dtype, kv_dtype, cos_dtype;
  int rot, rot_i, max_pos;
  // the rotary width is the head dim and the caches take vector loads (128-
  // and 64-element heads): partners one shuffle away, no per-element checks
  int full, full_i;
  float eps;
  SeqLens lens;
};

__device__ __forceinline__ float half_to_float(uint16_t u, bool fp16) {
  if (fp16) return __half2float(__ushort_as_half(u));
  return __uint_as_float(static_cast<uint32_t>(u) << 16);
}

__device__ __forceinline__ uint16_t float_to_half(float v, bool fp16) {
  if (fp16) return __half_as_ushort(__float2half_rn(v));
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

template <int E>
__device__ __forceinline__ void load_row(const void* base, long long i, uint16_t* u) {
  const uint16_t* q = static_cast<const uint16_t*>(base) + i;
  if constexpr (E == 4) {
    const uint2 w = *reinterpret_cast<const uint2*>(q);
    u[0] = w.x & 0xffffu; u[1] = w.x >> 16; u[2] = w.y & 0xffffu; u[3] = w.y >> 16;
  } else {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(q);
    u[0] = w & 0xffffu; u[1] = w >> 16;
  }
}

template <int E>
__device__ __forceinline__ void store_row(void* base, long long i, const uint16_t* u) {
  uint16_t* q = static_cast<uint16_t*>(base) + i;
  if constexpr (E == 4)
    *reinterpret_cast<uint2*>(q) = make_uint2(u[0] | (static_cast<uint32_t>(u[1]) << 16),
                                              u[2] | (static_cast<uint32_t>(u[3]) << 16));
  else
    *reinterpret_cast<uint32_t*>(q) = u[0] | (static_cast<uint32_t>(u[1]) << 16);
}

// RMSNorm + RoPE of one head vector of token `tok`; returns the E rotated
// fp32 values of this lane, before the output rounding.
template <int D>
__device__ __forceinline__ void rope_row(const RopeAppendParams& p, const void* src, bool src_f16,
                                         long long elem0, long long tok, const float* gamma, int rot,
                                         const void* cs, const void* sn, float* s_y, float* out,
                                         bool full) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int i0 = lane * E;
  uint16_t u[E];
  load_row<E>(src, elem0 + i0, u);
  float x[E], g[E], y[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    x[e] = half_to_float(u[e], src_f16);
    g[e] = __ldg(gamma + i0 + e);
  }
  rms_normalize<E, D>(x, g, p.eps, y);
  const int h = rot >> 1;
  if (full) {
    // rot = D: every element rotates; element i's partner i +- D/2 sits in
    // lane ^ 16 (D/2 / E = 16), lanes 0-15 hold the first halves, and the
    // lane's E angles are consecutive
    const int b = static_cast<int>(tok / p.S);
    const int s = static_cast<int>(tok - static_cast<long long>(b) * p.S);
    int pos = p.lens.T[b] - p.S + s;
    pos = pos < 0 ? 0 : (pos >= p.max_pos ? p.max_pos - 1 : pos);   // clamped to the cache
    const long long j0 = static_cast<long long>(pos) * h + (lane < 16 ? i0 : i0 - h);
    float c[E], sv[E];
    if (p.cos_dtype == DSA_FP32) {
      const float* cf = static_cast<const float*>(cs) + j0;
      const float* sf = static_cast<const float*>(sn) + j0;
      if constexpr (E == 4) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(cf)), bq = __ldg(reinterpret_cast<const float4*>(sf));
        c[0] = a.x; c[1] = a.y; c[2] = a.z; c[3] = a.w;
        sv[0] = bq.x; sv[1] = bq.y; sv[2] = bq.z; sv[3] = bq.w;
      } else {
        const float2 a = __ldg(reinterpret_cast<const float2*>(cf)), bq = __ldg(reinterpret_cast<const float2*>(sf));
        c[0] = a.x; c[1] = a.y;
        sv[0] = bq.x; sv[1] = bq.y;
      }
    } else {
      uint16_t cu[E], su[E];
      load_row<E>(cs, j0, cu);
      load_row<E>(sn, j0, su);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        c[e] = half_to_float(cu[e], false);
        sv[e] = half_to_float(su[e], false);
      }
    }
#pragma unroll
    for (int e = 0; e < E; ++e)
      out[e] = rope_rotate(y[e], __shfl_xor_sync(0xffffffffu, y[e], 16), c[e], sv[e], lane < 16);
    return;
  }
  if (h > 0) {
    const int b = static_cast<int>(tok / p.S);
    const int s = static_cast<int>(tok - static_cast<long long>(b) * p.S);
    int pos = p.lens.T[b] - p.S + s;
    pos = pos < 0 ? 0 : (pos >= p.max_pos ? p.max_pos - 1 : pos);   // clamped to the cache
#pragma unroll
    for (int e = 0; e < E; ++e) s_y[i0 + e] = y[e];
    __syncwarp();
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = i0 + e;
      out[e] = y[e];
      if (i < rot) {
        const long long ci = static_cast<long long>(pos) * h + (i < h ? i : i - h);
        const bool f32 = p.cos_dtype == DSA_FP32;
        const float c = f32 ? __ldg(static_cast<const float*>(cs) + ci)
                            : half_to_float(static_cast<const uint16_t*>(cs)[ci], false);
        const float sv = f32 ? __ldg(static_cast<const float*>(sn) + ci)
                             : half_to_float(static_cast<const uint16_t*>(sn)[ci], false);
        out[e] = rope_rotate(y[e], s_y[i < h ? i + h : i - h], c, sv, i < h);
      }
    }
    __syncwarp();   // partner reads done before the warp's next row writes
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) out[e] = y[e];
  }
}

// Append one 128-element K or V row (values exact in the q dtype) to cache row
// `drow` (token row * Hkv + head): a copy, a round-to-nearest conversion, or
// INT8 codes with an absmax/127 scale.
__device__ __forceinline__ void append_row(const RopeAppendParams& p, const float* xv,
                                           const uint16_t* bits, bool is_k, long long drow) {
  constexpr int E = 4;
  const int lane = threadIdx.x & 31;
  if (p.kv_dtype == DSA_INT8) {
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(xv[e]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float scale = __fdiv_rn(amax, 127.0f);
    uint32_t w = 0;
    if (scale != 0.0f) {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float c = fminf(fmaxf(rintf(__fdiv_rn(xv[e], scale)), -127.0f), 127.0f);
        w |= (static_cast<uint32_t>(static_cast<int>(c)) & 0xffu) << (8 * e);
      }
    }
    *reinterpret_cast<uint32_t*>(static_cast<int8_t*>(is_k ? p.k : p.v) + drow * DSA_HEAD_DIM + lane * E) = w;
    if (lane == 0) (is_k ? p.k_scale : p.v_scale)[drow] = scale;
  } else {
    uint16_t o[E];
#pragma unroll
    for (int e = 0; e < E; ++e)
      o[e] = p.kv_dtype == p.q_dtype ? bits[e] : float_to_half(xv[e], p.kv_dtype == DSA_FP16);
    store_row<E>(is_k ? p.k : p.v, drow * DSA_HEAD_DIM + lane * E, o);
  }
}

__global__ void __launch_bounds__(kRaWarps * 32) rope_append_kernel(const RopeAppendParams p) {
  __shared__ float s_y[kRaWarps][DSA_HEAD_DIM];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool qf16 = p.q_dtype == DSA_FP16;
  const long long total = p.n_q + p.n_qi + p.n_k + p.n_ki + p.n_v;
  for (long long u = static_cast<long long>(blockIdx.x) * kRaWarps + warp; u < total;
       u += static_cast<long long>(gridDim.x) * kRaWarps) {
    long long r = u;
    float out[4];
    if (r < p.n_q) {                                   // q: rotate in place
      rope_row<128>(p, p.q, qf16, r * DSA_HEAD_DIM, r / p.Hq, p.g_q, p.rot, p.cos, p.sin, s_y[warp], out,
                    p.full != 0);
      uint16_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) o[e] = float_to_half(out[e], qf16);
      store_row<4>(p.q, r * DSA_HEAD_DIM + lane * 4, o);
      continue;
    }
    r -= p.n_q;
    if (r < p.n_qi) {                                  // qI: rotate in place (BF16)
      rope_row<64>(p, p.qI, false, r * DSA_IDX_DIM, r / DSA_IDX_HEADS, p.g_qI, p.rot_i, p.cos_i,
                   p.sin_i, s_y[warp], out, p.full_i != 0);
      uint16_t o[2] = {float_to_half(out[0], false), float_to_half(out[1], false)};
      store_row<2>(p.qI, r * DSA_IDX_DIM + lane * 2, o);
      continue;
    }
    r -= p.n_qi;
    if (r < p.n_k + p.n_v) {                           // k: rotate, round, append; v: append
      const bool is_k = r < p.n_k;
      const long long row = is_k ? r : r - p.n_k;      // (token, head) row of k_new / v_new
      const long long tok = row / p.Hkv;
      const int g = static_cast<int>(row - tok * p.Hkv);
      const int b = static_cast<int>(tok / p.S);
      const int s = static_cast<int>(tok - static_cast<long long>(b) * p.S);
      const long long drow = (static_cast<long long>(b) * p.cap + (p.lens.T[b] - p.S + s)) * p.Hkv + g;
      uint16_t bits[4];
      float xv[4];
      if (is_k) {
        rope_row<128>(p, p.k_new, qf16, row * DSA_HEAD_DIM, tok, p.g_k, p.rot, p.cos, p.sin, s_y[warp], out,
                      p.full != 0);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          bits[e] = float_to_half(out[e], qf16);        // the rotated k in the q dtype
          xv[e] = half_to_float(bits[e], qf16);
        }
      } else {
        load_row<4>(p.v_new, row * DSA_HEAD_DIM + lane * 4, bits);
#pragma unroll
        for (int e = 0; e < 4; ++e) xv[e] = half_to_float(bits[e], qf16);
      }
      append_row(p, xv, bits, is_k, drow);
      continue;
    }
    r -= p.n_k + p.n_v;                                // kI: rotate (BF16), append
    {
      const long long tok = r;
      const int b = static_cast<int>(tok / p.S);
      const int s = static_cast<int>(tok - static_cast<long long>(b) * p.S);
      rope_row<64>(p, p.kI_new, false, tok * DSA_IDX_DIM, tok, p.g_kI, p.rot_i, p.cos_i, p.sin_i,
                   s_y[warp], out, p.full_i != 0);
      uint16_t o[2] = {float_to_half(out[0], false), float_to_half(out[1], false)};
      const long long dst = (static_cast<long long>(b) * p.cap + (p.lens.T[b] - p.S + s)) * DSA_IDX_DIM;
      store_row<2>(p.kI, dst + lane * 2, o);
    }
  }
}

bool aligned_to(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

}  // namespace

int problem_check_for_append(const dsa_problem* p);   // dsa_api.cu: validates as for prefill

}  // namespace dsa

using namespace dsa;

extern "C" int dsa_rope_append(const dsa_problem* p, const dsa_rope_params* rp, void* q, void* qI,
                               const void* k_new, const void* kI_new, const void* v_new, void* kI,
                               void* k, void* v, float* k_scale, float* v_scale, void* stream) {
  reset_launches();
  int rc = problem_check_for_append(p);
  if (rc) return rc;
  if (!rp) return report_error(DSA_ERR_INVALID_ARG, "rope parameters are NULL");
  if (rp->rotary_dim < 0 || rp->rotary_dim > DSA_HEAD_DIM || (rp->rotary_dim & 1) ||
      rp->rotary_dim_index < 0 || rp->rotary_dim_index > DSA_IDX_DIM || (rp->rotary_dim_index & 1))
    return report_error(DSA_ERR_INVALID_ARG, "rotary widths must be even, at most 128 (q, k) and 64 (qI, kI)");
  const bool any_rot = rp->rotary_dim > 0 || rp->rotary_dim_index > 0;
  if (any_rot && rp->max_pos < 1) return report_error(DSA_ERR_INVALID_ARG, "max_pos must be >= 1");
  if (any_rot && rp->cos_dtype != DSA_FP32 && rp->cos_dtype != DSA_BF16)
    return report_error(DSA_ERR_UNSUPPORTED, "the cos / sin caches must be FP32 or BF16");
  if (!(rp->eps >= 0.0f) || std::isinf(rp->eps)) return report_error(DSA_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (!rp->gamma_q || !rp->gamma_k || !rp->gamma_qI || !rp->gamma_kI)
    return report_error(DSA_ERR_INVALID_ARG, "the four gamma vectors are required");
  if ((rp->rotary_dim > 0 && (!rp->cos || !rp->sin)) ||
      (rp->rotary_dim_index > 0 && (!rp->cos_index || !rp->sin_index)))
    return report_error(DSA_ERR_INVALID_ARG, "a rotary width > 0 needs its cos / sin caches");
  if (!q || !qI || !k_new || !kI_new || !v_new || !kI || !k || !v)
    return report_error(DSA_ERR_INVALID_ARG, "a required tensor pointer is NULL");
  const bool int8 = p->kv_dtype == DSA_INT8;
  if (int8 != (k_scale != nullptr) || int8 != (v_scale != nullptr))
    return report_error(DSA_ERR_INVALID_ARG, "k_scale / v_scale are required iff the cache is INT8");
  const size_t ca = rp->cos_dtype == DSA_FP32 ? 4 : 2;
  if (!aligned_to(q, 16) || !aligned_to(qI, 16) || !aligned_to(k_new, 16) || !aligned_to(kI_new, 16) ||
      !aligned_to(v_new, 16) || !aligned_to(kI, 16) || !aligned_to(k, 16) || !aligned_to(v, 16) ||
      (int8 && (!aligned_to(k_scale, 4) || !aligned_to(v_scale, 4))) ||
      !aligned_to(rp->gamma_q, 4) || !aligned_to(rp->gamma_k, 4) || !aligned_to(rp->gamma_qI, 4) ||
      !aligned_to(rp->gamma_kI, 4) ||
      (rp->rotary_dim > 0 && (!aligned_to(rp->cos, ca) || !aligned_to(rp->sin, ca))) ||
      (rp->rotary_dim_index > 0 && (!aligned_to(rp->cos_index, ca) || !aligned_to(rp->sin_index, ca))))
    return report_error(DSA_ERR_MISALIGNED, "tensors must be 16-byte aligned; gamma, scales and caches element-aligned");
  // the new vectors are read while the caches are written: no overlap
  const long long B = p->batch, S = p->q_len, H = p->num_kv_heads, cap = p->cache_capacity;
  const long long row_bytes = int8 ? DSA_HEAD_DIM : DSA_HEAD_DIM * 2;
  struct Span { const void* ptr; long long n; };
  const Span in[5] = {{q, B * S * p->num_q_heads * DSA_HEAD_DIM * 2}, {qI, B * S * 16 * DSA_IDX_DIM * 2},
                      {k_new, B * S * H * DSA_HEAD_DIM * 2}, {kI_new, B * S * DSA_IDX_DIM * 2},
                      {v_new, B * S * H * DSA_HEAD_DIM * 2}};
  const Span out[5] = {{kI, B * cap * DSA_IDX_DIM * 2}, {k, B * cap * H * row_bytes},
                       {v, B * cap * H * row_bytes}, {k_scale, int8 ? B * cap * H * 4 : 0},
                       {v_scale, int8 ? B * cap * H * 4 : 0}};
  for (const Span& a : in)
    for (const Span& o : out) {
      const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.ptr), o0 = reinterpret_cast<uintptr_t>(o.ptr);
      if (o.n > 0 && a0 < o0 + static_cast<uintptr_t>(o.n) && o0 < a0 + static_cast<uintptr_t>(a.n))
        return report_error(DSA_ERR_INVALID_ARG, "a new-token tensor overlaps a cache");
    }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
    cudaGetLastError();
    return report_error(DSA_ERR_NO_DEVICE, "no usable CUDA device");
  }
  RopeAppendParams a;
  a.q = q;
  a.qI = qI;
  a.k_new = k_new;
  a.kI_new = kI_new;
  a.v_new = v_new;
  a.kI = kI;
  a.k = k;
  a.v = v;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.g_q = rp->gamma_q;
  a.g_k = rp->gamma_k;
  a.g_qI = rp->gamma_qI;
  a.g_kI = rp->gamma_kI;
  a.cos = rp->cos;
  a.sin = rp->sin;
  a.cos_i = rp->cos_index;
  a.sin_i = rp->sin_index;
  a.n_q = B * S * p->num_q_heads;
  a.n_qi = B * S * DSA_IDX_HEADS;
  a.n_k = B * S * H;
  a.n_v = B * S * H;
  a.n_ki = B * S;
  a.B = p->batch;
  a.S = p->q_len;
  a.Hq = p->num_q_heads;
  a.Hkv = p->num_kv_heads;
  a.cap = p->cache_capacity;
  a.q_dtype = p->q_dtype;
  a.kv_dtype = p->kv_dtype;
  a.cos_dtype = rp->cos_dtype;
  a.rot = rp->rotary_dim;
  a.rot_i = rp->rotary_dim_index;
  {
    // vector loads of a lane's E consecutive angles need the caches aligned
    // to E elements (the row starts then stay aligned)
    const size_t es = rp->cos_dtype == DSA_FP32 ? 4 : 2;
    auto al = [](const void* ptr, size_t n) { return (reinterpret_cast<uintptr_t>(ptr) % n) == 0; };
    a.full = rp->rotary_dim == DSA_HEAD_DIM && al(rp->cos, 4 * es) && al(rp->sin, 4 * es);
    a.full_i = rp->rotary_dim_index == DSA_IDX_DIM && al(rp->cos_index, 2 * es) && al(rp->sin_index, 2 * es);
  }
  a.max_pos = rp->max_pos;
  a.eps = rp->eps;
  for (int b = 0; b < p->batch; ++b) a.lens.T[b] = p->total_len[b];
  const long long units = a.n_q + a.n_qi + a.n_k + a.n_v + a.n_ki;
  long long blocks = (units + kRaWarps - 1) / kRaWarps;
  const long long most = static_cast<long long>(sms) * 64;
  if (blocks > most) blocks = most;
  const cudaError_t e = launch_kernel("rope_append_kernel", rope_append_kernel,
                                      dim3(static_cast<unsigned>(blocks)), dim3(kRaWarps * 32), 0,
                                      static_cast<cudaStream_t>(stream), false, a);
  if (e != cudaSuccess) {
    char buf[160];
    snprintf(buf, sizeof(buf), "rope_append launch: %s", cudaGetErrorString(e));
    return report_error(DSA_ERR_CUDA, buf);
  }
  return DSA_OK;
}
