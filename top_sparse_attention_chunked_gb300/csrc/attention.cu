// Sparse GQA attention over the selected K/V rows, split over the selected
// keys, with an online-softmax combine.
//
// PR #33997 "[CUDA] Support FP16 KV cache and FP16 query/key in
// DynamicSparseAttention<BFloat16> ...", Description item 2: a grouped decode
// kernel processes the query heads of one KV head together over the selected
// rows (the pages' test is a group ratio of 12) and a tensor-core prefill kernel
// with FP16 operands (mma m16n8k16 f32.f16.f16.f32) for BF16 activations with
// an FP16 cache. PR #33802 Summary item 1: INT8 cache with split-K decode.
// Follow-up PR #33847: rescaling the PV accumulator by exp2(old_max - new_max)
// must not flush the earlier tiles to zero when the max rises by ~88 nats.
//
// Layout of the work: one CTA per (split of the selected keys, KV head x group
// of <= 16 query heads, query row). The group's query heads form the M = 16
// rows of warp-level m16n8k16 MMAs; each warp gathers 16 selected rows of K
// and V per tile into a double buffer -- TMA row gathers (tile::gather4,
// four rows per instruction, 128-byte swizzle applied by the copy engine) for
// a 16-bit cache, 16-byte cp.async for INT8 codes -- computes
// S = Q K^T (16 heads x 16 keys), the online softmax in registers, and
// O += P V. Warps, then splits, are merged with an LSE combine whose scaling
// never forms a subnormal factor (mul_exp2).
//
// Precision: QK^T uses the cache's 16-bit type (a BF16 query is converted to
// FP16 for an FP16 cache, as the pages' MmaFp16 path does); the probabilities
// enter PV as FP16 for an FP16 cache and as a BF16 hi+lo pair otherwise, so
// P keeps 16 significant bits. INT8 codes are exact in BF16/FP16; k_scale
// multiplies the logit after the dot product and v_scale is folded into P.
#include <cooperative_groups.h>
#include <mutex>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dsa_common.cuh"
#include "dsa_internal.h"
#include "sm100_ptx.cuh"

namespace dsa {

constexpr int kAttnThreads = 128;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kTileKeys = 16;
constexpr int kD = DSA_HEAD_DIM;
constexpr int kTile16 = kTileKeys * kD * 2;      // 4 KB: one 16-key tile, 16-bit
constexpr int kTile8 = kTileKeys * kD;           // 2 KB: one 16-key tile, INT8
// Per-warp shared memory, every tile 1024-byte aligned (the swizzle of the
// row gathers follows the address bits). 16-bit caches: K stage 0/1, V stage
// 0/1 (4 x 4 KB). INT8: converted K and V tiles (2 x 4 KB), code staging K
// 0/1, V 0/1 (4 x 2 KB). The INT8 scales sit in static shared memory. Three
// CTAs fit on an SM.
constexpr int kWarpSmem = 4 * kTile16;
// the split combine merges up to kAttnMaxSplits partial states
constexpr int kMaxCombine = kAttnMaxSplits;
// per-warp partial state in shared memory: m[16], l[16], o[16][kORow] (rows
// padded to 136 floats so the fragment stores of a half-warp hit distinct banks)
constexpr int kORow = DSA_HEAD_DIM + 8;
constexpr int kWarpState = 2 * kAttnRows + kAttnRows * kORow;
// (one more state than warps: the auxiliary keys' own, when there are any)
constexpr int kMergeFloats = (kAttnWarps + 1) * kWarpState + 2 * kMaxCombine * kAttnRows + 2 * kAttnRows;
constexpr int kStageBytes = (kAttnWarps * kWarpSmem > kMergeFloats * 4) ? kAttnWarps * kWarpSmem
                                                                       : kMergeFloats * 4;
// Cluster combine: every CTA receives from each peer q its M, L (32 floats at
// q * 32) and, for the output columns this CTA owns, q's unnormalised rows
// (column-major, 16 rows per column, at 512 + (q * cols + c) * 16): at most
// 16 * 32 + 2,048 floats, written by the peers with st.async while this CTA
// may still be gathering, so it has its own region.
constexpr int kRecvFloats = 16 * 2 * kAttnRows + kAttnRows * DSA_HEAD_DIM;
// dynamic shared memory (+ slack to align the base): the stage buffers, and
// in a cluster the receive area after them (outside a cluster three CTAs fit
// on an SM, in one two)
constexpr int kAttnSmem = kStageBytes + 1024;
constexpr int kAttnSmemCluster = kStageBytes + kRecvFloats * 4 + 1024;

enum { KV_BF16 = 0, KV_FP16 = 1, KV_INT8 = 2 };

// 16-bit K/V rows are gathered with 16-byte cp.async (each warp instruction
// moves two whole 256-byte rows) unless built with DSA_ATTN_TMA_GATHER, which
// selects TMA tile::gather4 row gathers.
#ifdef DSA_ATTN_TMA_GATHER
constexpr bool kTmaGather16 = true;
#else
constexpr bool kTmaGather16 = false;
#endif

// Byte offset of 16-byte chunk c (0..15) of row r in a 16-row 16-bit tile:
// two 64-column blocks of 16 x 128 B, chunk positions XOR-swizzled by the row
// within each 128-byte row (the layout a 128-byte-swizzled TMA copy writes).
__device__ __forceinline__ int swz(int r, int c) {
  return ((c >> 3) << 11) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// Bounded wait used on the unwinding path: ignores the abort flag.
__device__ __forceinline__ void mbar_drain_attn(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kWaitBudgetCycles) return;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <bool F16>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
  if constexpr (F16) return pack_f16(lo, hi);
  else return pack_bf16(lo, hi);
}

// Load 2 consecutive query elements as the MMA operand type.
template <bool Q_F16, bool OP_F16>
__device__ __forceinline__ uint32_t load_q2(const void* q, size_t elem) {
  const uint32_t raw = *reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(q) + elem);
  if constexpr (Q_F16 == OP_F16) {
    return raw;
  } else if constexpr (Q_F16) {   // fp16 query, bf16 operand (INT8 cache only)
    __half2 h = *reinterpret_cast<const __half2*>(&raw);
    float2 f = __half22float2(h);
    return pack_bf16(f.x, f.y);
  } else {                        // bf16 query, fp16 operand
    __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&raw);
    float2 f = __bfloat1622float2(h);
    return pack_f16(f.x, f.y);
  }
}

// Query-dtype (BF16 or FP16) values as fp32: two consecutive, or one.
template <bool F16>
__device__ __forceinline__ float2 load_f2(const void* base, size_t elem) {
  const uint32_t raw = *reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(base) + elem);
  if constexpr (F16) return __half22float2(*reinterpret_cast<const __half2*>(&raw));
  else return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw));
}
template <bool F16>
__device__ __forceinline__ float load_f1(const void* base, size_t elem) {
  const uint16_t raw = static_cast<const uint16_t*>(base)[elem];
  if constexpr (F16) return __half2float(*reinterpret_cast<const __half*>(&raw));
  else return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(&raw));
}

// Exact float value of the signed byte `i` of `x`: the byte plus 128 lands in
// the low mantissa bits of 2^23 (a byte permute), and subtracting 2^23 + 128
// leaves the code. Two plain ALU operations, no int-to-float conversion.
__device__ __forceinline__ float code_to_float(uint32_t x_biased, int i) {
  return __uint_as_float(__byte_perm(x_biased, 0x4B000000u, 0x7540u | static_cast<uint32_t>(i))) -
         8388736.0f;
}

// 16 INT8 codes -> 16 exact 16-bit values written as two swizzled chunks
template <bool F16>
__device__ __forceinline__ void convert_codes16(const uint4 src, uint8_t* tile, int row, int c0) {
  const uint32_t wsrc[4] = {src.x ^ 0x80808080u, src.y ^ 0x80808080u, src.z ^ 0x80808080u,
                            src.w ^ 0x80808080u};
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w[i] = pack16<F16>(code_to_float(wsrc[i >> 1], (2 * i) & 3), code_to_float(wsrc[i >> 1], (2 * i + 1) & 3));
  *reinterpret_cast<uint4*>(tile + swz(row, c0)) = make_uint4(w[0], w[1], w[2], w[3]);
  *reinterpret_cast<uint4*>(tile + swz(row, c0 + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
}

template <int OUT>
__device__ __forceinline__ void store_out(void* out, size_t i, float v) {
  if constexpr (OUT == DSA_BF16) static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
  else if constexpr (OUT == DSA_FP16) static_cast<__half*>(out)[i] = __float2half_rn(v);
  else static_cast<float*>(out)[i] = v;
}

// x * 2^e == (x * f1) * f2 with both factors formed without underflow where
// it matters: f1 = 2^max(e, -120) is normal, f2 = 2^(e - max(e, -120)) is 1
// unless e < -120. A state that saw no keys (m = -inf) gets weight 0.
__device__ __forceinline__ void exp2_pair(float e, float* f1, float* f2) {
  if (!(e > -1.0e30f)) {
    *f1 = 0.0f;
    *f2 = 0.0f;
    return;
  }
  const float a = fmaxf(e, -120.0f);
  *f1 = exp2f(a);
  *f2 = exp2f(e - a);
}

// Thread `row` (< 16) merges `n` online-softmax states whose m / l live at
// st[j * stride + row] / st[j * stride + 16 + row]: writes the factors that
// bring state j to the common max and the merged M, L.
__device__ __forceinline__ void combine_factors(const float* st, int stride, int n, float* fac1,
                                                float* fac2, float* sML) {
  const int row = threadIdx.x;
  float M = -INFINITY;
  for (int j = 0; j < n; ++j) M = fmaxf(M, st[j * stride + row]);
  float L = 0.0f;
  for (int j = 0; j < n; ++j) {
    float f1, f2;
    exp2_pair(st[j * stride + row] - M, &f1, &f2);
    fac1[j * kAttnRows + row] = f1;
    fac2[j * kAttnRows + row] = f2;
    L += st[j * stride + kAttnRows + row] * f1 * f2;
  }
  sML[row] = M;
  sML[kAttnRows + row] = L;
}

// tm_k / tm_v view the caches as [B * cap * Hkv rows, 128] (16-bit: box 64 x 1;
// INT8: box 128 x 1), 128-byte swizzle; row (b * cap + key) * Hkv + g.
template <int KV, bool Q_F16, int OUT>
__global__ void __launch_bounds__(kAttnThreads) sparse_attn_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                   const __grid_constant__ CUtensorMap tm_v,
                                                                   const AttnParams p) {
  constexpr bool QK_F16 = (KV == KV_FP16) || (KV == KV_INT8 && Q_F16);
  constexpr bool PV_F16 = (KV == KV_FP16);
  constexpr bool PV_SPLIT = !PV_F16;   // BF16 P as hi + lo
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ int s_last;
  __shared__ int32_t s_idx[kAttnMaxSplitKeys];
  __shared__ uint64_t s_bar[kAttnWarps][2];     // per warp and stage: the tile's rows landed
  __shared__ int s_abort;
  __shared__ float s_sc[kAttnWarps][64];        // INT8: [stage][k 16 | v 16] scales per warp
  __shared__ uint64_t s_merge_bar;              // cluster combine: every peer's slice landed
  __shared__ float s_auxp[kAttnRows][kAttnRows];  // auxiliary keys: logits, then weights

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  DSA_TS_DECL;
  if (threadIdx.x == 0) DSA_TS(0);
  const int gq = lane >> 2, tq = lane & 3;   // MMA fragment coordinates
  const int r = blockIdx.z;                  // query row = b * S + s
  const int b = r / p.S, s = r % p.S;
  const int gh = blockIdx.y;                 // KV head x head group
  const int g = gh / p.HG, hg = gh % p.HG;
  const int h0 = g * p.G + hg * kAttnRows;
  const int nh = min(kAttnRows, p.G - hg * kAttnRows);
  const int T = p.lens.T[b];
  const int keff = min(p.topk, visible_len(T, p.S, s));
  const int split_begin = blockIdx.x * p.split_keys;
  // in a cluster every split takes part in the combine, empty or not
  if (split_begin >= keff && !p.cluster) return;
  const int split_len = max(0, min(p.split_keys, keff - split_begin));
  // keys of this split read from the cache; with auxiliary K/V the split's
  // keys at or after the first new token (its tail: the indices ascend) are
  // attended separately from the auxiliary rows, after the tile loop
  int split_main = split_len;
  const int nreal = (keff + p.split_keys - 1) / p.split_keys;
  int ntiles = (split_len + kTileKeys - 1) / kTileKeys;

  uint8_t* wsm = smem + warp * kWarpSmem;
  uint8_t* sK[2] = {wsm, wsm + kTile16};
  uint8_t* sV[2] = {wsm + 2 * kTile16, wsm + 3 * kTile16};
  // INT8 only: converted tiles live in sK[0] / sK[1]'s space, staging after
  uint8_t* sKc[2] = {wsm + 2 * kTile16, wsm + 2 * kTile16 + kTile8};
  uint8_t* sVc[2] = {wsm + 3 * kTile16, wsm + 3 * kTile16 + kTile8};
  float* sSc = s_sc[warp];
  if (lane == 0) {
    mbar_init(&s_bar[warp][0], 1);
    mbar_init(&s_bar[warp][1], 1);
    fence_mbar_init();
  }
  if (threadIdx.x == 0) s_abort = 0;
  float* recv = reinterpret_cast<float*>(smem + kStageBytes);
  if (p.cluster) {
    // the combine's receive barrier expects every peer's M, L and column
    // slice; peers push into it only after the cluster barrier below, which
    // every CTA arrives at once its barrier is armed
    if (threadIdx.x == 0) {
      mbar_init(&s_merge_bar, 1);
      fence_mbar_init();
      mbar_arrive_expect_tx(&s_merge_bar,
                            static_cast<uint32_t>((p.nsplit * 2 * kAttnRows + kAttnRows * kD) * 4));
    }
    cluster_arrive();
  }

  const int32_t* idx_row = p.idx + static_cast<size_t>(r) * p.topk + split_begin;
  bool bad_page = false;   // a gathered key's block-table entry lay outside the pool

  // gather the 16 selected rows of tile `it` (this warp's it-th tile) into
  // stage st: lane l < 16 holds key l's row; rows past the split (and any
  // index outside the visible cache) read key 0, whose logits are masked
  auto issue_tile = [&](int it, int st) {
    const int tile = warp + it * kAttnWarps;
    const int o = tile * kTileKeys;
    int key = -1;
    if (lane < kTileKeys && o + lane < split_main) {
      key = s_idx[o + lane];
      if (key < 0 || key >= T) key = -1;
    }
    // the key's cache row (key 0's for invalid keys, whose logits are masked)
    const long long crow = cache_row(p.pg, b, p.cap, key < 0 ? 0 : key, &bad_page);
    // the K / V row (128 values) of this key and KV head
    long long kvr = p.pg.table ? crow * p.Hkv + g
                               : b * p.kv_sb + static_cast<long long>(key < 0 ? 0 : key) * p.kv_st +
                                     g * p.kv_sh;
    if (!bounds_ok(kvr >= 0 && kvr < p.kv_rows && crow * p.Hkv + g < p.scale_rows, p.status)) {
      kvr = 0;     // read row 0 and mask the key
      key = -1;
    }
    if constexpr (KV == KV_INT8) {
      // INT8 rows (128 B): 16-byte cp.async measured faster here than row
      // gathers; codes and scales land zero-filled for invalid keys
      const int8_t* kb = static_cast<const int8_t*>(p.k);
      const int8_t* vb = static_cast<const int8_t*>(p.v);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int j = lane + 32 * i;            // 0..127: row j/8, chunk j%8
        const int row = j >> 3, c = j & 7;
        const int kr = __shfl_sync(0xffffffffu, key, row);
        const long long kr2 = __shfl_sync(0xffffffffu, kvr, row);
        const size_t off = static_cast<size_t>(kr2) * kD + c * 16;
        cp_async16(sKc[st] + row * kD + c * 16, kb + off, kr >= 0);
        cp_async16(sVc[st] + row * kD + c * 16, vb + off, kr >= 0);
      }
      const int kr = __shfl_sync(0xffffffffu, key, lane & 15);
      const long long cr = __shfl_sync(0xffffffffu, crow, lane & 15);
      const size_t so = static_cast<size_t>(cr) * p.Hkv + g;
      if (lane < 16) cp_async4(sSc + st * 32 + lane, p.k_scale + so, kr >= 0);
      else cp_async4(sSc + st * 32 + lane, p.v_scale + so, kr >= 0);
    } else if constexpr (!kTmaGather16) {
      // 16-bit rows (256 B): lanes 0-15 copy chunk `lane` of row 2i, lanes
      // 16-31 of row 2i + 1, into the swizzled layout ldmatrix reads; invalid
      // keys land as zeros (their logits are masked)
      const uint8_t* kb = static_cast<const uint8_t*>(p.k);
      const uint8_t* vb = static_cast<const uint8_t*>(p.v);
      const int c = lane & 15;
#pragma unroll
      for (int i = 0; i < kTileKeys / 2; ++i) {
        const int row = 2 * i + (lane >> 4);
        const int kr = __shfl_sync(0xffffffffu, key, row);
        const long long kr2 = __shfl_sync(0xffffffffu, kvr, row);
        const size_t off = (static_cast<size_t>(kr2) * kD) * 2 + c * 16;
        cp_async16(sK[st] + swz(row, c), kb + off, kr >= 0);
        cp_async16(sV[st] + swz(row, c), vb + off, kr >= 0);
      }
    } else {
      // 16-bit rows (256 B): TMA row gathers, lane l of the first 16 issuing
      // one for 4 rows (grp) of one column block (blk) of K or V (tsr)
      const int yrow = static_cast<int>(kvr);
      const int grp = lane & 3, blk = (lane >> 2) & 1, tsr = lane >> 3;
      const int y0 = __shfl_sync(0xffffffffu, yrow, 4 * grp);
      const int y1 = __shfl_sync(0xffffffffu, yrow, 4 * grp + 1);
      const int y2 = __shfl_sync(0xffffffffu, yrow, 4 * grp + 2);
      const int y3 = __shfl_sync(0xffffffffu, yrow, 4 * grp + 3);
      if (lane == 0) mbar_arrive_expect_tx(&s_bar[warp][st], 2 * kTile16);
      __syncwarp();
      if (lane < 16)
        tma_gather4((tsr ? sV[st] : sK[st]) + blk * 2048 + grp * 512,
                    tsr ? static_cast<const void*>(&tm_v) : static_cast<const void*>(&tm_k),
                    &s_bar[warp][st], blk * 64, y0, y1, y2, y3);
    }
  };

  float o_acc[kD / 8][4];
#pragma unroll
  for (int i = 0; i < kD / 8; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.0f;
  float m_run[2] = {-INFINITY, -INFINITY};   // rows gq, gq+8 (log2 units)
  float l_run[2] = {0.0f, 0.0f};             // thread-partial sums

  int my_tiles = ntiles > warp ? (ntiles - warp + kAttnWarps - 1) / kAttnWarps : 0;
  // ---- query fragments (A operand of QK^T), resident for the whole CTA
  uint32_t qa[kD / 16][4];
  {
    const size_t qrow0 = (static_cast<size_t>(r) * p.Hq + h0 + gq) * kD;
    const size_t qrow1 = qrow0 + 8 * kD;
    const bool ok0 = gq < nh, ok1 = gq + 8 < nh;
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      const int c = kk * 16 + 2 * tq;
      qa[kk][0] = ok0 ? load_q2<Q_F16, QK_F16>(p.q, qrow0 + c) : 0u;
      qa[kk][1] = ok1 ? load_q2<Q_F16, QK_F16>(p.q, qrow1 + c) : 0u;
      qa[kk][2] = ok0 ? load_q2<Q_F16, QK_F16>(p.q, qrow0 + c + 8) : 0u;
      qa[kk][3] = ok1 ? load_q2<Q_F16, QK_F16>(p.q, qrow1 + c + 8) : 0u;
    }
  }
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  pdl_wait();       // the selected indices come from the previous kernel
  if (threadIdx.x == 0) DSA_TS(1);
  pdl_trigger();
  // the split's selected indices, loaded once (all loads in flight together)
  for (int i = threadIdx.x; i < split_len; i += kAttnThreads) s_idx[i] = __ldcg(idx_row + i);
  __syncthreads();
  const int past = T - p.S;                   // the sequence's first new token
  if (p.k_aux != nullptr) {
    // the split's keys below `past` (s_idx ascends): a binary search
    int lo = 0, hi = split_len;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s_idx[mid] < past) lo = mid + 1;
      else hi = mid;
    }
    split_main = lo;
    ntiles = (split_main + kTileKeys - 1) / kTileKeys;
    my_tiles = ntiles > warp ? (ntiles - warp + kAttnWarps - 1) / kAttnWarps : 0;
  }
  const int naux = split_len - split_main;    // the same in every thread
  if (threadIdx.x == 0) DSA_TS(2);
  if (my_tiles > 0) issue_tile(0, 0);
  cp_async_commit();
  int issued = my_tiles > 0 ? 1 : 0, landed = 0;

  for (int it = 0; it < my_tiles; ++it) {
    const int st = it & 1;
    if (it + 1 < my_tiles) {
      issue_tile(it + 1, st ^ 1);
      ++issued;
    }
    cp_async_commit();
    cp_async_wait<1>();   // cp.async tiles
    if constexpr (KV != KV_INT8 && kTmaGather16) {
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&s_bar[warp][st],
                                                      static_cast<uint32_t>((it >> 1) & 1), &s_abort)))
        break;
    }
    landed = it + 1;
    if (it == 0 && lane == 0) DSA_TS(3);
    __syncwarp();
    const int tile = warp + it * kAttnWarps;
    const int nvalid = min(kTileKeys, split_main - tile * kTileKeys);

    const uint8_t* tK = sK[st];
    const uint8_t* tV = sV[st];
    if constexpr (KV == KV_INT8) {
      // codes -> exact 16-bit values in the swizzled layout ldmatrix expects
      const int row = lane >> 1, half = lane & 1;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = half * 4 + i;             // 16-code chunk of the row
        const uint4 kc = *reinterpret_cast<const uint4*>(sKc[st] + row * kD + c * 16);
        const uint4 vc = *reinterpret_cast<const uint4*>(sVc[st] + row * kD + c * 16);
        convert_codes16<QK_F16>(kc, sK[0], row, 2 * c);
        convert_codes16<false>(vc, sK[1], row, 2 * c);
      }
      __syncwarp();
      tK = sK[0];
      tV = sK[1];
    }

    // ---- S = Q K^T : 16 heads x 16 keys
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int mi = lane >> 3;
      const int krow = ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) {
        uint32_t bk[4];
        ldmatrix_x4(bk, tK + swz(krow, 2 * kk + (mi & 1)));
        mma_16816<QK_F16>(sc[0], qa[kk], bk);
        mma_16816<QK_F16>(sc[1], qa[kk], bk + 2);
      }
    }

    // ---- online softmax (log2 domain)
    float kscale[2][2], vscale[2][2];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int kl = 8 * n + 2 * tq + e;
        if constexpr (KV == KV_INT8) {
          kscale[n][e] = sSc[st * 32 + kl];
          vscale[n][e] = sSc[st * 32 + 16 + kl];
        } else {
          kscale[n][e] = 1.0f;
          vscale[n][e] = 1.0f;
        }
      }
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int kl = 8 * n + 2 * tq + (e & 1);
        float v = sc[n][e] * kscale[n][e & 1] * p.scale_log2;
        if (kl >= nvalid) v = -INFINITY;
        sc[n][e] = v;
        mx[e >> 1] = fmaxf(mx[e >> 1], v);
      }
    float m_new[2], d_old[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
      m_new[i] = fmaxf(m_run[i], mx[i]);
      d_old[i] = m_run[i] - m_new[i];   // <= 0; NaN/-inf when nothing was accumulated
    }
    float pt[2][4];
    float tile_sum[2] = {0.0f, 0.0f};
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float dlt = sc[n][e] - m_new[e >> 1];
        float pv = 0.0f, ptv = 0.0f;
        if (sc[n][e] != -INFINITY) {
          pv = exp2f(dlt);
          if constexpr (KV == KV_INT8) ptv = mul_exp2(vscale[n][e & 1], dlt);
          else ptv = pv;
        }
        tile_sum[e >> 1] += pv;
        pt[n][e] = ptv;
      }
    // rescale the running state to the new max: x * 2^d_old as (x * a1) * a2
    // with both factors formed without underflow (exp2_pair)
    float a1[2], a2[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      exp2_pair(d_old[i], &a1[i], &a2[i]);
      l_run[i] = l_run[i] * a1[i] * a2[i] + tile_sum[i];
      m_run[i] = m_new[i];
    }
#pragma unroll
    for (int nd = 0; nd < kD / 8; ++nd)
#pragma unroll
      for (int e = 0; e < 4; ++e) o_acc[nd][e] = o_acc[nd][e] * a1[e >> 1] * a2[e >> 1];

    // ---- O += P V
    uint32_t pa[4], pl[4];
    if constexpr (PV_F16) {
      pa[0] = pack_f16(pt[0][0], pt[0][1]);
      pa[1] = pack_f16(pt[0][2], pt[0][3]);
      pa[2] = pack_f16(pt[1][0], pt[1][1]);
      pa[3] = pack_f16(pt[1][2], pt[1][3]);
    } else {
      float hi[2][4], lo[2][4];
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          hi[n][e] = __bfloat162float(__float2bfloat16_rn(pt[n][e]));
          lo[n][e] = pt[n][e] - hi[n][e];
        }
      pa[0] = pack_bf16(hi[0][0], hi[0][1]);
      pa[1] = pack_bf16(hi[0][2], hi[0][3]);
      pa[2] = pack_bf16(hi[1][0], hi[1][1]);
      pa[3] = pack_bf16(hi[1][2], hi[1][3]);
      pl[0] = pack_bf16(lo[0][0], lo[0][1]);
      pl[1] = pack_bf16(lo[0][2], lo[0][3]);
      pl[2] = pack_bf16(lo[1][0], lo[1][1]);
      pl[3] = pack_bf16(lo[1][2], lo[1][3]);
    }
    {
      const int mi = lane >> 3;
      const int vrow = ((mi & 1) << 3) + (lane & 7);
#pragma unroll
      for (int nd = 0; nd < kD / 8; nd += 2) {
        uint32_t bv[4];
        ldmatrix_x4_trans(bv, tV + swz(vrow, nd + (mi >> 1)));
        mma_16816<PV_F16>(o_acc[nd], pa, bv);
        mma_16816<PV_F16>(o_acc[nd + 1], pa, bv + 2);
        if constexpr (PV_SPLIT) {
          mma_16816<PV_F16>(o_acc[nd], pl, bv);
          mma_16816<PV_F16>(o_acc[nd + 1], pl, bv + 2);
        }
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();
  // after a wait that gave up, let this warp's copies land before the
  // buffers are reused
  if (KV != KV_INT8 && kTmaGather16 && landed < issued && lane == 0)
    for (int t = landed; t < issued; ++t)
      mbar_drain_attn(&s_bar[warp][t & 1], static_cast<uint32_t>((t >> 1) & 1));

  if (lane == 0) DSA_TS(4);
  // ---- merge the warps of this CTA
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], 1);
    l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], 2);
  }
  __syncthreads();   // stage buffers become the merge area
  if (threadIdx.x == 0 && s_abort && p.status) atomicOr(p.status, kDevTimeout);
  if (__any_sync(0xffffffffu, bad_page) && lane == 0 && p.status) atomicOr(p.status, kDevBadPage);
  float* ws = reinterpret_cast<float*>(smem);      // [warps + 1][kWarpState]
  float* fac1 = ws + (kAttnWarps + 1) * kWarpState;  // [max(warps + 1, splits)][16]
  float* fac2 = fac1 + kMaxCombine * kAttnRows;
  float* sML = fac2 + kMaxCombine * kAttnRows;     // M[16], L[16]
  float* mine = ws + warp * kWarpState;
  if (tq == 0) {
    mine[gq] = m_run[0];
    mine[gq + 8] = m_run[1];
    mine[kAttnRows + gq] = l_run[0];
    mine[kAttnRows + gq + 8] = l_run[1];
  }
#pragma unroll
  for (int nd = 0; nd < kD / 8; ++nd)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = gq + 8 * h, col = nd * 8 + 2 * tq;
      *reinterpret_cast<float2*>(mine + 2 * kAttnRows + row * kORow + col) =
          make_float2(o_acc[nd][2 * h], o_acc[nd][2 * h + 1]);
    }
  __syncthreads();
  const int nparts = kAttnWarps + (naux > 0 ? 1 : 0);
  if (naux > 0) {
    // ---- the split's auxiliary keys (the new tokens' own K / V, read at
    // their values in fp32): one more online-softmax state, merged like a warp's
    float* st = ws + kAttnWarps * kWarpState;   // m[16], l[16], o[16][kORow]
    for (int pr = threadIdx.x; pr < naux * kAttnRows; pr += kAttnThreads) {
      const int a = pr / kAttnRows, row = pr % kAttnRows;
      float dot = 0.0f;
      if (row < nh) {
        int j = s_idx[split_main + a] - past;         // auxiliary row of this key
        if (!bounds_ok(j >= 0 && j < p.S, p.status)) j = 0;
        const size_t qo = (static_cast<size_t>(r) * p.Hq + h0 + row) * kD;
        const size_t ko = ((static_cast<size_t>(b) * p.S + j) * p.Hkv + g) * kD;
#pragma unroll 8
        for (int c = 0; c < kD; c += 2) {
          const float2 qv = load_f2<Q_F16>(p.q, qo + c);
          const float2 kv = load_f2<Q_F16>(p.k_aux, ko + c);
          dot = fmaf(qv.x, kv.x, dot);
          dot = fmaf(qv.y, kv.y, dot);
        }
      }
      s_auxp[a][row] = dot * p.scale_log2;
    }
    __syncthreads();
    if (threadIdx.x < kAttnRows) {
      const int row = threadIdx.x;
      float m = -INFINITY;
      for (int a = 0; a < naux; ++a) m = fmaxf(m, s_auxp[a][row]);
      float l = 0.0f;
      for (int a = 0; a < naux; ++a) {
        const float pa = exp2f(s_auxp[a][row] - m);
        s_auxp[a][row] = pa;
        l += pa;
      }
      st[row] = m;
      st[kAttnRows + row] = l;
    }
    __syncthreads();
    float o[kAttnRows];
#pragma unroll
    for (int row = 0; row < kAttnRows; ++row) o[row] = 0.0f;
    for (int a = 0; a < naux; ++a) {
      int j = s_idx[split_main + a] - past;
      if (!bounds_ok(j >= 0 && j < p.S, p.status)) j = 0;
      const size_t vo = ((static_cast<size_t>(b) * p.S + j) * p.Hkv + g) * kD + threadIdx.x;
      const float vv = load_f1<Q_F16>(p.v_aux, vo);
#pragma unroll
      for (int row = 0; row < kAttnRows; ++row) o[row] = fmaf(s_auxp[a][row], vv, o[row]);
    }
#pragma unroll
    for (int row = 0; row < kAttnRows; ++row) st[2 * kAttnRows + row * kORow + threadIdx.x] = o[row];
    __syncthreads();
  }
  if (threadIdx.x < kAttnRows)
    combine_factors(ws, kWarpState, nparts, fac1, fac2, sML);
  __syncthreads();
  if (threadIdx.x == 0) DSA_TS(5);

  const int d = threadIdx.x;   // one output column per thread
  const bool single = (p.nsplit == 1);
  const size_t out_row = static_cast<size_t>(r) * p.Hq + h0;
  float acc[kAttnRows];
#pragma unroll
  for (int row = 0; row < kAttnRows; ++row) acc[row] = 0.0f;
#pragma unroll
  for (int w = 0; w < kAttnWarps + 1; ++w)
    if (w < nparts) {
#pragma unroll
      for (int row = 0; row < kAttnRows; ++row)
        acc[row] += ws[w * kWarpState + 2 * kAttnRows + row * kORow + d] *
                    fac1[w * kAttnRows + row] * fac2[w * kAttnRows + row];
    }
  if (single) {
#pragma unroll
    for (int row = 0; row < kAttnRows; ++row)
      if (row < nh) store_out<OUT>(p.out, (out_row + row) * kD + d, acc[row] / sML[kAttnRows + row]);
    return;
  }
  if (p.cluster) {
    // ---- split combine inside the thread-block cluster. CTA q owns output
    // columns [q * cols, (q + 1) * cols). Every CTA pushes, with st.async into
    // the owners' shared memory, each column's 16 rows and its M, L; the
    // owner's barrier completes when all peers' bytes have landed. Nothing is
    // read from a peer, so no CTA waits for another to leave.
    const int ns = p.nsplit;
    const int cols = kD / ns;                      // ns divides 128 (power of two)
    const uint32_t rank = cluster_ctarank();
    if (threadIdx.x == 0) DSA_TS(6);
    cluster_wait();                                // every peer's barrier is armed
    {
      const uint32_t q = static_cast<uint32_t>(d / cols), c = static_cast<uint32_t>(d % cols);
      const uint32_t bar_q = cluster_map(&s_merge_bar, q);
      const uint32_t dst = cluster_map(recv + 16 * 2 * kAttnRows + (rank * cols + c) * kAttnRows, q);
#pragma unroll
      for (int j = 0; j < kAttnRows / 4; ++j)
        st_async_v4(dst + 16u * j, acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3], bar_q);
      if (threadIdx.x < static_cast<unsigned>(ns)) {
        const uint32_t q2 = threadIdx.x;
        const uint32_t bar2 = cluster_map(&s_merge_bar, q2);
        const uint32_t dml = cluster_map(recv + rank * 2 * kAttnRows, q2);
#pragma unroll
        for (int j = 0; j < 2 * kAttnRows / 4; ++j)
          st_async_v4(dml + 16u * j, sML[4 * j], sML[4 * j + 1], sML[4 * j + 2], sML[4 * j + 3], bar2);
      }
    }
    if (threadIdx.x == 0) DSA_TS(7);
    // every peer pushes, even one whose gathers gave up, so this wait ignores
    // the abort flag (a CTA must not leave while peers may still write to it)
    bool landed_all = mbar_try_wait(&s_merge_bar, 0u);
    for (const long long t0 = clock64(); !landed_all && clock64() - t0 <= kWaitBudgetCycles;)
      landed_all = mbar_try_wait(&s_merge_bar, 0u);
    if (!landed_all) {
      if (threadIdx.x == 0 && p.status) atomicOr(p.status, kDevTimeout);
      return;
    }
    if (threadIdx.x == 0) DSA_TS(8);
    for (int o = threadIdx.x; o < kAttnRows * cols; o += kAttnThreads) {
      const int row = o % kAttnRows, c = o / kAttnRows;
      float mq[16], lq[16], ov[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const bool in = q < ns;
        mq[q] = in ? recv[q * 2 * kAttnRows + row] : -INFINITY;
        lq[q] = in ? recv[q * 2 * kAttnRows + kAttnRows + row] : 0.0f;
        ov[q] = in ? recv[16 * 2 * kAttnRows + (q * cols + c) * kAttnRows + row] : 0.0f;
      }
      float M = -INFINITY;
#pragma unroll
      for (int q = 0; q < 16; ++q) M = fmaxf(M, mq[q]);
      // the peers' weights 2^(m_q - M), summed in a fixed order (deterministic)
      float L = 0.0f, O = 0.0f;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        float f1, f2;
        exp2_pair(mq[q] - M, &f1, &f2);
        L += lq[q] * f1 * f2;
        O += ov[q] * f1 * f2;
      }
      if (row < nh) store_out<OUT>(p.out, (out_row + row) * kD + rank * cols + c, O / L);
    }
    if (threadIdx.x == 0) DSA_TS(9);
    DSA_TS_FLUSH(p.status, 2);
    return;
  }
  float* part = p.partial + ((static_cast<size_t>(r) * gridDim.y + gh) * p.nsplit + blockIdx.x) *
                                kPartialFloats;
  if (d < kAttnRows) {
    part[d] = sML[d];
    part[kAttnRows + d] = sML[kAttnRows + d];
  }
#pragma unroll
  for (int row = 0; row < kAttnRows; ++row) part[2 * kAttnRows + row * kD + d] = acc[row];

  // ---- split combine by the last CTA of this (row, head group)
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t prev = atomicAdd(&p.ticket[static_cast<size_t>(r) * gridDim.y + gh], 1u);
    s_last = (prev == static_cast<uint32_t>(nreal - 1));
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float* parts = p.partial + (static_cast<size_t>(r) * gridDim.y + gh) * p.nsplit * kPartialFloats;
  // m and l of every split into shared memory, then the per-split factors
  float* sm = ws;   // [nreal][2 * 16] (m, l)
  for (int i = threadIdx.x; i < nreal * 2 * kAttnRows; i += kAttnThreads) {
    const int j = i / (2 * kAttnRows), o = i % (2 * kAttnRows);
    sm[j * 2 * kAttnRows + o] = __ldcg(parts + static_cast<size_t>(j) * kPartialFloats + o);
  }
  __syncthreads();
  if (threadIdx.x < kAttnRows)
    combine_factors(sm, 2 * kAttnRows, nreal, fac1, fac2, sML);
  __syncthreads();
#pragma unroll
  for (int row = 0; row < kAttnRows; ++row) acc[row] = 0.0f;
#pragma unroll 2
  for (int j = 0; j < nreal; ++j) {
    const float* oj = parts + static_cast<size_t>(j) * kPartialFloats + 2 * kAttnRows + d;
    float v[kAttnRows];
#pragma unroll
    for (int row = 0; row < kAttnRows; ++row) v[row] = __ldcg(oj + row * kD);
#pragma unroll
    for (int row = 0; row < kAttnRows; ++row)
      acc[row] += v[row] * fac1[j * kAttnRows + row] * fac2[j * kAttnRows + row];
  }
#pragma unroll
  for (int row = 0; row < kAttnRows; ++row)
    if (row < nh) store_out<OUT>(p.out, (out_row + row) * kD + d, acc[row] / sML[kAttnRows + row]);
}

template <int KV, bool Q_F16, int OUT>
static cudaError_t launch_t(const AttnParams& p, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                            cudaStream_t stream) {
  auto kern = sparse_attn_kernel<KV, Q_F16, OUT>;
  const int smem = p.cluster ? kAttnSmemCluster : kAttnSmem;
  cudaError_t e = set_max_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(p.nsplit, p.Hkv * p.HG, p.B * p.S);
  if (!p.cluster)
    return launch_kernel("sparse_attn_kernel", kern, grid, dim3(kAttnThreads), smem, stream, true,
                         tm_k, tm_v, p);
  if (p.nsplit > 8) {
    e = set_nonportable_cluster(reinterpret_cast<const void*>(kern));
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.nsplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kern, tm_k, tm_v, p);
  if (e == cudaSuccess) note_launch("sparse_attn_kernel");
  return e;
}

template <int KV, bool Q_F16>
static cudaError_t launch_out(const AttnParams& p, int out_dtype, const CUtensorMap& tm_k,
                              const CUtensorMap& tm_v, cudaStream_t stream) {
  switch (out_dtype) {
    case DSA_BF16: return launch_t<KV, Q_F16, DSA_BF16>(p, tm_k, tm_v, stream);
    case DSA_FP16: return launch_t<KV, Q_F16, DSA_FP16>(p, tm_k, tm_v, stream);
    case DSA_FP32: return launch_t<KV, Q_F16, DSA_FP32>(p, tm_k, tm_v, stream);
    default: return cudaErrorInvalidValue;
  }
}

int attn_cluster_capacity(int size) {
  // per device and cluster size (2, 4, 8, 16): clusters resident at once
  static std::mutex mu;
  static int cached[64][5] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int si = size == 2 ? 0 : size == 4 ? 1 : size == 8 ? 2 : size == 16 ? 3 : 4;
  if (si == 4) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev][si]) return cached[dev][si] - 1;
  int n = 0;
  auto kern = sparse_attn_kernel<KV_FP16, false, DSA_BF16>;
  if (set_max_smem(reinterpret_cast<const void*>(kern), kAttnSmemCluster) == cudaSuccess &&
      (size <= 8 || set_nonportable_cluster(reinterpret_cast<const void*>(kern)) == cudaSuccess)) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(size, 1, 1);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = kAttnSmemCluster;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = size;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  cached[dev][si] = n + 1;
  return n;
}

int attn_max_cluster() { return attn_cluster_capacity(16) >= 1 ? 16 : 8; }

cudaError_t launch_attention(const AttnParams& p, int q_dtype, int kv_dtype, int out_dtype,
                             const CUtensorMap& tm_k, const CUtensorMap& tm_v, cudaStream_t stream) {
  const bool qf16 = (q_dtype == DSA_FP16);
  switch (kv_dtype) {
    case DSA_BF16:
      if (qf16) return cudaErrorInvalidValue;
      return launch_out<KV_BF16, false>(p, out_dtype, tm_k, tm_v, stream);
    case DSA_FP16:
      return qf16 ? launch_out<KV_FP16, true>(p, out_dtype, tm_k, tm_v, stream)
                  : launch_out<KV_FP16, false>(p, out_dtype, tm_k, tm_v, stream);
    case DSA_INT8:
      return qf16 ? launch_out<KV_INT8, true>(p, out_dtype, tm_k, tm_v, stream)
                  : launch_out<KV_INT8, false>(p, out_dtype, tm_k, tm_v, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace dsa
