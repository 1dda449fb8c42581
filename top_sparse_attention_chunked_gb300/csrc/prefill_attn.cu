// Sparse GQA attention for prefill on tcgen05 tensor cores.
//
// PR #33997 "[CUDA] Support FP16 KV cache and FP16 query/key in
// DynamicSparseAttention<BFloat16> ...", Description item 2: the pages run the
// sparse-attention prefill on tensor cores (mma.sync m16n8k16 f32.f16.f16.f32)
// over each query token's selected K/V rows. Here the dense tiles run on the
// 5th-generation tensor cores with tensor-memory accumulators.
//
// One work item = (query token, KV head, group of <= 16 query heads) with up to
// 2,048 selected keys (16 tiles of 128). Per item:
//   1. QK^T, "swap-AB": for each tile of 128 gathered K rows (A, K-major, 128-byte
//      swizzle) against the 16 head queries (B), tcgen05.mma writes a 128 x 16
//      fp32 block of logits into tensor memory; all 16 blocks stay resident
//      (256 TMEM columns), so the softmax needs no online rescaling at all;
//   2. the epilogue warps (one TMEM lane = one key each) take the exact per-head
//      maximum over every selected key, then form P = exp2(s - max) tile by
//      tile and write it to shared memory as a K-major [16 heads x 128 keys]
//      operand (BF16 hi + lo pair for a BF16 cache, FP16 for an FP16 cache);
//   3. PV^T: for each tile of 128 gathered V rows, read MN-major (head dim
//      contiguous) as the A operand, tcgen05.mma accumulates O^T[128 dims x 16
//      heads] in tensor memory; the epilogue divides by the row sums and stores.
// Four loader warps gather the selected rows with TMA row gathers (four rows
// of 128 bytes per instruction, 128-byte swizzle applied by the copy engine)
// into a ring of shared stages; a single warp issues row gathers at only a
// fraction of the L2 bandwidth, so each loader warp fills a quarter of every
// tile. One warp issues the MMAs and owns tensor memory. A persistent grid of two CTAs
// per SM (256 tensor-memory columns and ~112 KB of shared memory each) walks
// the work items, so one CTA's gather overlaps the other's softmax and MMAs.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dsa_common.cuh"
#include "dsa_internal.h"
#include "sm100_ptx.cuh"

namespace dsa {

namespace pf {
constexpr int kThreads = 288;          // warp 0 MMA, warps 1-4 softmax, warps 5-8 loaders
constexpr int kLoadWarps = 4;
constexpr int kKeys = 128;             // keys per tile (MMA M for QK^T, K for PV^T)
constexpr int kMaxTiles = 16;          // 2,048 selected keys
constexpr int kStages = 3;             // two CTAs share an SM
constexpr uint32_t kTileBytes = kKeys * DSA_HEAD_DIM * 2;   // 32 KB: 2 column blocks of 16 KB
constexpr uint32_t kBlockBytes = kKeys * 128;               // one 64-wide column block
constexpr uint32_t kQBytes = 16 * DSA_HEAD_DIM * 2;         // 4 KB
constexpr uint32_t kPBytes = 16 * kKeys * 2;                // 4 KB: [16 heads x 128 keys]
// 16 logit tiles x 16 columns fill the 256 columns; O^T reuses the first
// logit tile's columns: PV(0) writes them only after P(0) has been formed
constexpr int kOCol = 0;
constexpr uint32_t kTmemCols = 256;

struct Bars {
  uint64_t full[kStages], empty[kStages];
  uint64_t q_ready, logits_ready, o_ready, tmem_free;
  uint64_t p_ready, p_free;
  uint64_t done;
  uint64_t grp;          // barrier of the 128 softmax threads
  uint32_t tmem_base;
  int abort_flag;
  float red[2][4][16];   // cross-warp max / sum scratch
};

constexpr size_t kSmemBytes = 1024 + kStages * kTileBytes + kQBytes + 2 * kPBytes + sizeof(Bars);
}  // namespace pf

// Shared-memory descriptor with explicit leading/stride byte offsets and
// 128-byte swizzle (K-major: stride = 8-row group pitch; MN-major: leading =
// pitch of 64-element MN blocks, stride = 8-row K group pitch).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// kind::f16 instruction descriptor: f32 accumulate, A/B both BF16 (F16 = false)
// or both FP16, A K-major or MN-major, B K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool f16, bool a_mn_major) {
  return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) |
         ((a_mn_major ? 1u : 0u) << 15) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Barrier of a thread group on an mbarrier whose count is the group size, with
// the bounded wait (a named barrier could strand threads that gave up).
__device__ __forceinline__ bool group_sync(uint64_t* bar, uint32_t* phase, volatile int* abort_flag) {
  mbar_arrive(bar);
  const bool ok = mbar_wait_bounded(bar, *phase, abort_flag);
  *phase ^= 1u;
  return ok;
}

// Byte offset of element (row, col) in a K-major SW128 operand whose rows hold
// `cols` 16-bit elements split in 64-element column blocks of `rows` * 128 B.
__device__ __forceinline__ uint32_t sw128_off(int row, int col, int rows) {
  const int blk = col >> 6, c = col & 63;
  return static_cast<uint32_t>(blk * rows * 128 + row * 128 + ((((c >> 3) ^ (row & 7))) << 4) +
                               (c & 7) * 2);
}

struct PfItem {
  int r, g, hg, keff, ntiles;
};

__device__ __forceinline__ PfItem pf_item(const AttnParams& p, long long it) {
  PfItem w;
  const int per_row = p.Hkv * p.HG;
  w.r = static_cast<int>(it / per_row);
  const int gh = static_cast<int>(it % per_row);
  w.g = gh / p.HG;
  w.hg = gh % p.HG;
  const int b = w.r / p.S, s = w.r % p.S;
  w.keff = min(p.topk, visible_len(p.lens.T[b], p.S, s));
  w.ntiles = (w.keff + pf::kKeys - 1) / pf::kKeys;
  return w;
}

// tm_k / tm_v view the caches as [B * cap * Hkv rows, 128] 16-bit matrices
// (row (b * cap + key) * Hkv + g), box 64 x 1, 128-byte swizzle.
template <bool F16, bool PAGED>
__global__ void __launch_bounds__(pf::kThreads, 2)
    sparse_attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                                  const __grid_constant__ CUtensorMap tm_v, const AttnParams p,
                                  long long n_items, uint32_t* status) {
  using namespace pf;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sKV = base;                                 // kStages x 32 KB
  uint8_t* sQ = sKV + kStages * kTileBytes;            // 4 KB
  uint8_t* sP = sQ + kQBytes;                          // [hi, lo] x 4 KB
  Bars* bars = reinterpret_cast<Bars*>(sP + 2 * kPBytes);
  volatile int* abort_flag = &bars->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // trace build: phase stamps of each CTA's third item (steady state)
  DSA_TS_DECL;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars->full[i], kLoadWarps);
      mbar_init(&bars->empty[i], 1);
    }
    mbar_init(&bars->q_ready, 128);
    mbar_init(&bars->logits_ready, 1);
    mbar_init(&bars->o_ready, 1);
    mbar_init(&bars->tmem_free, 128);
    mbar_init(&bars->p_ready, 128);
    mbar_init(&bars->p_free, 1);
    mbar_init(&bars->done, 1);
    mbar_init(&bars->grp, 128);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&bars->tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const long long my_first = blockIdx.x;
  const long long stride = gridDim.x;

  if (warp >= 5) {
    // ------------------------------------------------------------ loaders
    const int lw = warp - 5;
    if (threadIdx.x == 160) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    pdl_wait();      // the selected indices come from the previous kernel
    // lanes 0-15 issue one gather each per tile: rows 4 * grp .. 4 * grp + 3
    // of the tile, column block cb
    const int grp = lw * 8 + (lane & 7);
    const int cb = (lane >> 3) & 1;
    const bool issuer = lane < 16;
    long long seq = 0;                   // position in the ring (tiles issued)
    bool ok = true;
    bool bad_page = false;               // a block-table entry outside the pool was read
    long long nit = 0;                   // items of this CTA so far (trace stamps)
    for (long long it = my_first; it < n_items && ok; it += stride, ++nit) {
      const PfItem w = pf_item(p, it);
      const int b = w.r / p.S;
      const int T = p.lens.T[b];
      const int32_t* idx_row = p.idx + static_cast<size_t>(w.r) * p.topk;
      // rows past k_eff (and any index outside the visible cache) read key 0,
      // whose logits the softmax masks
      auto rows_of = [&](int t, int* y) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = t * kKeys + 4 * grp + e;
          int key = j < w.keff ? __ldg(idx_row + j) : 0;
          if (key < 0 || key >= T) key = 0;
          // dense rows in 32-bit arithmetic: the loaders' issue rate bounds
          // this kernel, so the paged lookup is a separate instantiation
          if constexpr (PAGED)
            y[e] = static_cast<int>(cache_row(p.pg, b, p.cap, key, &bad_page) * p.Hkv + w.g);
          else
            y[e] = b * static_cast<int>(p.kv_sb) + key * static_cast<int>(p.kv_st) +
                   w.g * static_cast<int>(p.kv_sh);   // the host keeps every row below 2^31
          if (!bounds_ok(y[e] >= 0 && y[e] < p.kv_rows, status)) y[e] = 0;
        }
      };
      for (int pass = 0; pass < 2 && ok; ++pass) {            // K tiles, then V tiles
        const CUtensorMap* tm = pass == 0 ? &tm_k : &tm_v;
        int nxt[4];
        if (issuer) rows_of(0, nxt);
        for (int t = 0; t < w.ntiles; ++t) {
          const int y0 = nxt[0], y1 = nxt[1], y2 = nxt[2], y3 = nxt[3];
          if (issuer && t + 1 < w.ntiles) rows_of(t + 1, nxt);
          const int st = static_cast<int>(seq % kStages);
          bool got = seq < kStages ||
                     mbar_wait_bounded(&bars->empty[st],
                                       static_cast<uint32_t>(((seq / kStages) - 1) & 1), abort_flag);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(&bars->full[st], kTileBytes / kLoadWarps);
          if (nit == 2 && lane == 0 && t == 0) DSA_TS(pass == 0 ? 0 : 1);
          if (nit == 2 && lane == 0 && pass == 1 && t == w.ntiles - 1) DSA_TS(2);
          __syncwarp();
          if (issuer)
            tma_gather4(sKV + st * kTileBytes + cb * kBlockBytes + grp * 512, tm, &bars->full[st],
                        cb * 64, y0, y1, y2, y3);
          ++seq;
        }
      }
    }
    if (bad_page) atomicOr(status, kDevBadPage);
    if (lane == 0) {
      // the ring's last copies may still be landing (the consumers may have
      // given up): wait, bounded, for them before the block can exit
      for (long long s2 = seq > kStages ? seq - kStages : 0; s2 < seq; ++s2) {
        const long long t0 = clock64();
        while (!mbar_try_wait(&bars->full[s2 % kStages], static_cast<uint32_t>((s2 / kStages) & 1)) &&
               clock64() - t0 < kWaitBudgetCycles) {
        }
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_f16(kKeys, 16, F16, false);
      constexpr uint32_t id_pv = idesc_f16(DSA_HEAD_DIM, 16, F16, true);
      long long seq = 0;
      long long n = 0;   // items handled by this CTA
      long long ptile = 0;
      for (long long it = my_first; it < n_items; it += stride, ++n) {
        const PfItem w = pf_item(p, it);
        // the softmax warps must be done with the previous item's tensor memory
        if (n > 0 && !mbar_wait_bounded(&bars->tmem_free, static_cast<uint32_t>((n - 1) & 1), abort_flag))
          break;
        if (!mbar_wait_bounded(&bars->q_ready, static_cast<uint32_t>(n & 1), abort_flag)) break;
        tc_fence_after();
        if (n == 2) DSA_TS(3);
        bool ok = true;
        for (int t = 0; t < w.ntiles; ++t, ++seq) {
          const int st = static_cast<int>(seq % kStages);
          if (!mbar_wait_bounded(&bars->full[st], static_cast<uint32_t>((seq / kStages) & 1), abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (n == 2 && t == 0) DSA_TS(4);
          const uint32_t a0 = smem_u32(sKV + st * kTileBytes);
          const uint32_t b0 = smem_u32(sQ);
#pragma unroll
          for (int kk = 0; kk < DSA_HEAD_DIM / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * kBlockBytes + (kk & 3) * 32;
            const uint32_t qoff = (kk >> 2) * (16 * 128) + (kk & 3) * 32;
            tc_mma_f16(tmem + t * 16, desc_sw128(a0 + koff, 16, 1024), desc_sw128(b0 + qoff, 16, 1024),
                       id_qk, kk > 0 ? 1u : 0u);
          }
          tc_commit(&bars->empty[st]);
        }
        if (!ok) break;
        if (n == 2) DSA_TS(5);
        tc_commit(&bars->logits_ready);
        for (int t = 0; t < w.ntiles; ++t, ++seq, ++ptile) {
          const int st = static_cast<int>(seq % kStages);
          if (!mbar_wait_bounded(&bars->full[st], static_cast<uint32_t>((seq / kStages) & 1), abort_flag)) {
            ok = false;
            break;
          }
          if (!mbar_wait_bounded(&bars->p_ready, static_cast<uint32_t>(ptile & 1), abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t v0 = smem_u32(sKV + st * kTileBytes);
          const uint32_t ph = smem_u32(sP);
          const uint32_t pl = ph + kPBytes;
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk) {
            const uint32_t voff = kk * 16 * 128;                       // 16 keys of both blocks
            const uint32_t poff = (kk >> 2) * (16 * 128) + (kk & 3) * 32;
            const uint64_t adesc = desc_sw128(v0 + voff, kBlockBytes, 1024);
            tc_mma_f16(tmem + kOCol, adesc, desc_sw128(ph + poff, 16, 1024), id_pv,
                       (t > 0 || kk > 0) ? 1u : 0u);
            if constexpr (!F16)
              tc_mma_f16(tmem + kOCol, adesc, desc_sw128(pl + poff, 16, 1024), id_pv, 1u);
          }
          tc_commit(&bars->empty[st]);
          tc_commit(&bars->p_free);
        }
        if (!ok) break;
        if (n == 2) DSA_TS(9);
        tc_commit(&bars->o_ready);
      }
      tc_commit(&bars->done);
      long long t0 = clock64();
      while (!mbar_try_wait(&bars->done, 0) && clock64() - t0 < kWaitBudgetCycles) {
      }
    }
  } else if (warp >= 1) {
    // ------------------------------------------------------------ softmax / epilogue
    const int et = threadIdx.x - 32;          // 0..127
    const int quarter = warp & 3;
    const int key_in_tile = quarter * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = p.scale_log2;
    long long n = 0, ptile = 0;
    uint32_t gphase = 0;

    auto load_q = [&](const PfItem& w) {
      // [16 heads x 128 dims] K-major SW128; heads past the group are zero
      const int h0 = w.g * p.G + w.hg * 16;
      const int nh = min(16, p.G - w.hg * 16);
      for (int i = et; i < 16 * 16; i += 128) {
        const int h = i >> 4, ch = i & 15;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (h < nh) {
          const uint16_t* qrow = static_cast<const uint16_t*>(p.q) +
                                 (static_cast<size_t>(w.r) * p.Hq + h0 + h) * DSA_HEAD_DIM + ch * 8;
          v = *reinterpret_cast<const uint4*>(qrow);
          if (F16 && p.q_dtype == DSA_BF16) {
            const __nv_bfloat16* bsrc = reinterpret_cast<const __nv_bfloat16*>(&v);
            __half hv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) hv[e] = __float2half_rn(__bfloat162float(bsrc[e]));
            v = *reinterpret_cast<const uint4*>(hv);
          }
        }
        *reinterpret_cast<uint4*>(sQ + sw128_off(h, ch * 8, 16)) = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->q_ready);
    };

    long long it = my_first;
    if (it < n_items) load_q(pf_item(p, it));
    for (; it < n_items; it += stride, ++n) {
      const PfItem w = pf_item(p, it);
      if (!mbar_wait_bounded(&bars->logits_ready, static_cast<uint32_t>(n & 1), abort_flag)) break;
      tc_fence_after();
      if (n == 2 && et == 0) DSA_TS(6);
      // the query buffer is free once the logits are in: stage the next item's
      if (it + stride < n_items) load_q(pf_item(p, it + stride));

      // ---- exact per-head max over all selected keys
      float mx[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) mx[h] = -INFINITY;
      for (int t = 0; t < w.ntiles; ++t) {
        float v[16];
        tmem_ld16(tmem + lane_addr + t * 16, v);
        tmem_ld_wait();
        if (t * kKeys + key_in_tile < w.keff) {
#pragma unroll
          for (int h = 0; h < 16; ++h) mx[h] = fmaxf(mx[h], v[h]);
        }
      }
#pragma unroll
      for (int h = 0; h < 16; ++h)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], o));
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < 16; ++h) bars->red[0][warp - 1][h] = mx[h];
      }
      if (!group_sync(&bars->grp, &gphase, abort_flag)) break;
      if (n == 2 && et == 0) DSA_TS(7);
      float M[16];
#pragma unroll
      for (int h = 0; h < 16; ++h)
        M[h] = fmaxf(fmaxf(bars->red[0][0][h], bars->red[0][1][h]),
                     fmaxf(bars->red[0][2][h], bars->red[0][3][h])) * c;

      // ---- P tiles
      float lsum[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) lsum[h] = 0.0f;
      for (int t = 0; t < w.ntiles; ++t, ++ptile) {
        if (ptile >= 1 &&
            !mbar_wait_bounded(&bars->p_free, static_cast<uint32_t>((ptile - 1) & 1), abort_flag))
          break;
        float v[16];
        tmem_ld16(tmem + lane_addr + t * 16, v);
        tmem_ld_wait();
        const bool valid = t * kKeys + key_in_tile < w.keff;
        uint8_t* ph = sP;
        uint8_t* pl = ph + kPBytes;
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          const float pv = valid ? exp2f(fmaf(v[h], c, -M[h])) : 0.0f;
          lsum[h] += pv;
          const uint32_t off = sw128_off(h, key_in_tile, 16);
          if constexpr (F16) {
            *reinterpret_cast<__half*>(ph + off) = __float2half_rn(pv);
          } else {
            const __nv_bfloat16 hi = __float2bfloat16_rn(pv);
            *reinterpret_cast<__nv_bfloat16*>(ph + off) = hi;
            *reinterpret_cast<__nv_bfloat16*>(pl + off) = __float2bfloat16_rn(pv - __bfloat162float(hi));
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars->p_ready);
      }
      if (n == 2 && et == 0) DSA_TS(8);
      // ---- row sums
#pragma unroll
      for (int h = 0; h < 16; ++h)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lsum[h] += __shfl_xor_sync(0xffffffffu, lsum[h], o);
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < 16; ++h) bars->red[1][warp - 1][h] = lsum[h];
      }
      if (!group_sync(&bars->grp, &gphase, abort_flag)) break;
      // ---- O^T: TMEM lane = head dim, columns = heads
      if (!mbar_wait_bounded(&bars->o_ready, static_cast<uint32_t>(n & 1), abort_flag)) break;
      tc_fence_after();
      if (n == 2 && et == 0) DSA_TS(10);
      float o[16];
      tmem_ld16(tmem + lane_addr + kOCol, o);
      tmem_ld_wait();
      const int h0 = w.g * p.G + w.hg * 16;
      const int nh = min(16, p.G - w.hg * 16);
      const int d = key_in_tile;   // lane of the O^T accumulator
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        if (h >= nh) break;
        const float L = bars->red[1][0][h] + bars->red[1][1][h] + bars->red[1][2][h] + bars->red[1][3][h];
        const size_t oi = (static_cast<size_t>(w.r) * p.Hq + h0 + h) * DSA_HEAD_DIM + d;
        const float val = o[h] / L;
        if (p.out_dtype == DSA_BF16) static_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(val);
        else if (p.out_dtype == DSA_FP16) static_cast<__half*>(p.out)[oi] = __float2half_rn(val);
        else static_cast<float*>(p.out)[oi] = val;
      }
      if (n == 2 && et == 0) DSA_TS(11);
      tc_fence_before();
      mbar_arrive(&bars->tmem_free);
      // red[] reads done before the next item reuses it
      if (!group_sync(&bars->grp, &gphase, abort_flag)) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0 && bars->abort_flag) atomicOr(status, kDevTimeout);
  DSA_TS_FLUSH(status, 2);
}

bool prefill_tc_supported(const AttnParams& p, int kv_dtype, size_t smem_optin) {
  // gather row coordinates are signed 32-bit
  const long long tokens = p.pg.table ? (static_cast<long long>(p.pg.num_blocks) << p.pg.shift)
                                      : static_cast<long long>(p.B) * p.cap;
  const long long rows = tokens * p.Hkv;
  return (kv_dtype == DSA_BF16 || kv_dtype == DSA_FP16) && p.topk <= pf::kMaxTiles * pf::kKeys &&
         rows < (1LL << 31) && pf::kSmemBytes <= smem_optin;
}

template <bool F16, bool PAGED>
static cudaError_t launch_prefill_variant(const AttnParams& p, int grid, const CUtensorMap& tm_k,
                                          const CUtensorMap& tm_v, long long n_items,
                                          uint32_t* status, cudaStream_t stream) {
  auto k = sparse_attn_prefill_tc_kernel<F16, PAGED>;
  cudaError_t e = set_max_smem(reinterpret_cast<const void*>(k), static_cast<int>(pf::kSmemBytes));
  if (e != cudaSuccess) return e;
  return launch_kernel("sparse_attn_prefill_tc_kernel", k, dim3(grid), dim3(pf::kThreads),
                       pf::kSmemBytes, stream, true, tm_k, tm_v, p, n_items, status);
}

cudaError_t launch_prefill_tc(const AttnParams& p, int kv_dtype, int sms, const CUtensorMap& tm_k,
                              const CUtensorMap& tm_v, uint32_t* status, cudaStream_t stream) {
  const long long n_items = static_cast<long long>(p.B) * p.S * p.Hkv * p.HG;
  // two CTAs per SM: one gathers while the other computes
  const int grid = static_cast<int>(n_items < 2 * sms ? n_items : 2 * sms);
  const bool paged = p.pg.table != nullptr;
  if (kv_dtype == DSA_FP16)
    return paged ? launch_prefill_variant<true, true>(p, grid, tm_k, tm_v, n_items, status, stream)
                 : launch_prefill_variant<true, false>(p, grid, tm_k, tm_v, n_items, status, stream);
  return paged ? launch_prefill_variant<false, true>(p, grid, tm_k, tm_v, n_items, status, stream)
               : launch_prefill_variant<false, false>(p, grid, tm_k, tm_v, n_items, status, stream);
}

}  // namespace dsa
