// Indexer on tcgen05 tensor cores.
//
//   score[b,s,t] = sum_h w[b,s,h] * max(0, qI[b,s,h,:] . kI[b,t,:])
//
// (PR #33802 "... DSA, Indexer, HC, and QMoE kernels for SM12x and 256K
// context", Summary item 2: every cached index key is scored against each
// query token's 16 index heads; the pages' SM12x kernel tiles 8 query tokens
// per CTA and reduces the 16 heads with a shuffle butterfly.)
//
// GB300 design. The contraction is laid out "keys as M": one 128-key tile of
// kI (128 rows x 64 bf16 = 16 KB, streamed from HBM by TMA) is the A operand,
// the query block's index queries (QB tokens x 16 heads = N rows x 64) are the
// B operand, and tcgen05.mma accumulates D[128 keys x N] in fp32 tensor
// memory. After tcgen05.ld every epilogue thread owns one key and holds all
// 16 head dot-products of a query in registers, so the ReLU, the head weights
// and the head sum are plain per-thread FMAs -- no shuffles, no shared-memory
// reduction. The same kernel serves decode (QB = S, all queries of a sequence
// in one block, the radix histograms of the top-k fused into the epilogue)
// and prefill (QB = 16, N = 256, causal: tile ranges stop at each block's
// last visible key).
//
// Warp roles (320 threads): warp 0 issues TMA loads into a ring of shared
// stages, warp 1 owns tensor memory and issues the MMAs, warps 2-9 are two
// epilogue groups of 4 warps (warp w reads TMEM lanes 32*(w%4) .. +31).
// Accumulators are double-buffered in TMEM so the MMA of tile i+1 overlaps
// the epilogue of tile i. Two epilogue organisations:
//   * alternate tiles (blocks under 8 queries: single-token decode): group g
//     takes the tiles of parity g with all of the block's queries, head
//     weights read from shared memory;
//   * split queries (blocks of 8 or 16 queries: prefill, multi-token decode):
//     both groups read every tile, group g taking half of the block's
//     queries, with those queries' head weights held in registers across the
//     block's tiles. At K = 64 the epilogue has about as many
//     instructions per tile as the MMA has cycles, so it sets the pace: a
//     warp-wide broadcast read of the weights from shared memory costs
//     several shared-pipe wavefronts per 16 bytes, enough to saturate that
//     pipe, and half of the heads take their ReLU on the FMA pipe (see
//     relu_weighted_sum_r) to relieve the half-rate ALU pipe.
// Work is a flat list of (sequence, query block, key tile) units split evenly
// over a persistent grid of one CTA per SM.
#include <cstdio>

#include "dsa_common.cuh"
#include "dsa_internal.h"
#include "sm100_ptx.cuh"

namespace dsa {

constexpr int kMaxAcc = 4;
// Backoff (ns) of the roles' mbarrier retries: the epilogue sets the pace, and
// the producer and MMA warps, which wait most of each tile, share schedulers
// with epilogue warps (prefill indexer 775 -> 761 us; 128 ns and a try_wait
// suspend hint were slower).
constexpr int kIdxNap = 32;
constexpr int kIdxMaxStages = 8;
constexpr uint32_t kATileBytes = kKeyTile * DSA_IDX_DIM * 2;   // 16 KB

struct UnitCursor {
  int b, qb, kt, ntiles;
};

__device__ __forceinline__ int block_tiles(const IndexerParams& p, int b, int qb) {
  const int last_s = min(p.S, (qb + 1) * p.QB) - 1;
  const int n = visible_len(p.lens.T[b], p.S, last_s);
  return (n + kKeyTile - 1) / kKeyTile;
}

__device__ __forceinline__ UnitCursor locate_unit(const IndexerParams& p, long long u) {
  UnitCursor c{p.B, 0, 0, 0};
  for (int b = 0; b < p.B; ++b)
    for (int qb = 0; qb < p.nqb; ++qb) {
      const int nt = block_tiles(p, b, qb);
      if (u < nt) {
        c.b = b; c.qb = qb; c.kt = static_cast<int>(u); c.ntiles = nt;
        return c;
      }
      u -= nt;
    }
  return c;
}

__device__ __forceinline__ void advance_unit(const IndexerParams& p, UnitCursor& c) {
  if (++c.kt < c.ntiles) return;
  c.kt = 0;
  do {
    if (++c.qb >= p.nqb) { c.qb = 0; ++c.b; }
    if (c.b >= p.B) return;
    c.ntiles = block_tiles(p, c.b, c.qb);
  } while (c.ntiles == 0);
}

// sum over heads of w_h * ReLU(dot_h), two heads per paired FMA, with the
// weights in registers. For the first kAbsHeads heads the weight is held
// halved (hw = w / 2) and ReLU(x) is taken as x + |x|: for finite x that is
// exactly 2 * ReLU(x), and (w / 2) * (2 * ReLU(x)) is the same real product
// as w * ReLU(x), so the sum rounds exactly as with max(x, 0) throughout. The
// addition (|x| is a free source modifier) runs on the FMA pipe, where a max
// takes a slot of the half-rate ALU pipe.
// heads whose ReLU is taken as x + |x| (FMA pipe) with a halved weight; the
// rest use max(x, 0) (ALU pipe), which balances the two pipes
constexpr int kAbsHeads = 8;
__device__ __forceinline__ float relu2(float x, int h) { return h < kAbsHeads ? x + fabsf(x) : fmaxf(x, 0.0f); }
__device__ __forceinline__ float relu_weighted_sum_r(const float (&d)[16], const float (&hw)[16]) {
  float2 acc2 = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int h2 = 0; h2 < DSA_IDX_HEADS / 2; ++h2)
    acc2 = fma_f32x2(make_float2(hw[2 * h2], hw[2 * h2 + 1]),
                     make_float2(relu2(d[2 * h2], 2 * h2), relu2(d[2 * h2 + 1], 2 * h2 + 1)), acc2);
  return acc2.x + acc2.y;
}

// the same with the weights read from shared memory
__device__ __forceinline__ float relu_weighted_sum(const float (&d)[16], const float* w) {
  const float4* w4p = reinterpret_cast<const float4*>(w);
  float2 acc2 = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int h4 = 0; h4 < DSA_IDX_HEADS / 4; ++h4) {
    const float4 w4 = w4p[h4];
    acc2 = fma_f32x2(make_float2(w4.x, w4.y), make_float2(fmaxf(d[4 * h4], 0.0f), fmaxf(d[4 * h4 + 1], 0.0f)), acc2);
    acc2 = fma_f32x2(make_float2(w4.z, w4.w), make_float2(fmaxf(d[4 * h4 + 2], 0.0f), fmaxf(d[4 * h4 + 3], 0.0f)), acc2);
  }
  return acc2.x + acc2.y;
}

// Bounded wait used on the unwinding path: ignores the abort flag.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitBudgetCycles) return;
  }
}

// Blocks of 8 or more queries split their queries between the two epilogue
// groups; smaller blocks alternate tiles between them.
constexpr int kIdxGroups = 2;
__host__ __device__ constexpr bool idx_qsplit(int QB, bool) { return QB >= 8; }

template <int N, bool HIST>
struct IdxCfg {
  static constexpr int QB = N / 16;
  static constexpr int NG = kIdxGroups;
  static constexpr bool QSPLIT = idx_qsplit(QB, HIST);
  static constexpr int QPG = QSPLIT ? QB / NG : QB;   // queries a group sums per tile
  static constexpr int kEpiThreads = 128 * NG;
  static constexpr int kThreads = 64 + kEpiThreads;   // warp 0 TMA, warp 1 MMA, epilogue
  static constexpr uint32_t kBBytes = N * DSA_IDX_DIM * 2;
  // accumulator buffers in tensor memory: 4 for narrow tiles, 2 for wide ones
  static constexpr int NACC = N <= 64 ? 4 : 2;
  static constexpr uint32_t kTmemCols = (NACC * N <= 32) ? 32 : (NACC * N <= 64) ? 64
                                      : (NACC * N <= 128) ? 128 : (NACC * N <= 256) ? 256 : 512;
  // queries whose accumulator columns are read per tcgen05.ld batch (two
  // batches in flight: the next is loaded while the current is summed); one
  // when the group's head weights live in registers
  static constexpr int QG = QSPLIT ? 1 : (QPG < 2 ? QPG : 2);
};

struct IdxBarriers {
  uint64_t full[kIdxMaxStages];
  uint64_t empty[kIdxMaxStages];
  uint64_t bfull[2], bempty[2];
  uint64_t accfull[kMaxAcc], accempty[kMaxAcc];
  uint64_t done;
  uint32_t tmem_base;
  int abort_flag;
};

__host__ __device__ inline size_t indexer_smem_layout(int N, bool with_hist, int stages,
                                                     size_t* off_b, size_t* off_w,
                                                     size_t* off_hist, size_t* off_bar) {
  const int QB = N / 16;
  size_t o = static_cast<size_t>(stages) * kATileBytes;
  *off_b = o;
  // two query-block buffers when a CTA may move to a new block (prefill);
  // with histograms a CTA owns one sequence's single block
  o += (with_hist ? 1ull : 2ull) * N * DSA_IDX_DIM * 2;
  // one copy per epilogue warp of the head weights of the queries it sums
  *off_w = o;
  const int ng = kIdxGroups;
  const int qpg = idx_qsplit(QB, with_hist) ? QB / ng : QB;
  o += static_cast<size_t>(4 * ng) * qpg * 16 * sizeof(float);
  o = (o + 15) & ~size_t(15);
  *off_hist = o;
  if (with_hist) o += static_cast<size_t>(QB) * kHistBins * sizeof(uint32_t);
  o = (o + 15) & ~size_t(15);
  *off_bar = o;
  o += sizeof(IdxBarriers);
  return o + 1024;   // slack to align the dynamic base to 1024 bytes
}

template <int N, bool HIST>
__global__ void __launch_bounds__(IdxCfg<N, HIST>::kThreads, 1)
    indexer_tc_kernel(const __grid_constant__ CUtensorMap tm_kI,
                      const __grid_constant__ CUtensorMap tm_qI, const IndexerParams p,
                      int stages) {
  using C = IdxCfg<N, HIST>;
  constexpr int QB = C::QB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  size_t off_b, off_w, off_hist, off_bar;
  indexer_smem_layout(N, HIST, stages, &off_b, &off_w, &off_hist, &off_bar);
  uint8_t* sA = base;
  uint8_t* sB = base + off_b;
  float* sW = reinterpret_cast<float*>(base + off_w);
  uint32_t* sHist = reinterpret_cast<uint32_t*>(base + off_hist);
  IdxBarriers* bars = reinterpret_cast<IdxBarriers*>(base + off_bar);
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Unit range of this CTA. A 2-D grid (decode) gives every sequence its own
  // CTAs (gridDim.y == B, one query block per sequence), so a CTA never
  // changes query block and its histograms are flushed once at the end.
  long long u0, u1;
  if (gridDim.y > 1) {
    long long start = 0;
    for (int b = 0; b < static_cast<int>(blockIdx.y); ++b)
      for (int qb = 0; qb < p.nqb; ++qb) start += block_tiles(p, b, qb);
    long long nb = 0;
    for (int qb = 0; qb < p.nqb; ++qb) nb += block_tiles(p, blockIdx.y, qb);
    u0 = start + nb * blockIdx.x / gridDim.x;
    u1 = start + nb * (blockIdx.x + 1) / gridDim.x;
  } else {
    u0 = p.total_units * blockIdx.x / gridDim.x;
    u1 = p.total_units * (blockIdx.x + 1) / gridDim.x;
  }
  const long long count = u1 - u0;

  DSA_TS_DECL;
  if (threadIdx.x == 0) DSA_TS(0);
  // the first block resets the call's device status word (no memset needed)
  if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) *p.status = 0u;
  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->bfull[i], 1);
      mbar_init(&bars->bempty[i], 1);
    }
    for (int i = 0; i < kMaxAcc; ++i) {
      mbar_init(&bars->accfull[i], 1);
      // the 4 warps of the group that owns the tile, or every epilogue warp
      mbar_init(&bars->accempty[i], C::QSPLIT ? 4 * C::NG : 4);
    }
    mbar_init(&bars->done, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  // Producer state (thread 0).
  struct ProducerState {
    UnitCursor c;
    int pb, pqb, nblk;
    long long i, issued;
    int s;         // stage of tile i (i % stages, kept as a running counter)
    uint32_t r;    // round of tile i (i / stages)
  } ps{};
  const bool paged = p.pg.table != nullptr;
  auto produce = [&](long long limit) {
    for (; ps.i < limit; ++ps.i) {
      UnitCursor& c = ps.c;
      if (c.b != ps.pb || c.qb != ps.pqb) {
        const int bi = ps.nblk & 1;
        if (ps.nblk >= 2 &&
            !mbar_wait_bounded<kIdxNap>(&bars->bempty[bi], ((ps.nblk >> 1) - 1) & 1, abort_flag, p.wait_budget))
          return;
        mbar_arrive_expect_tx(&bars->bfull[bi], C::kBBytes);
        tma_load_2d(sB + bi * C::kBBytes, &tm_qI, &bars->bfull[bi], 0,
                    (c.b * p.S + c.qb * QB) * DSA_IDX_HEADS);
        ++ps.nblk;
        ps.pb = c.b;
        ps.pqb = c.qb;
      }
      const int s = ps.s;
      if (ps.r > 0 && !mbar_wait_bounded<kIdxNap>(&bars->empty[s], (ps.r - 1) & 1u, abort_flag, p.wait_budget)) return;
      mbar_arrive_expect_tx(&bars->full[s], kATileBytes);
      // a 128-key tile never straddles a cache block (block sizes are
      // multiples of 128); an entry outside the pool reads block 0 (the
      // attention reports it when it gathers from that block)
      bool bad = false;
      const int row = !paged ? c.b * p.cap + c.kt * kKeyTile
                             : static_cast<int>(cache_row(p.pg, c.b, p.cap, c.kt * kKeyTile, &bad));
      tma_load_2d(sA + s * kATileBytes, &tm_kI, &bars->full[s], 0, row);
      ++ps.issued;
      if (++ps.s == stages) {
        ps.s = 0;
        ++ps.r;
      }
      advance_unit(p, c);
    }
  };
  if (warp == 1) tmem_alloc(&bars->tmem_base, C::kTmemCols);
  if constexpr (HIST) {
    for (int i = threadIdx.x; i < QB * kHistBins; i += C::kThreads) sHist[i] = 0u;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_base;
  pdl_trigger();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && count > 0) {
      tma_prefetch_desc(&tm_kI);
      tma_prefetch_desc(&tm_qI);
      ps.c = locate_unit(p, u0);
      ps.pb = -1;
      ps.pqb = -1;
      produce(count);
      if (*abort_flag) {
        // let the copies still in flight land before the CTA can exit
        const long long first = ps.issued > stages ? ps.issued - stages : 0;
        for (long long i = first; i < ps.issued; ++i)
          mbar_drain(&bars->full[i % stages], static_cast<uint32_t>((i / stages) & 1));
        for (int k = 0; k < ps.nblk && k < 2; ++k) {
          const int blk = ps.nblk - 1 - k;
          mbar_drain(&bars->bfull[blk & 1], (blk >> 1) & 1);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && count > 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kKeyTile, N);
      UnitCursor c = locate_unit(p, u0);
      int pb = -1, pqb = -1, nblk = 0, bi = 0;
      int s = 0;           // stage of tile i, running
      uint32_t round = 0;  // i / stages, running
      for (long long i = 0; i < count; ++i) {
        if (c.b != pb || c.qb != pqb) {
          if (nblk > 0) tc_commit(&bars->bempty[bi]);
          bi = nblk & 1;
          if (!mbar_wait_bounded<kIdxNap>(&bars->bfull[bi], (nblk >> 1) & 1, abort_flag, p.wait_budget)) break;
          ++nblk;
          pb = c.b;
          pqb = c.qb;
        }
        if (!mbar_wait_bounded<kIdxNap>(&bars->full[s], round & 1u, abort_flag, p.wait_budget)) break;
        if (i == 0) DSA_TS(1);
        if (i == count - 1) DSA_TS(2);
        const int a = static_cast<int>(i % C::NACC);
        if (i >= C::NACC &&
            !mbar_wait_bounded<kIdxNap>(&bars->accempty[a], static_cast<uint32_t>(((i / C::NACC) - 1) & 1), abort_flag, p.wait_budget))
          break;
        tc_fence_after();
        const uint32_t d = tmem_base + a * N;
        const uint32_t a_addr = smem_u32(sA + s * kATileBytes);
        const uint32_t b_addr = smem_u32(sB + bi * C::kBBytes);
#pragma unroll
        for (int k = 0; k < DSA_IDX_DIM / 16; ++k)
          tc_mma_f16(d, desc_kmajor_sw128(a_addr + 32 * k), desc_kmajor_sw128(b_addr + 32 * k),
                     idesc, k > 0 ? 1u : 0u);
        tc_commit(&bars->empty[s]);
        tc_commit(&bars->accfull[a]);
        advance_unit(p, c);
        if (++s == stages) {
          s = 0;
          ++round;
        }
      }
      // every MMA this CTA issued must finish before tensor memory is freed
      tc_commit(&bars->done);
      mbar_drain(&bars->done, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Groups of 4 warps, each covering all 4 TMEM lane quarters: they take
    // alternate tiles (group = tile index parity) or, with QSPLIT, queries
    // q0 .. q0 + QPG - 1 of every tile.
    constexpr int QPG = C::QPG;
    const int et = threadIdx.x - 64;            // 0 .. kEpiThreads - 1
    const int group = (warp - 2) >> 2;
    const int q0 = C::QSPLIT ? group * QPG : 0;
    const int quarter = warp & 3;               // TMEM lanes 32*quarter ..
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    float* wv_warp = sW + (warp - 2) * QPG * DSA_IDX_HEADS;
    UnitCursor c = count > 0 ? locate_unit(p, u0) : UnitCursor{p.B, 0, 0, 0};
    const int hist_b = c.b;
    int pb = -1, pqb = -1;
    // Split-query groups keep their queries' head weights in registers,
    // reloaded when the block changes: a warp-wide broadcast of 16 bytes from
    // shared memory takes several shared-pipe wavefronts, and per tile those
    // reads would outrun the MMA.
    float wreg[C::QSPLIT ? QPG : 1][16];

    // No CTA-wide barrier inside this loop: a bounded wait that gives up
    // leaves the loop early, and every epilogue thread still reaches the
    // single named barrier after it exactly once.
    for (long long i = 0; i < count; ++i) {
      if (c.b != pb || c.qb != pqb) {
        __syncwarp();
        for (int j = lane; j < QPG * DSA_IDX_HEADS; j += 32) {
          const int s = c.qb * QB + q0 + j / DSA_IDX_HEADS;
          wv_warp[j] = s < p.S
              ? p.w[(static_cast<size_t>(c.b) * p.S + s) * DSA_IDX_HEADS + (j % DSA_IDX_HEADS)]
              : 0.0f;
        }
        __syncwarp();
        if constexpr (C::QSPLIT) {
#pragma unroll
          for (int g = 0; g < QPG; ++g)
#pragma unroll
            for (int h = 0; h < DSA_IDX_HEADS; ++h) wreg[g][h] = (h < kAbsHeads ? 0.5f : 1.0f) * wv_warp[g * DSA_IDX_HEADS + h];
        }
        pb = c.b;
        pqb = c.qb;
      }
      if (!C::QSPLIT && (i & 1) != group) {
        advance_unit(p, c);
        continue;
      }
      const int a = static_cast<int>(i % C::NACC);
      // every lane of the warp leaves together (tcgen05.ld below is warp-wide)
      if (!__all_sync(0xffffffffu, mbar_wait_bounded<kIdxNap>(&bars->accfull[a], static_cast<uint32_t>((i / C::NACC) & 1),
                                                     abort_flag, p.wait_budget)))
        break;
      tc_fence_after();
      const int t = c.kt * kKeyTile + quarter * 32 + lane;
      const int T = p.lens.T[c.b];
      float* srow = p.scores + (static_cast<size_t>(c.b) * p.S + c.qb * QB + q0) * p.cap + t;
      const uint32_t acc_addr = tmem_base + lane_addr + a * N + q0 * 16;
      // this key is kept for the warp's queries j in [jlo, jhi): query
      // s0 + j exists (s < S) and sees key t (t < T - S + s + 1)
      const int s0 = c.qb * QB + q0;
      const int jlo = t - (T - p.S) - s0;
      const int jhi = p.S - s0;
      // weighted head sum of query column group jq (buffer vb), then store
      auto finish = [&](const float (&vb)[C::QG][16], int jq) {
#pragma unroll
        for (int g = 0; g < C::QG; ++g) {
          float acc;
          if constexpr (C::QSPLIT) acc = relu_weighted_sum_r(vb[g], wreg[jq + g]);
          else acc = relu_weighted_sum(vb[g], wv_warp + (jq + g) * DSA_IDX_HEADS);
          // queries past S (padding of the last block) are computed, not kept
          const bool valid = jq + g >= jlo && jq + g < jhi;
          if (valid) srow[static_cast<size_t>(jq + g) * p.cap] = acc;
          if constexpr (HIST) {
            // plain shared atomics: cheaper than warp-aggregating each update
            if (valid) atomicAdd(&sHist[(q0 + jq + g) * kHistBins + (float_key(acc) >> (32 - kHistBits))], 1u);
          }
        }
      };
      float v0[C::QG][16], v1[C::QG][16];
#pragma unroll
      for (int g = 0; g < C::QG; ++g) tmem_ld16(acc_addr + g * 16, v0[g]);
      tmem_ld_wait();
#pragma unroll
      for (int jq = 0; jq < QPG; jq += 2 * C::QG) {
        // buffer v0 holds group jq; load jq + QG into v1 while v0 is summed
        if (jq + C::QG < QPG) {
#pragma unroll
          for (int g = 0; g < C::QG; ++g) tmem_ld16(acc_addr + (jq + C::QG + g) * 16, v1[g]);
        }
        finish(v0, jq);
        tmem_ld_wait();
        if (jq + C::QG < QPG) {
          if (jq + 2 * C::QG < QPG) {
#pragma unroll
            for (int g = 0; g < C::QG; ++g) tmem_ld16(acc_addr + (jq + 2 * C::QG + g) * 16, v0[g]);
          }
          finish(v1, jq + C::QG);
          tmem_ld_wait();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->accempty[a]);
      advance_unit(p, c);
    }
    if (et == 0) DSA_TS(3);
    if constexpr (HIST) {
      // one query block per CTA here (see the unit ranges above); the global
      // histograms were cleared by the previous kernel of the call
      pdl_wait();
      if (et == 0) DSA_TS(4);
      named_bar_sync(1, C::kEpiThreads);
      if (count > 0) {
        for (int j = 0; j < QB; ++j) {
          const int s = j;
          if (s >= p.S) break;
          uint32_t* g = p.hist + static_cast<size_t>(hist_b * p.S + s) * kHistBins;
          for (int bin = et; bin < kHistBins; bin += C::kEpiThreads) {
            const uint32_t v = sHist[j * kHistBins + bin];
            if (v) atomicAdd(g + bin, v);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::kTmemCols);
  if (threadIdx.x == 0 && bars->abort_flag) atomicOr(p.status, kDevTimeout);
  if (threadIdx.x == 0) DSA_TS(5);
  DSA_TS_FLUSH(p.status, 0);
}

// Clears call scratch (histograms, tickets, counters). It lets the next
// kernel launch at once; that kernel waits for it only where it needs zeros.
__global__ void zero_scratch_kernel(uint4* base, long long n16) {
  DSA_TS_DECL;
  if (threadIdx.x == 0) DSA_TS(0);
  pdl_trigger();
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n16;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    base[i] = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) DSA_TS(1);
  DSA_TS_FLUSH(reinterpret_cast<uint8_t*>(base) - 256, 3);
}

cudaError_t launch_zero_scratch(void* base, size_t bytes, cudaStream_t stream) {
  const long long n16 = static_cast<long long>(bytes / 16);
  const int blocks = static_cast<int>(n16 / 256 + 1 < 64 ? n16 / 256 + 1 : 64);
  return launch_kernel("zero_scratch_kernel", zero_scratch_kernel, dim3(blocks), dim3(256), 0, stream, false,
                       static_cast<uint4*>(base), n16);
}

size_t indexer_smem_bytes(int QB, bool with_hist, int* stages_out, size_t smem_limit) {
  const int N = QB * 16;
  size_t ob, ow, oh, obar;
  int stages = kIdxMaxStages;
  if (with_hist && QB >= 8) stages = 6;
  while (stages > 2 && indexer_smem_layout(N, with_hist, stages, &ob, &ow, &oh, &obar) > smem_limit)
    --stages;
  *stages_out = stages;
  return indexer_smem_layout(N, with_hist, stages, &ob, &ow, &oh, &obar);
}

template <int N, bool HIST>
static cudaError_t launch_n(const IndexerParams& p, const CUtensorMap& tm_kI,
                            const CUtensorMap& tm_qI, dim3 grid, size_t smem, int stages,
                            cudaStream_t stream) {
  auto kern = indexer_tc_kernel<N, HIST>;
  cudaError_t e = set_max_smem(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // with histograms the kernel follows the scratch-clearing kernel and waits
  // for it only before its final flush
  return launch_kernel("indexer_tc_kernel", kern, grid, dim3(IdxCfg<N, HIST>::kThreads), smem, stream, HIST, tm_kI,
                       tm_qI, p, stages);
}

cudaError_t launch_indexer(const IndexerParams& p, const CUtensorMap& tm_kI,
                           const CUtensorMap& tm_qI, dim3 grid, size_t smem, int stages,
                           cudaStream_t stream) {
  const bool hist = p.hist != nullptr;
  switch (p.QB) {
#define DSA_IDX_CASE(QBV)                                                                  \
  case QBV:                                                                                \
    return hist ? launch_n<QBV * 16, true>(p, tm_kI, tm_qI, grid, smem, stages, stream)   \
                : launch_n<QBV * 16, false>(p, tm_kI, tm_qI, grid, smem, stages, stream);
    DSA_IDX_CASE(1)
    DSA_IDX_CASE(2)
    DSA_IDX_CASE(4)
    DSA_IDX_CASE(8)
    DSA_IDX_CASE(16)
#undef DSA_IDX_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace dsa
