// Exact radix top-k over fp32 scores.
//
// PR #33802 "... for SM12x and 256K context", Summary item 2: the pages'
// selection is a radix-histogram partial top-k per 2,048-key chunk (histogram
// updates aggregated per warp with __match_any_sync) followed by one
// single-launch final merge-and-emit kernel. With top_k = 2,048 equal to the
// chunk size a per-chunk top-k prunes nothing, so here the chunks build ONE
// global radix histogram per query row and the selection is a global radix
// select:
//
//   1. histogram of the top 11 bits of every visible key (fused into the
//      indexer epilogue in decode; topk_hist_kernel for dsa_topk);
//   2. topk_chunk_select_kernel, one CTA per (chunk, row): every CTA finds the
//      threshold bin from the row histogram, writes its chunk's "certainly
//      selected" bits into a selection bitmap and appends the threshold-bin
//      candidates to a list; the last CTA of the row to finish (an atomic
//      ticket, no waiting) resolves the candidates exactly (radix select over
//      64-bit (key, ~index) composites, so equal scores go to the lower index)
//      and emits the selected indices in ascending order from the bitmap;
//   3. topk_row_kernel: when there are many rows and each fits in shared
//      memory (prefill), one CTA per row runs the whole radix select in
//      shared memory and emits with block scans.
//
// Keys: float_key() maps fp32 to an order-preserving uint32 (-0.0 == +0.0).
#include <cooperative_groups.h>

#include "dsa_common.cuh"
#include "dsa_internal.h"
#include "sm100_ptx.cuh"

namespace dsa {

constexpr int kHistThreads = 256;
constexpr int kSelThreads = 512;
constexpr int kRowThreads = 1024;
constexpr int kCandSmem = 6144;   // candidates resolved from shared memory up to this many

struct RowInfo {
  int n, keff;
};

__device__ __forceinline__ RowInfo row_info(const TopkParams& p, int r) {
  const int b = r / p.S, s = r % p.S;
  RowInfo ri;
  ri.n = visible_len(p.lens.T[b], p.S, s);
  ri.keff = min(p.k, ri.n);
  return ri;
}

// Warp-aggregated shared-memory histogram increment (lanes with equal bins
// add once); bin == 0xFFFFFFFF marks an inactive lane. All lanes call.
__device__ __forceinline__ void hist_add_warp(uint32_t* h, uint32_t bin) {
  const uint32_t peers = __match_any_sync(0xffffffffu, bin);
  if (bin != 0xFFFFFFFFu && (threadIdx.x & 31) == __ffs(peers) - 1)
    atomicAdd(&h[bin], static_cast<uint32_t>(__popc(peers)));
}

// ---------------------------------------------------------------------------
// 1. chunk histograms -> one histogram per row (top 11 key bits)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kHistThreads) topk_hist_kernel(const TopkParams p) {
  __shared__ uint32_t h[kHistBins];
  const int rl = blockIdx.y, r = p.row0 + rl, c = blockIdx.x;
  pdl_trigger();
  const RowInfo ri = row_info(p, r);
  const int t0 = c * kChunk;
  if (t0 >= ri.n) return;
  for (int i = threadIdx.x; i < kHistBins; i += kHistThreads) h[i] = 0u;
  __syncthreads();
  const float* row = p.scores + static_cast<size_t>(r) * p.cap;
  for (int j = threadIdx.x; j < kChunk; j += kHistThreads) {
    const int t = t0 + j;
    const uint32_t bin = t < ri.n ? (float_key(row[t]) >> (32 - kHistBits)) : 0xFFFFFFFFu;
    hist_add_warp(h, bin);
  }
  __syncthreads();
  uint32_t* g = p.hist + static_cast<size_t>(rl) * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += kHistThreads)
    if (h[i]) atomicAdd(g + i, h[i]);
}

// ---------------------------------------------------------------------------
// Exact select among candidate composites (key << 32 | ~index), all sharing
// the top 11 key bits `bin`: marks the `need` largest in the row bitmap.
// `cands` may point to shared or global memory.
// ---------------------------------------------------------------------------
__device__ void resolve_candidates(const unsigned long long* cands, int count, uint32_t bin,
                                   uint32_t need, uint32_t* bitmap_row, uint32_t* hist,
                                   uint32_t* warp_tot, int* sd, uint32_t* sabove,
                                   uint32_t* scnt) {
  unsigned long long prefix = static_cast<unsigned long long>(bin) << 53;
  unsigned long long mask = ~0ull << 53;
  int hi = 52;
  while (hi >= 0) {
    const int w = hi + 1 < 11 ? hi + 1 : 11;
    const int sh = hi - w + 1;
    const uint32_t dm = (1u << w) - 1u;
    for (int i = threadIdx.x; i < (1 << w); i += kSelThreads) hist[i] = 0u;
    __syncthreads();
    const int cround = ((count + 31) / 32) * 32;   // whole warps take part
    for (int i = threadIdx.x; i < cround; i += kSelThreads) {
      uint32_t d = 0xFFFFFFFFu;
      if (i < count) {
        const unsigned long long cc = cands[i];
        if ((cc & mask) == prefix) d = static_cast<uint32_t>(cc >> sh) & dm;
      }
      hist_add_warp(hist, d);
    }
    __syncthreads();
    if (threadIdx.x == 0) { *sd = 0; *sabove = 0; *scnt = 0; }
    __syncthreads();
    find_threshold_digit<kSelThreads>(hist, 1 << w, need, warp_tot, sd, sabove, scnt);
    const uint32_t d = static_cast<uint32_t>(*sd);
    need -= *sabove;
    prefix |= static_cast<unsigned long long>(d) << sh;
    mask |= static_cast<unsigned long long>(dm) << sh;
    const bool all = (*scnt == need);
    __syncthreads();
    if (all) break;
    hi -= w;
  }
  // selected: determined bits >= the threshold prefix
  for (int i = threadIdx.x; i < count; i += kSelThreads) {
    const unsigned long long cc = cands[i];
    if ((cc & mask) >= prefix) {
      const uint32_t t = 0xFFFFFFFFu - static_cast<uint32_t>(cc & 0xFFFFFFFFull);
      atomicOr(&bitmap_row[t >> 5], 1u << (t & 31));
    }
  }
}

// Emit the set bits of bitmap words [0, nwords) as ascending indices into
// out[0 ..), then -1 up to k.
__device__ void emit_bitmap(const uint32_t* bitmap_row, int nwords, int32_t* out, int keff,
                            int k, uint32_t* warp_tot) {
  const int per = (nwords + kSelThreads - 1) / kSelThreads;
  const int w0 = threadIdx.x * per;
  uint32_t cnt = 0;
  for (int j = 0; j < per; ++j) {
    const int wi = w0 + j;
    if (wi < nwords) cnt += __popc(__ldcg(bitmap_row + wi));
  }
  uint32_t total;
  uint32_t pos = block_exclusive_scan<kSelThreads>(cnt, warp_tot, &total);
  for (int j = 0; j < per; ++j) {
    const int wi = w0 + j;
    if (wi >= nwords) break;
    uint32_t bits = __ldcg(bitmap_row + wi);
    while (bits) {
      const int bpos = __ffs(bits) - 1;
      bits &= bits - 1;
      if (pos < static_cast<uint32_t>(keff)) out[pos] = wi * 32 + bpos;
      ++pos;
    }
  }
  for (int i = keff + threadIdx.x; i < k; i += kSelThreads) out[i] = -1;
}

// ---------------------------------------------------------------------------
// 2. per-chunk select + last-CTA merge-and-emit
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSelThreads) topk_chunk_select_kernel(const TopkParams p) {
  extern __shared__ unsigned long long s_cands[];   // kCandSmem entries
  __shared__ uint32_t h[kHistBins];
  __shared__ uint32_t warp_tot[32];
  __shared__ int s_d;
  __shared__ uint32_t s_above, s_cnt;
  __shared__ int s_last;
  __shared__ uint32_t s_cbase;

  const int rl = blockIdx.y, r = p.row0 + rl, c = blockIdx.x;
  pdl_wait();      // scores and histograms come from the previous kernel
  pdl_trigger();
  const RowInfo ri = row_info(p, r);
  const int nch = (ri.n + kChunk - 1) / kChunk;
  if (c >= nch) return;

  // threshold bin of the row from its histogram
  const uint32_t* gh = p.hist + static_cast<size_t>(rl) * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) h[i] = __ldcg(gh + i);
  if (threadIdx.x == 0) { s_d = 0; s_above = 0; s_cnt = 0; }
  __syncthreads();
  find_threshold_digit<kSelThreads>(h, kHistBins, static_cast<uint32_t>(ri.keff), warp_tot, &s_d,
                                    &s_above, &s_cnt);
  const uint32_t bin = static_cast<uint32_t>(s_d);
  const uint32_t need = static_cast<uint32_t>(ri.keff) - s_above;
  const bool take_all = (need == s_cnt);

  // scan the chunk: bitmap words for sure keys, candidates for the threshold
  // bin. Each warp covers kChunk / 16 = 128 keys in 4 groups of 32; the
  // candidate slots of the whole CTA are reserved with one atomic.
  const float* row = p.scores + static_cast<size_t>(r) * p.cap;
  uint32_t* bm = p.bitmap + static_cast<size_t>(rl) * p.bitmap_stride;
  unsigned long long* cl = p.cands + static_cast<size_t>(rl) * p.cand_stride;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t_end = min(ri.n, (c + 1) * kChunk);
  constexpr int kGroups = kChunk / kSelThreads;   // 4
  uint32_t keys[kGroups], cmask[kGroups];
  uint32_t wcount = 0;
#pragma unroll
  for (int gi = 0; gi < kGroups; ++gi) {
    const int base = c * kChunk + gi * kSelThreads + warp * 32;
    const int t = base + lane;
    bool sel = false, cand = false;
    uint32_t key = 0;
    if (t < t_end) {
      key = float_key(row[t]);
      const uint32_t kb = key >> (32 - kHistBits);
      sel = kb > bin || (take_all && kb == bin);
      cand = !take_all && kb == bin;
    }
    const uint32_t word = __ballot_sync(0xffffffffu, sel);
    if (lane == 0 && base < ri.n) bm[base >> 5] = word;
    keys[gi] = key;
    cmask[gi] = __ballot_sync(0xffffffffu, cand);
    wcount += __popc(cmask[gi]);
  }
  uint32_t ctotal;
  const uint32_t wbefore =
      block_exclusive_scan<kSelThreads>(lane == 0 ? wcount : 0u, warp_tot, &ctotal);
  if (threadIdx.x == 0 && ctotal) s_cbase = atomicAdd(&p.cand_count[rl], ctotal);
  __syncthreads();
  if (ctotal) {
    uint32_t pos = s_cbase + __shfl_sync(0xffffffffu, wbefore, 0);
#pragma unroll
    for (int gi = 0; gi < kGroups; ++gi) {
      const uint32_t cm = cmask[gi];
      if ((cm >> lane) & 1u) {
        const int t = c * kChunk + gi * kSelThreads + warp * 32 + lane;
        cl[pos + __popc(cm & ((1u << lane) - 1u))] =
            (static_cast<unsigned long long>(keys[gi]) << 32) |
            static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(t));
      }
      pos += __popc(cm);
    }
  }

  // ticket: the last CTA of the row finishes the selection
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t prev = atomicAdd(&p.ticket[rl], 1u);
    s_last = (prev == static_cast<uint32_t>(nch - 1));
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  if (!take_all) {
    const int count = static_cast<int>(__ldcg(&p.cand_count[rl]));
    const unsigned long long* src = cl;
    if (count <= kCandSmem) {
      for (int i = threadIdx.x; i < count; i += kSelThreads) s_cands[i] = __ldcg(cl + i);
      __syncthreads();
      src = s_cands;
    }
    resolve_candidates(src, count, bin, need, bm, h, warp_tot, &s_d, &s_above, &s_cnt);
    __threadfence();
    __syncthreads();
  }
  emit_bitmap(bm, (ri.n + 31) / 32, p.idx + static_cast<size_t>(r) * p.k, ri.keff, p.k,
              warp_tot);
}

// ---------------------------------------------------------------------------
// 3. whole-row select in shared memory (one CTA per row)
// ---------------------------------------------------------------------------
int topk_row_max_len(size_t smem_limit) {
  const size_t fixed = (kHistBins + 64) * sizeof(uint32_t) + 1024;
  if (smem_limit <= fixed) return 0;
  return static_cast<int>(((smem_limit - fixed) / sizeof(uint32_t)) & ~size_t(3));
}

__global__ void __launch_bounds__(kRowThreads) topk_row_kernel(const TopkParams p) {
  extern __shared__ uint32_t skeys[];          // n keys, then the histogram
  __shared__ uint32_t warp_tot[32];
  __shared__ int s_d;
  __shared__ uint32_t s_above, s_cnt;

  const int r = blockIdx.x;
  pdl_wait();      // scores come from the previous kernel
  pdl_trigger();
  const RowInfo ri = row_info(p, r);
  const int n = ri.n;
  uint32_t* h = skeys + ((n + 3) & ~3);
  const float* row = p.scores + static_cast<size_t>(r) * p.cap;
  for (int i = threadIdx.x; i < n; i += kRowThreads) skeys[i] = float_key(row[i]);
  const int nround = ((n + 31) / 32) * 32;

  uint32_t prefix = 0, mask = 0, need = static_cast<uint32_t>(ri.keff);
  bool all = false;
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
  for (int pass = 0; pass < 3 && !all; ++pass) {
    const int sh = shifts[pass], w = widths[pass];
    const uint32_t dm = (1u << w) - 1u;
    for (int i = threadIdx.x; i < (1 << w); i += kRowThreads) h[i] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < nround; i += kRowThreads) {
      uint32_t d = 0xFFFFFFFFu;
      if (i < n) {
        const uint32_t key = skeys[i];
        if ((key & mask) == prefix) d = (key >> sh) & dm;
      }
      hist_add_warp(h, d);
    }
    __syncthreads();
    if (threadIdx.x == 0) { s_d = 0; s_above = 0; s_cnt = 0; }
    __syncthreads();
    find_threshold_digit<kRowThreads>(h, 1 << w, need, warp_tot, &s_d, &s_above, &s_cnt);
    need -= s_above;
    prefix |= static_cast<uint32_t>(s_d) << sh;
    mask |= dm << sh;
    all = (s_cnt == need);
    __syncthreads();
  }
  // keys above the threshold are selected; keys equal to it are selected in
  // index order until `need` of them are taken (all of them when `all`)
  const uint32_t eq_limit = all ? 0xFFFFFFFFu : need;
  int32_t* out = p.idx + static_cast<size_t>(r) * p.k;
  uint32_t eq_run = 0, sel_run = 0;
  for (int tile = 0; tile < n; tile += 4 * kRowThreads) {
    const int i0 = tile + 4 * threadIdx.x;
    uint32_t gt = 0, eq = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = i0 + j;
      if (i < n) {
        const uint32_t km = skeys[i] & mask;
        if (km > prefix) gt |= 1u << j;
        else if (km == prefix) eq |= 1u << j;
      }
    }
    uint32_t eq_tot;
    uint32_t eq_before = eq_run + block_exclusive_scan<kRowThreads>(__popc(eq), warp_tot, &eq_tot);
    uint32_t sel = gt;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if ((eq >> j) & 1u) {
        if (eq_before < eq_limit) sel |= 1u << j;
        ++eq_before;
      }
    uint32_t sel_tot;
    uint32_t pos = sel_run + block_exclusive_scan<kRowThreads>(__popc(sel), warp_tot, &sel_tot);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if ((sel >> j) & 1u) {
        if (pos < static_cast<uint32_t>(ri.keff)) out[pos] = i0 + j;
        ++pos;
      }
    eq_run += eq_tot;
    sel_run += sel_tot;
  }
  for (int i = ri.keff + threadIdx.x; i < p.k; i += kRowThreads) out[i] = -1;
}

constexpr int kClThreads = 512;   // cluster select CTA size with 32 keys a thread (1,024 with 8 to 24)
// Candidates gathered into every CTA of the cluster: 8,192, or 4,096 for the
// shortest slices, whose CTAs then fit two to an SM (many short rows, as in
// grouped decode, run in one wave), or 3,072 with 24 keys a thread, whose
// 24,576-key slice leaves no more room. The first 16 KB of the gathered list
// also hold the cluster's histogram exchange, which is over before any
// candidate is gathered.
__host__ __device__ constexpr int cl_gather_max(int per) { return per <= 8 ? 4096 : per == 24 ? 3072 : 8192; }

// Exact threshold over a list of candidate composites held by this CTA:
// refines (prefix, mask) until `need` candidates are at or above it.
// `hi` is the highest composite bit not yet fixed by (prefix, mask).
template <int NT>
__device__ void local_composite_select(const unsigned long long* list, int n,
                                       unsigned long long* prefix, unsigned long long* mask,
                                       uint32_t need, uint32_t* h, uint32_t* warp_tot, int* sd,
                                       uint32_t* sabove, uint32_t* scnt, int hi = 52) {
  bool all = false;
  while (!all && hi >= 0) {
    const int w = hi + 1 < 11 ? hi + 1 : 11;
    const int sh = hi - w + 1;
    const uint32_t dm = (1u << w) - 1u;
    for (int i = threadIdx.x; i < (1 << w); i += NT) h[i] = 0u;
    __syncthreads();
    for (int c = threadIdx.x; c < n; c += NT) {
      const unsigned long long cc = list[c];
      if ((cc & *mask) == *prefix) atomicAdd(&h[static_cast<uint32_t>(cc >> sh) & dm], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) { *sd = 0; *sabove = 0; *scnt = 0; }
    __syncthreads();
    find_threshold_digit<NT>(h, 1 << w, need, warp_tot, sd, sabove, scnt);
    need -= *sabove;
    *prefix |= static_cast<unsigned long long>(*sd) << sh;
    *mask |= static_cast<unsigned long long>(dm) << sh;
    all = (*scnt == need);
    __syncthreads();
    hi -= w;
  }
}

// Refines the threshold among n composites in shared memory whose bits above
// `hi` are fixed by prefix/mask, 11 bits per round: the block histograms the
// composites that match the prefix and scans it for the digit. `hbuf` is
// 2,048 words of shared scratch, `warp_tot` the block scan's.
template <int NT>
__device__ void resolve_composites(const unsigned long long* list, int n, unsigned long long* prefix,
                                   unsigned long long* mask, uint32_t need, uint32_t* hbuf,
                                   uint32_t* warp_tot, int* sd, uint32_t* sabove, uint32_t* scnt,
                                   int hi) {
  bool all = false;
  while (!all && hi >= 0) {
    const int w = hi + 1 < 11 ? hi + 1 : 11;
    const int sh = hi - w + 1;
    const uint32_t dm = (1u << w) - 1u;
    for (int i = threadIdx.x; i < kHistBins; i += NT) hbuf[i] = 0u;
    __syncthreads();   // every thread is also past the previous round's reads
    if (threadIdx.x == 0) { *sd = 0; *sabove = 0; *scnt = 0; }
    for (int c = threadIdx.x; c < n; c += NT) {
      const unsigned long long cc = list[c];
      if ((cc & *mask) == *prefix) atomicAdd(&hbuf[static_cast<uint32_t>(cc >> sh) & dm], 1u);
    }
    __syncthreads();
    find_threshold_digit<NT>(hbuf, 1 << w, need, warp_tot, sd, sabove, scnt);
    need -= *sabove;
    *prefix |= static_cast<unsigned long long>(*sd) << sh;
    *mask |= static_cast<unsigned long long>(dm) << sh;
    all = (*scnt == need);
    hi -= w;
  }
}

// ---------------------------------------------------------------------------
// 3b. whole-row select with the keys in registers (one CTA of 640 threads per
// row, up to 64 keys per thread: 40,960 keys). Warp w owns keys
// [w * 32 * PER, (w + 1) * 32 * PER) and lane l
// holds key w * 32 * PER + 32 * i + l in key[i]. A sample of the row (every
// 16th key) gives a provisional threshold theta a little below the k-th key;
// the keys at or above theta (a few thousand) are resolved exactly in shared
// memory. If the sample misleads (fewer than k keys at or above theta, or too
// many), the threshold is found by radix passes over all keys instead. The
// selection is emitted in index order with one scan over the warps' counts.
// ---------------------------------------------------------------------------
constexpr int kRrThreads = 640;   // 20 warps; at most ~100 registers each, keys included
constexpr int kRrWarps = kRrThreads / 32;
constexpr int kRrCandMax = 4096;
constexpr int kRrMaxPer = 64;

template <int PER>
__global__ void __launch_bounds__(kRrThreads, 1) topk_row_reg_kernel(const TopkParams p) {
  __shared__ uint32_t h[kHistBins];
  __shared__ unsigned long long scand[kRrCandMax];
  __shared__ uint32_t warp_tot[32];
  __shared__ uint32_t s_wcnt[kRrWarps];
  __shared__ int s_d;
  __shared__ uint32_t s_above, s_cnt;

  const int r = blockIdx.x;
  pdl_wait();      // scores come from the previous kernel
  pdl_trigger();
  const RowInfo ri = row_info(p, r);
  const int n = ri.n, keff = ri.keff;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int wbase = warp * 32 * PER;
  const float* row = p.scores + static_cast<size_t>(r) * p.cap;
  uint32_t key[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int t = wbase + 32 * i + lane;
    key[i] = t < n ? float_key(__ldcg(row + t)) : 0u;
  }
  auto valid = [&](int i) { return wbase + 32 * i + lane < n; };
  auto comp = [&](int i) {
    return (static_cast<unsigned long long>(key[i]) << 32) |
           (0xFFFFFFFFull - static_cast<uint32_t>(wbase + 32 * i + lane));
  };

  // ---- provisional threshold from a sample
  for (int i = threadIdx.x; i < kHistBins; i += kRrThreads) h[i] = 0u;
  if (threadIdx.x == 0) { s_d = 0; s_above = 0; s_cnt = 0; }
  __syncthreads();
  uint32_t nsmp = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i)
    if (((i + lane) & 15) == 0 && valid(i)) {
      atomicAdd(&h[key[i] >> 21], 1u);
      ++nsmp;
    }
  uint32_t ns;
  block_exclusive_scan<kRrThreads>(nsmp, warp_tot, &ns);
  // target rank in the sample: 25 % and 16 keys of slack above k's share
  uint32_t rs = static_cast<uint32_t>((static_cast<unsigned long long>(keff) * ns * 5 + 4ull * n - 1) /
                                      (4ull * n)) + 16u;
  if (rs > ns) rs = ns;
  uint32_t theta = 0;
  if (rs > 0) {
    find_threshold_digit<kRrThreads>(h, kHistBins, rs, warp_tot, &s_d, &s_above, &s_cnt);
    const uint32_t b1 = static_cast<uint32_t>(s_d);
    const uint32_t need2 = rs - s_above;
    for (int i = threadIdx.x; i < kHistBins; i += kRrThreads) h[i] = 0u;
    // every thread has read the search's outputs before they are reset
    __syncthreads();
    if (threadIdx.x == 0) { s_d = 0; s_above = 0; s_cnt = 0; }
#pragma unroll
    for (int i = 0; i < PER; ++i)
      if (((i + lane) & 15) == 0 && valid(i) && (key[i] >> 21) == b1)
        atomicAdd(&h[(key[i] >> 10) & 0x7FFu], 1u);
    __syncthreads();
    find_threshold_digit<kRrThreads>(h, kHistBins, need2, warp_tot, &s_d, &s_above, &s_cnt);
    theta = (b1 << 21) | (static_cast<uint32_t>(s_d) << 10);
  }
  // ---- keys at or above theta
  uint32_t mine = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) mine += (valid(i) && key[i] >= theta) ? 1u : 0u;
  for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
  if (lane == 0) s_wcnt[warp] = mine;
  __syncthreads();
  uint32_t c = 0, wb = 0;
  for (int w = 0; w < kRrWarps; ++w) {
    if (w == warp) wb = c;
    c += s_wcnt[w];
  }
  unsigned long long prefix = 0ull, mask = 0ull;
  const bool use_cand = c >= static_cast<uint32_t>(keff) && c <= static_cast<uint32_t>(kRrCandMax);
  // only keys at or above theta can be selected on the candidate path (the
  // resolve may stop at a prefix that keys below theta share)
  const uint32_t floor_key = use_cand ? theta : 0u;
  if (use_cand) {
    // few candidates: gather their composites and resolve exactly
    uint32_t off = wb;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const bool f = valid(i) && key[i] >= theta;
      const uint32_t bal = __ballot_sync(0xffffffffu, f);
      if (f) scand[off + __popc(bal & ((1u << lane) - 1u))] = comp(i);
      off += __popc(bal);
    }
    __syncthreads();
    local_composite_select<kRrThreads>(scand, static_cast<int>(c), &prefix, &mask,
                                       static_cast<uint32_t>(keff), h, warp_tot, &s_d, &s_above,
                                       &s_cnt, 63);
  } else {
    // the sample misled: radix passes over every key (11 composite bits each)
    uint32_t need = static_cast<uint32_t>(keff);
    bool all = false;
    int hi = 63;
    while (!all && hi >= 0) {
      const int w = hi + 1 < 11 ? hi + 1 : 11;
      const int sh = hi - w + 1;
      const uint32_t dm = (1u << w) - 1u;
      for (int i = threadIdx.x; i < (1 << w); i += kRrThreads) h[i] = 0u;
      __syncthreads();
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const unsigned long long cc = comp(i);
        const uint32_t dg = (valid(i) && (cc & mask) == prefix)
                                ? static_cast<uint32_t>(cc >> sh) & dm : 0xFFFFFFFFu;
        hist_add_warp(h, dg);
      }
      __syncthreads();
      if (threadIdx.x == 0) { s_d = 0; s_above = 0; s_cnt = 0; }
      __syncthreads();
      find_threshold_digit<kRrThreads>(h, 1 << w, need, warp_tot, &s_d, &s_above, &s_cnt);
      need -= s_above;
      prefix |= static_cast<unsigned long long>(s_d) << sh;
      mask |= static_cast<unsigned long long>(dm) << sh;
      all = (s_cnt == need);
      __syncthreads();
      hi -= w;
    }
  }
  // ---- emit the selection in index order
  __syncthreads();
  mine = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i)
    mine += (valid(i) && key[i] >= floor_key && (comp(i) & mask) >= prefix) ? 1u : 0u;
  for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
  if (lane == 0) s_wcnt[warp] = mine;
  __syncthreads();
  uint32_t pos = 0;
  for (int w = 0; w < warp; ++w) pos += s_wcnt[w];
  int32_t* out = p.idx + static_cast<size_t>(r) * p.k;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const bool f = valid(i) && key[i] >= floor_key && (comp(i) & mask) >= prefix;
    const uint32_t bal = __ballot_sync(0xffffffffu, f);
    const uint32_t at = pos + __popc(bal & ((1u << lane) - 1u));
    if (f && at < static_cast<uint32_t>(keff)) out[at] = wbase + 32 * i + lane;
    pos += __popc(bal);
  }
  for (int i = keff + threadIdx.x; i < p.k; i += kRrThreads) out[i] = -1;
}

// ---------------------------------------------------------------------------
// 3c. streaming whole-row select (many rows: prefill). One CTA of 256 threads
// per row keeps no keys in registers:
//   1. a sample of the row (every 16th 128-byte line, so no extra DRAM
//      sectors) gives a provisional threshold theta a little below the k-th
//      key: its share of keff plus 25 % and 16 keys of slack, resolved on 22
//      key bits of the sample;
//   2. one pass over the row lists the keys at or above theta (composites
//      key << 32 | ~index) in shared memory -- its reads of the sampled lines
//      hit L2;
//   3. the exact keff-th composite among the listed keys is resolved in
//      11-bit rounds (equal keys go to the lower index) and the selected ones
//      are marked in a bitmap of the row in shared memory;
//   4. the bitmap is emitted in index order.
// If the sample misleads (fewer than keff keys at or above theta, or more
// than kRsCandMax), an exact path takes over: a histogram of the row's top 11
// key bits, a pass that marks the keys above the threshold bin and lists the
// bin's keys, and the same resolve (for a bin of more than kRsCandMax keys,
// rounds that re-read the row). Each row's phases are chains of dependent
// loads and block barriers, so throughput comes from rows in flight: with
// ~46 KB of shared memory and at most 64 registers, four 256-thread rows run
// per SM (against two 512-thread rows at 56 registers: 8K-on-32K 563 -> 524
// us; four 512-thread rows at 32 registers 541 us, five 256-thread rows with
// a smaller list 660 us, six 128-thread rows 966 us).
// ---------------------------------------------------------------------------
constexpr int kRsThreads = 256;
constexpr int kRsCandMax = 4096;
constexpr int kRsMaxLen = 262144;
#ifndef RS_UNROLL
#define RS_UNROLL 4
#endif

// Exact threshold among n listed composites whose bits above `hi` are fixed by
// (prefix, mask): refines 11 bits a round until `need` composites are at or
// above the prefix; returns the prefix (zero below its determined bits).
__device__ unsigned long long rs_resolve(const unsigned long long* list, uint32_t n, uint32_t need,
                                         unsigned long long prefix, unsigned long long mask, int hi,
                                         uint32_t* h, uint32_t* warp_tot, int* sd, uint32_t* sabove,
                                         uint32_t* scnt) {
  bool all = false;
  while (!all && hi >= 0) {
    const int w = hi + 1 < 11 ? hi + 1 : 11;
    const int sh = hi - w + 1;
    const uint32_t dm = (1u << w) - 1u;
    for (int i = threadIdx.x; i < kHistBins; i += kRsThreads) h[i] = 0u;
    // every thread has read the previous round's outputs before they are
    // reset (the barrier after the counting orders the reset before the
    // next search)
    __syncthreads();
    if (threadIdx.x == 0) { *sd = 0; *sabove = 0; *scnt = 0; }
    for (uint32_t i = threadIdx.x; i < n; i += kRsThreads) {
      const unsigned long long cc = list[i];
      if ((cc & mask) == prefix) atomicAdd(&h[static_cast<uint32_t>(cc >> sh) & dm], 1u);
    }
    __syncthreads();
    find_threshold_digit<kRsThreads>(h, 1 << w, need, warp_tot, sd, sabove, scnt);
    need -= *sabove;
    prefix |= static_cast<unsigned long long>(*sd) << sh;
    mask |= static_cast<unsigned long long>(dm) << sh;
    all = (*scnt == need);
    hi -= w;
  }
  return prefix;
}

__global__ void __launch_bounds__(kRsThreads, 4) topk_row_stream_kernel(const TopkParams p) {
  extern __shared__ uint32_t rs_bm[];                  // [ceil(n / 32)] selection bits
  __shared__ unsigned long long rs_c[kRsCandMax];      // listed composites
  __shared__ __align__(16) uint32_t h[kHistBins];
  __shared__ uint32_t warp_tot[32];
  __shared__ int s_d;
  __shared__ uint32_t s_above, s_cnt, s_nc;
  const int rl = blockIdx.x, r = p.row0 + rl;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kWarps = kRsThreads / 32;
  DSA_TS_DECL;
  if (threadIdx.x == 0) DSA_TS(0);
  pdl_wait();      // scores come from the previous kernel
  if (threadIdx.x == 0) DSA_TS(1);
  pdl_trigger();
  const RowInfo ri = row_info(p, r);
  const int n = ri.n, keff = ri.keff;
  const int nw = (n + 31) >> 5;
  const float* row = p.scores + static_cast<size_t>(r) * p.cap;
  if (threadIdx.x < 32) {
    // the whole row into L2 at once (the 16-byte-aligned part of it, in
    // 16 KB pieces): the passes below then read at L2 latency
    const uintptr_t a0 = (reinterpret_cast<uintptr_t>(row) + 15) & ~uintptr_t(15);
    const uintptr_t a1 = reinterpret_cast<uintptr_t>(row + n) & ~uintptr_t(15);
    for (uintptr_t a = a0 + static_cast<uintptr_t>(threadIdx.x) * 16384u; a < a1; a += 32u * 16384u)
      prefetch_l2_bulk(reinterpret_cast<const void*>(a), static_cast<uint32_t>(a1 - a < 16384u ? a1 - a : 16384u));
  }
  for (int i = threadIdx.x; i < kHistBins; i += kRsThreads) h[i] = 0u;
  for (int i = threadIdx.x; i < nw; i += kRsThreads) rs_bm[i] = 0u;
  if (threadIdx.x == 0) { s_d = 0; s_above = 0; s_cnt = 0; s_nc = 0; }
  __syncthreads();
  constexpr int U = RS_UNROLL;                         // loads in flight per thread
  auto composite = [](uint32_t k, int t) {
    return (static_cast<unsigned long long>(k) << 32) | (0xFFFFFFFFull - static_cast<uint32_t>(t));
  };

  // ---- 1. provisional threshold from every 16th line (warp w reads lines
  // 16 (w + kWarps j), lane l key l of the line); the first kRsSmpReg sampled
  // keys stay in registers for the second level
  constexpr int kRsSmpReg = 8;
  uint32_t ks[kRsSmpReg];
  uint32_t nsmp = 0;
  const int nlines = nw;
  {
#pragma unroll
    for (int j = 0; j < kRsSmpReg; ++j) {
      const int t = 32 * 16 * (warp + kWarps * j) + lane;
      ks[j] = t < n ? float_key(__ldcg(row + t)) : 0u;
    }
#pragma unroll
    for (int j = 0; j < kRsSmpReg; ++j) {
      const int t = 32 * 16 * (warp + kWarps * j) + lane;
      if (t < n) {
        atomicAdd(&h[ks[j] >> (32 - kHistBits)], 1u);
        ++nsmp;
      }
    }
    for (int j = kRsSmpReg; 16 * (warp + kWarps * j) < nlines; ++j) {
      const int t = 32 * 16 * (warp + kWarps * j) + lane;
      if (t < n) {
        atomicAdd(&h[float_key(__ldcg(row + t)) >> (32 - kHistBits)], 1u);
        ++nsmp;
      }
    }
  }
  uint32_t ns;
  block_exclusive_scan<kRsThreads>(nsmp, warp_tot, &ns);
  uint32_t rs = static_cast<uint32_t>((static_cast<unsigned long long>(keff) * ns * 5 + 4ull * n - 1) /
                                      (4ull * n)) + 16u;
  if (rs > ns) rs = ns;
  uint32_t theta = 0;
  if (rs > 0) {
    find_threshold_digit<kRsThreads>(h, kHistBins, rs, warp_tot, &s_d, &s_above, &s_cnt);
    const uint32_t sb = static_cast<uint32_t>(s_d);
    const uint32_t need2 = rs - s_above;
    for (int i = threadIdx.x; i < kHistBins; i += kRsThreads) h[i] = 0u;
    // every thread has read the search's outputs before they are reset
    __syncthreads();
    if (threadIdx.x == 0) { s_d = 0; s_above = 0; s_cnt = 0; }
#pragma unroll
    for (int j = 0; j < kRsSmpReg; ++j) {
      const int t = 32 * 16 * (warp + kWarps * j) + lane;
      if (t < n && (ks[j] >> (32 - kHistBits)) == sb)
        atomicAdd(&h[(ks[j] >> (32 - 2 * kHistBits)) & (kHistBins - 1)], 1u);
    }
    for (int j = kRsSmpReg; 16 * (warp + kWarps * j) < nlines; ++j) {
      const int t = 32 * 16 * (warp + kWarps * j) + lane;
      if (t < n) {
        const uint32_t k = float_key(__ldcg(row + t));   // an L2 hit: read just above
        if ((k >> (32 - kHistBits)) == sb) atomicAdd(&h[(k >> (32 - 2 * kHistBits)) & (kHistBins - 1)], 1u);
      }
    }
    __syncthreads();
    find_threshold_digit<kRsThreads>(h, kHistBins, need2, warp_tot, &s_d, &s_above, &s_cnt);
    theta = (sb << (32 - kHistBits)) | (static_cast<uint32_t>(s_d) << (32 - 2 * kHistBits));
  }
  if (threadIdx.x == 0) DSA_TS(2);

  // ---- 2. the keys at or above theta into the list: warp w appends to its
  // own region [w * kRsWarpCand, (w + 1) * kRsWarpCand) (count in a register);
  // the next batch's loads are issued before the current batch is examined
  constexpr int kRsWarpCand = kRsCandMax / kWarps;
  unsigned long long* wlist = rs_c + warp * kRsWarpCand;
  uint32_t wcount = 0;
  {
    uint32_t k[U], kn[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = u * kRsThreads + threadIdx.x;
      k[u] = t < n ? float_key(__ldcg(row + t)) : 0u;
    }
    for (int base = 0; base < n; base += U * kRsThreads) {
      const int nb = base + U * kRsThreads;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int t = nb + u * kRsThreads + threadIdx.x;
        kn[u] = t < n ? float_key(__ldcg(row + t)) : 0u;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int t = base + u * kRsThreads + threadIdx.x;
        const bool cand = t < n && k[u] >= theta;
        const uint32_t cb = __ballot_sync(0xffffffffu, cand);
        const uint32_t at = wcount + __popc(cb & ((1u << lane) - 1u));
        if (cand && at < static_cast<uint32_t>(kRsWarpCand)) wlist[at] = composite(k[u], t);
        wcount += __popc(cb);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) k[u] = kn[u];
    }
  }
  if (lane == 0) atomicAdd(&s_nc, wcount);
  __syncthreads();
  if (threadIdx.x == 0) DSA_TS(3);
  const uint32_t nc = s_nc;
  // every warp region held its keys; then keys that are not listed are below theta
  const bool fits = __syncthreads_and(wcount <= static_cast<uint32_t>(kRsWarpCand));
  if (fits && nc >= static_cast<uint32_t>(keff)) {
    // ---- 3. compact the regions, resolve the exact threshold among the
    // listed keys and mark those at or above it
    __shared__ uint32_t s_wc[kWarps];
    if (lane == 0) s_wc[warp] = wcount;
    __syncthreads();
    uint32_t off = 0;
    for (int w = 0; w < warp; ++w) off += s_wc[w];
    // move regions left in order: region w lands at off >= w * kRsWarpCand
    // never below; copy through registers one warp at a time
    for (int w = 1; w < kWarps; ++w) {
      if (warp == w) {
        // batches of 32 (wcount is the same in every lane), every lane in
        // every batch: the reads of a batch land before its writes
        for (uint32_t i0 = 0; i0 < wcount; i0 += 32) {
          const uint32_t i = i0 + lane;
          const unsigned long long v = i < wcount ? wlist[i] : 0ull;
          __syncwarp();
          if (i < wcount) rs_c[off + i] = v;
          __syncwarp();
        }
      }
      __syncthreads();
    }
    const unsigned long long T = rs_resolve(rs_c, nc, static_cast<uint32_t>(keff), 0ull, 0ull, 63, h,
                                            warp_tot, &s_d, &s_above, &s_cnt);
    if (threadIdx.x == 0) DSA_TS(4);
    for (uint32_t i = threadIdx.x; i < nc; i += kRsThreads) {
      const unsigned long long cc = rs_c[i];
      if (cc >= T) {
        const uint32_t t = 0xFFFFFFFFu - static_cast<uint32_t>(cc & 0xFFFFFFFFull);
        atomicOr(&rs_bm[t >> 5], 1u << (t & 31));
      }
    }
  } else {
    // ---- the sample misled: exact path. Histogram of the row's top 11 bits,
    for (int i = threadIdx.x; i < kHistBins; i += kRsThreads) h[i] = 0u;
    if (threadIdx.x == 0) { s_d = 0; s_above = 0; s_cnt = 0; s_nc = 0; }
    __syncthreads();
    for (int base = 0; base < n; base += kRsThreads) {
      const int t = base + threadIdx.x;
      hist_add_warp(h, t < n ? float_key(__ldcg(row + t)) >> (32 - kHistBits) : 0xFFFFFFFFu);
    }
    __syncthreads();
    find_threshold_digit<kRsThreads>(h, kHistBins, static_cast<uint32_t>(keff), warp_tot, &s_d,
                                     &s_above, &s_cnt);
    const uint32_t b1 = static_cast<uint32_t>(s_d);
    const uint32_t need = static_cast<uint32_t>(keff) - s_above;
    const uint32_t n1 = s_cnt;
    const uint32_t lo1 = b1 << (32 - kHistBits);
    const uint32_t hi1 = lo1 + (1u << (32 - kHistBits)) - 1u;
    const bool listed = n1 <= static_cast<uint32_t>(kRsCandMax);
    // keys above bin b1 into the bitmap (warp w of a round: one word), the
    // bin's keys into the list
    for (int base = 0; base < n; base += kRsThreads) {
      const int t = base + threadIdx.x;
      const uint32_t k = t < n ? float_key(__ldcg(row + t)) : 0u;
      const uint32_t word = __ballot_sync(0xffffffffu, t < n && k > hi1);
      if (lane == 0 && t < n) rs_bm[t >> 5] = word;
      if (listed) {
        const bool cand = t < n && k >= lo1 && k <= hi1;
        const uint32_t cb = __ballot_sync(0xffffffffu, cand);
        if (cb) {
          uint32_t slot = 0;
          if (lane == 0) slot = atomicAdd(&s_nc, static_cast<uint32_t>(__popc(cb)));
          slot = __shfl_sync(0xffffffffu, slot, 0);
          if (cand) rs_c[slot + __popc(cb & ((1u << lane) - 1u))] = composite(k, t);
        }
      }
    }
    __syncthreads();
    unsigned long long T = static_cast<unsigned long long>(b1) << 53;   // need == n1: the whole bin
    if (need < n1) {
      if (listed) {
        T = rs_resolve(rs_c, n1, need, T, ~0ull << 53, 52, h, warp_tot, &s_d, &s_above, &s_cnt);
      } else {
        // a heavy tie: rounds that re-read the row
        unsigned long long mask = ~0ull << 53;
        uint32_t nd = need;
        bool all = false;
        int hi = 52;
        while (!all && hi >= 0) {
          const int w = hi + 1 < 11 ? hi + 1 : 11;
          const int sh = hi - w + 1;
          const uint32_t dm = (1u << w) - 1u;
          for (int i = threadIdx.x; i < kHistBins; i += kRsThreads) h[i] = 0u;
          // every thread has read the previous round's outputs before they
          // are reset (the barrier after the counting orders the reset
          // before the next search)
          __syncthreads();
          if (threadIdx.x == 0) { s_d = 0; s_above = 0; s_cnt = 0; }
          for (int base = 0; base < n; base += kRsThreads) {
            const int t = base + threadIdx.x;
            uint32_t dg = 0xFFFFFFFFu;
            if (t < n) {
              const unsigned long long cc = composite(float_key(__ldcg(row + t)), t);
              if ((cc & mask) == T) dg = static_cast<uint32_t>(cc >> sh) & dm;
            }
            hist_add_warp(h, dg);
          }
          __syncthreads();
          find_threshold_digit<kRsThreads>(h, 1 << w, nd, warp_tot, &s_d, &s_above, &s_cnt);
          nd -= s_above;
          T |= static_cast<unsigned long long>(s_d) << sh;
          mask |= static_cast<unsigned long long>(dm) << sh;
          all = (s_cnt == nd);
          hi -= w;
        }
      }
    }
    if (listed) {
      for (uint32_t i = threadIdx.x; i < n1; i += kRsThreads) {
        const unsigned long long cc = rs_c[i];
        if (cc >= T) {
          const uint32_t t = 0xFFFFFFFFu - static_cast<uint32_t>(cc & 0xFFFFFFFFull);
          atomicOr(&rs_bm[t >> 5], 1u << (t & 31));
        }
      }
    } else {
      for (int t = threadIdx.x; t < n; t += kRsThreads) {
        const uint32_t k = float_key(__ldcg(row + t));
        if (k >= lo1 && k <= hi1 && composite(k, t) >= T) atomicOr(&rs_bm[t >> 5], 1u << (t & 31));
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) DSA_TS(5);
  // ---- 4. emit in index order: thread i owns words [i * wpt, (i + 1) * wpt)
  const int wpt = (nw + kRsThreads - 1) / kRsThreads;
  const int w0 = threadIdx.x * wpt;
  uint32_t cnt = 0;
  for (int j = 0; j < wpt; ++j)
    if (w0 + j < nw) cnt += __popc(rs_bm[w0 + j]);
  uint32_t tot;
  uint32_t pos = block_exclusive_scan<kRsThreads>(cnt, warp_tot, &tot);
  int32_t* out = p.idx + static_cast<size_t>(r) * p.k;
  for (int j = 0; j < wpt; ++j) {
    if (w0 + j >= nw) break;
    uint32_t bits = rs_bm[w0 + j];
    while (bits) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1;
      if (pos < static_cast<uint32_t>(keff)) out[pos] = (w0 + j) * 32 + b;
      ++pos;
    }
  }
  for (int i = keff + threadIdx.x; i < p.k; i += kRsThreads) out[i] = -1;
  if (threadIdx.x == 0) DSA_TS(6);
  DSA_TS_FLUSH(p.status, 1);
}

int topk_row_stream_max_len() { return kRsMaxLen; }

cudaError_t launch_topk_row_stream(const TopkParams& p, int max_n, bool pdl, cudaStream_t stream) {
  if (max_n > kRsMaxLen) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>((max_n + 31) / 32) * sizeof(uint32_t);
  cudaError_t e = set_max_smem(reinterpret_cast<const void*>(topk_row_stream_kernel), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_kernel("topk_row_stream_kernel", topk_row_stream_kernel, dim3(p.nrows),
                       dim3(kRsThreads), smem, stream, pdl, p);
}

int topk_row_reg_per(int max_n) {
  const int per = (max_n + kRrThreads - 1) / kRrThreads;
  const int per16 = ((per + 15) / 16) * 16;
  return per16 <= kRrMaxPer ? per16 : 0;
}

cudaError_t launch_topk_row_reg(const TopkParams& p, int max_n, bool pdl, cudaStream_t stream) {
  const int per = topk_row_reg_per(max_n);
  void (*kern)(const TopkParams) = nullptr;
  switch (per) {
    case 16: kern = topk_row_reg_kernel<16>; break;
    case 32: kern = topk_row_reg_kernel<32>; break;
    case 48: kern = topk_row_reg_kernel<48>; break;
    case 64: kern = topk_row_reg_kernel<64>; break;
    default: return cudaErrorInvalidValue;
  }
  return launch_kernel("topk_row_reg_kernel", kern, dim3(p.B * p.S), dim3(kRrThreads), 0, stream, pdl, p);
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
cudaError_t launch_topk_hist(const TopkParams& p, cudaStream_t stream) {
  return launch_kernel("topk_hist_kernel", topk_hist_kernel, dim3(p.nchunks, p.nrows), dim3(kHistThreads), 0, stream,
                       false, p);
}

cudaError_t launch_topk_chunk_select(const TopkParams& p, cudaStream_t stream) {
  const size_t smem = kCandSmem * sizeof(unsigned long long);
  cudaError_t e = set_max_smem(reinterpret_cast<const void*>(topk_chunk_select_kernel), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_kernel("topk_chunk_select_kernel", topk_chunk_select_kernel, dim3(p.nchunks, p.nrows), dim3(kSelThreads), smem,
                       stream, true, p);
}

// ---------------------------------------------------------------------------
// 2b. cluster select: one thread-block cluster of up to 16 CTAs per row. Each
// CTA holds a contiguous slice of the row's keys in registers. From the
// row histogram every CTA finds the threshold bin and compacts its keys in
// that bin (the candidates, usually a few hundred to a few thousand). Every
// CTA gathers all candidates through distributed shared memory and resolves
// the exact threshold composite (key << 32 | ~index) locally in 11-bit digit
// rounds; with more candidates than the gather holds (heavy ties) the digits
// are refined 8 bits at a time with the CTAs' digit histograms summed through
// distributed shared memory. Finally each CTA emits its own slice in ascending
// order (one block scan) at the offset given by the peers' selected counts. No
// global scratch beyond the histogram and no serial tail.
// ---------------------------------------------------------------------------
// Each of the NT threads owns PER consecutive keys of the slice, held in
// registers (PER = 8 or 16 with 1,024 threads, 32 with 512), so the emit needs
// a single block scan and no shared-memory bank conflicts arise; the
// threshold-bin candidates go to shared memory.
template <int PER, int NT>
__global__ void __launch_bounds__(NT, (PER <= 8 && NT <= 512) ? 2 : 1) topk_cluster_select_kernel(const TopkParams p) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  constexpr int kSlice = PER * NT;
  // candidate composites of this CTA (PER * NT), then the gathered list
  // (cl_gather_max(PER)), whose start first holds this CTA's slice histogram
  // and the range of bins it sums for the cluster (read by peers only before
  // the cluster barrier that precedes any gather)
  extern __shared__ unsigned long long scand[];
  static_assert(cl_gather_max(PER) * sizeof(unsigned long long) >= 2 * kHistBins * sizeof(uint32_t),
                "the histogram exchange must fit in the gather area");
  uint32_t* hloc = reinterpret_cast<uint32_t*>(scand + PER * NT);   // this CTA's slice histogram
  uint32_t* hred = hloc + kHistBins;             // the range of bins this CTA sums
  __shared__ __align__(16) uint32_t h[kHistBins];   // row histogram, then digit counts
  __shared__ uint32_t hd[256];                   // this CTA's digit histogram
  __shared__ uint32_t warp_tot[32];
  __shared__ int s_d;
  __shared__ uint32_t s_above, s_cnt;
  __shared__ uint32_t s_count;                   // keys this CTA selects
  __shared__ uint32_t s_ncand, s_nsure;          // published candidate / sure counts
  __shared__ uint32_t s_pc[kTopkClusterMax], s_ps[kTopkClusterMax];

  const int rl = blockIdx.y, r = p.row0 + rl;
  const int rank = static_cast<int>(cluster.block_rank());
  const int ncta = static_cast<int>(cluster.num_blocks());
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  DSA_TS_DECL;
  if (threadIdx.x == 0) DSA_TS(0);
  pdl_wait();      // scores and the histogram come from the previous kernel
  if (threadIdx.x == 0) DSA_TS(1);
  pdl_trigger();
  const RowInfo ri = row_info(p, r);
  const int t0 = rank * kSlice;
  const int m = max(0, min(ri.n, t0 + kSlice) - t0);
  const int tb = threadIdx.x * PER;              // this thread's first key in the slice
  const float* src = p.scores + static_cast<size_t>(r) * p.cap + t0 + tb;

  // ---- this thread's keys into registers (all loads in flight together)
  uint32_t key[PER];
  if (tb + PER <= m && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
#pragma unroll
    for (int v = 0; v < PER / 4; ++v) {
      const float4 f = __ldcg(reinterpret_cast<const float4*>(src) + v);
      key[4 * v] = float_key(f.x);
      key[4 * v + 1] = float_key(f.y);
      key[4 * v + 2] = float_key(f.z);
      key[4 * v + 3] = float_key(f.w);
    }
  } else {
#pragma unroll
    for (int j = 0; j < PER; ++j) key[j] = tb + j < m ? float_key(__ldcg(src + j)) : 0u;
  }
  const int nval = max(0, min(PER, m - tb));     // valid keys of this thread
  if (threadIdx.x == 0) { s_count = 0; s_ncand = 0; s_nsure = 0; s_d = 0; s_above = 0; s_cnt = 0; }
  if (p.hist_ready) {
    // ---- the row histogram came with the scores (indexer epilogue)
    const uint32_t* gh = p.hist + static_cast<size_t>(rl) * kHistBins;
#pragma unroll
    for (int u = 0; u < kHistBins / NT; ++u)
      h[u * NT + threadIdx.x] = __ldcg(gh + u * NT + threadIdx.x);
    __syncthreads();
  } else {
    // ---- the row histogram of the top 11 key bits, built by the cluster:
    // each CTA counts its slice, each CTA then sums one range of bins over all
    // peers, and every CTA reads the summed ranges back
    for (int i = threadIdx.x; i < kHistBins; i += NT) hloc[i] = 0u;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < PER; ++j)
      if (j < nval) atomicAdd(&hloc[key[j] >> (32 - kHistBits)], 1u);
    cluster.sync();                              // every CTA's slice histogram is complete
    {
      const int b0 = rank * kHistBins / ncta, b1 = (rank + 1) * kHistBins / ncta;
      for (int b = b0 + static_cast<int>(threadIdx.x); b < b1; b += NT) {
        uint32_t tot = 0;
        for (int q = 0; q < ncta; ++q) tot += cluster.map_shared_rank(hloc, q)[b];
        hred[b] = tot;
      }
    }
    cluster.sync();                              // every range is summed
#pragma unroll
    for (int u = 0; u < kHistBins / NT; ++u) {
      const int b = u * NT + threadIdx.x;
      const int owner = ((b + 1) * ncta - 1) / kHistBins;
      h[b] = cluster.map_shared_rank(hred, owner)[b];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) DSA_TS(2);
  // ---- threshold bin: a block-wide scan of the histogram
  find_threshold_digit<NT>(h, kHistBins, static_cast<uint32_t>(ri.keff), warp_tot, &s_d,
                                   &s_above, &s_cnt);
  if (threadIdx.x == 0) DSA_TS(3);
  const uint32_t bin = static_cast<uint32_t>(s_d);
  uint32_t need = static_cast<uint32_t>(ri.keff) - s_above;
  const bool all0 = (need == s_cnt);             // the whole threshold bin is selected
  bool all = all0;

  // ---- candidates (this thread's keys in the threshold bin) and sure keys
  // (above it); each warp reserves its candidates' slots with one atomic
  uint32_t cmask[(PER + 31) / 32] = {};
  uint32_t ncmine = 0, nsure = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j)
    if (j < nval) {
      const uint32_t kb = key[j] >> (32 - kHistBits);
      if (kb == bin) {
        cmask[j >> 5] |= 1u << (j & 31);
        ++ncmine;
      } else if (kb > bin) {
        ++nsure;
      }
    }
  {
    uint32_t incl = ncmine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    uint32_t wbase = 0;
    if (lane == 31 && incl) wbase = atomicAdd(&s_ncand, incl);
    uint32_t cpos = __shfl_sync(0xffffffffu, wbase, 31) + incl - ncmine;
#pragma unroll
    for (int j = 0; j < PER; ++j)
      if ((cmask[j >> 5] >> (j & 31)) & 1u)
        scand[cpos++] = (static_cast<unsigned long long>(key[j]) << 32) |
                        (0xFFFFFFFFull - static_cast<uint32_t>(t0 + tb + j));
    uint32_t ns = nsure;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ns += __shfl_xor_sync(0xffffffffu, ns, o);
    if (lane == 0 && ns) atomicAdd(&s_nsure, ns);
  }
  unsigned long long prefix = static_cast<unsigned long long>(bin) << 53;
  unsigned long long mask = ~0ull << 53;
  int32_t* out = p.idx + static_cast<size_t>(r) * p.k;
  // the threshold bin's total (s_cnt) is the same in every CTA: all take the
  // same path
  const bool gather = all || s_cnt <= static_cast<uint32_t>(cl_gather_max(PER));
  cluster.sync();                                // candidates and counts are published
  if (threadIdx.x == 0) DSA_TS(4);

  uint32_t pos = 0;                              // this CTA's first output slot
  int off_mine = 0;                              // gathered candidates of lower ranks
  if (gather) {
    // ---- every CTA gathers all candidates and counts, then resolves locally
    unsigned long long* sg = scand + PER * NT;   // gathered candidates
    if (threadIdx.x < ncta) {
      s_pc[threadIdx.x] = ld_cluster_u32(cluster_map(&s_ncand, threadIdx.x));
      s_ps[threadIdx.x] = ld_cluster_u32(cluster_map(&s_nsure, threadIdx.x));
    }
    __syncthreads();
    int off = 0;
    for (int q = 0; q < ncta; ++q) {
      if (q == rank) off_mine = off;
      off += static_cast<int>(s_pc[q]);
      if (q < rank) pos += s_ps[q] + (all0 ? s_pc[q] : 0u);
    }
    if (!all0) {
      // warp q copies peer q's list (at most 16 peers, 16 warps), four
      // loads in flight per lane
      if (warp < ncta) {
        int base = 0;
        for (int q = 0; q < warp; ++q) base += static_cast<int>(s_pc[q]);
        const int cnt = static_cast<int>(s_pc[warp]);
        const uint32_t peer = cluster_map(scand, warp);
        for (int i0 = 0; i0 < cnt; i0 += 128) {
          unsigned long long v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * 32 + lane;
            v[u] = i < cnt ? ld_cluster_u64(peer + 8u * i) : 0ull;
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * 32 + lane;
            if (i < cnt) sg[base + i] = v[u];
          }
        }
      }
      __syncthreads();
    }
    // this CTA is done reading its peers: arrive now, wait before exiting
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    if (threadIdx.x == 0) DSA_TS(5);
    if (!all0)
      resolve_composites<NT>(sg, off, &prefix, &mask, need, h, warp_tot, &s_d, &s_above,
                                     &s_cnt, 52);
  } else {
    // ---- many candidates (heavy ties): refine the threshold 8 bits at a time,
    // summing the CTAs' digit histograms through distributed shared memory
    const uint32_t ncand = s_ncand;
    int hi = 52;
    while (!all && hi >= 0) {
      const int w = hi + 1 < 8 ? hi + 1 : 8;
      const int sh = hi - w + 1;
      const uint32_t dm = (1u << w) - 1u;
      if (threadIdx.x < 256) hd[threadIdx.x] = 0u;
      __syncthreads();
      const int cround = ((static_cast<int>(ncand) + 31) / 32) * 32;   // whole warps take part
      for (int c = threadIdx.x; c < cround; c += NT) {
        uint32_t dg = 0xFFFFFFFFu;
        if (c < static_cast<int>(ncand)) {
          const unsigned long long cc = scand[c];
          if ((cc & mask) == prefix) dg = static_cast<uint32_t>(cc >> sh) & dm;
        }
        hist_add_warp(hd, dg);
      }
      cluster.sync();                            // every CTA's digit histogram is complete
      if (threadIdx.x < 256) {
        uint32_t tot = 0;
        for (int q = 0; q < ncta; ++q) tot += cluster.map_shared_rank(hd, q)[threadIdx.x];
        h[threadIdx.x] = tot;
      }
      if (threadIdx.x == 0) { s_d = 0; s_above = 0; s_cnt = 0; }
      __syncthreads();
      find_threshold_digit<NT>(h, 1 << w, need, warp_tot, &s_d, &s_above, &s_cnt);
      need -= s_above;
      prefix |= static_cast<unsigned long long>(s_d) << sh;
      mask |= static_cast<unsigned long long>(dm) << sh;
      all = (s_cnt == need);
      cluster.sync();                            // peers are done reading hd
      hi -= w;
    }
  }

  if (threadIdx.x == 0) DSA_TS(6);
  // ---- selection bits: bins above the threshold bin, or in it with the
  // determined composite bits at or above the threshold prefix; one block
  // scan gives both the in-CTA positions (low half) and, on the gather path,
  // the lower ranks' selected candidates (high half)
  uint32_t selm[(PER + 31) / 32] = {};
  uint32_t mine = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    if (j >= nval) break;
    const uint32_t kb = key[j] >> (32 - kHistBits);
    bool sel = kb > bin;
    if (kb == bin) {
      const unsigned long long cc = (static_cast<unsigned long long>(key[j]) << 32) |
                                    (0xFFFFFFFFull - static_cast<uint32_t>(t0 + tb + j));
      sel = (cc & mask) >= prefix;
    }
    if (sel) {
      selm[j >> 5] |= 1u << (j & 31);
      ++mine;
    }
  }
  uint32_t lower = 0;
  if (gather && !all0) {
    const unsigned long long* sg = scand + PER * NT;
    for (int c = threadIdx.x; c < off_mine; c += NT) lower += (sg[c] & mask) >= prefix ? 1u : 0u;
  }
  uint32_t total;
  const uint32_t packed = block_exclusive_scan<NT>(mine | (lower << 16), warp_tot, &total);
  if (threadIdx.x == 0) DSA_TS(7);
  pos += (packed & 0xFFFFu) + (total >> 16);
  if (!gather) {
    if (threadIdx.x == 0) s_count = total & 0xFFFFu;
    cluster.sync();                              // every CTA's count is published
    for (int q = 0; q < rank; ++q) pos += *cluster.map_shared_rank(&s_count, q);
  }
  const int seq = r / p.S;
#pragma unroll
  for (int wd = 0; wd < (PER + 31) / 32; ++wd) {
    uint32_t bits = selm[wd];
    while (bits) {
      const int j = __ffs(bits) - 1;
      bits &= bits - 1;
      if (pos < static_cast<uint32_t>(ri.keff)) {
        const int t = t0 + tb + wd * 32 + j;
        out[pos] = t;
        if (p.pf_k) {
          // the attention gathers this token's rows next: start them into L2
          bool bad = false;
          const long long row = cache_row(p.pg, seq, p.cap, t, &bad);
          prefetch_l2_bulk(p.pf_k + row * p.pf_row_bytes, p.pf_row_bytes);
          prefetch_l2_bulk(p.pf_v + row * p.pf_row_bytes, p.pf_row_bytes);
          if (p.pf_ks) {
            prefetch_l2_line(p.pf_ks + row * p.pf_heads);
            prefetch_l2_line(p.pf_vs + row * p.pf_heads);
          }
        }
      }
      ++pos;
    }
  }
  if (rank == 0)
    for (int i = ri.keff + threadIdx.x; i < p.k; i += NT) out[i] = -1;
  if (gather) asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  else cluster.sync();                           // peers may still read this CTA's s_count
  if (threadIdx.x == 0) DSA_TS(8);
  DSA_TS_FLUSH(p.status, 1);
}

// Threads of a cluster-select CTA holding `per` keys a thread: 1,024 with 8,
// 16 or 24 (64 registers, no spills), 512 with 32 (the keys need more
// registers than 1,024 threads leave).
static int cl_threads(int per) { return per <= 24 ? 1024 : kClThreads; }
static size_t cl_smem(int per) {
  return (static_cast<size_t>(per) * cl_threads(per) + cl_gather_max(per)) * sizeof(unsigned long long);
}
static const void* cl_kernel(int per) {
  return per == 8    ? reinterpret_cast<const void*>(topk_cluster_select_kernel<8, 1024>)
         : per == 16 ? reinterpret_cast<const void*>(topk_cluster_select_kernel<16, 1024>)
         : per == 24 ? reinterpret_cast<const void*>(topk_cluster_select_kernel<24, 1024>)
                     : reinterpret_cast<const void*>(topk_cluster_select_kernel<32, 512>);
}
// CTAs per row with `per` keys a thread (0: more than a cluster can hold).
static int cl_ctas(int max_n, int per) {
  const int slice = per * cl_threads(per);
  const int ctas = (max_n + slice - 1) / slice;
  return ctas > kTopkClusterMax ? 0 : ctas;
}
// Clusters of `ctas` CTAs of the `per` kernel that are resident at once on
// the current device, cached (0 if it cannot launch). A cluster must fit in
// one GPC, so on this GPU 15 clusters of 8 or 9 fit, 8 of 11 or 12 and 7 of
// 13 to 16.
static int cl_capacity(int per, int ctas) {
  static int cached[64][4][kTopkClusterMax + 1] = {};   // capacity + 1; 0: not queried
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int pi = per == 8 ? 0 : per == 16 ? 1 : per == 24 ? 2 : 3;
  int& slot = cached[dev][pi][ctas];
  if (slot) return slot - 1;
  const void* kern = cl_kernel(per);
  int n = 0;
  bool ok = set_max_smem(kern, static_cast<int>(cl_smem(per))) == cudaSuccess &&
            (ctas <= 8 || set_nonportable_cluster(kern) == cudaSuccess);
  if (ok) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas, 1);
    cfg.blockDim = dim3(cl_threads(per));
    cfg.dynamicSmemBytes = cl_smem(per);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ctas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  slot = n + 1;
  return n;
}
// Cluster shape for `nrows` rows of up to max_n keys: the fewest keys a
// thread (the slice load from L2 and the per-thread work shrink with them)
// whose clusters, one per row, are all resident at once; if none is, the
// fewest keys a thread that launch at all. ctas = 0: no shape fits.
static void cluster_shape(int max_n, int nrows, int* per, int* ctas) {
  static const int kPers[4] = {8, 16, 24, 32};
  *per = 0;
  *ctas = 0;
  for (int pass = 0; pass < 2 && *ctas == 0; ++pass)
    for (int i = 0; i < 4; ++i) {
      const int c = cl_ctas(max_n, kPers[i]);
      if (c == 0) continue;
      const int cap = cl_capacity(kPers[i], c);
      if (cap >= (pass == 0 ? nrows : 1)) {
        *per = kPers[i];
        *ctas = c;
        break;
      }
    }
}

bool topk_cluster_feasible(int max_n) {
  int per, ctas;
  cluster_shape(max_n, 1, &per, &ctas);
  return ctas > 0;
}

int topk_cluster_ctas(int max_n) {
  int per, ctas;
  cluster_shape(max_n, 1, &per, &ctas);
  return ctas;
}

cudaError_t launch_topk_cluster_select(const TopkParams& p, int max_n, bool pdl,
                                       cudaStream_t stream) {
  int per, ctas;
  cluster_shape(max_n, p.nrows, &per, &ctas);
  if (ctas == 0) return cudaErrorNotSupported;
  // worst case every key of the slice is a candidate; then the gathered list
  const size_t smem = cl_smem(per);
  const void* kern = cl_kernel(per);
  cudaError_t e = set_max_smem(kern, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (ctas > 8) {
    e = set_nonportable_cluster(kern);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas, p.nrows);
  cfg.blockDim = dim3(cl_threads(per));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ctas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  void* args[] = {const_cast<TopkParams*>(&p)};
  const cudaError_t le = cudaLaunchKernelExC(&cfg, kern, args);
  if (le == cudaSuccess) note_launch("topk_cluster_select_kernel");
  return le;
}

cudaError_t launch_topk_row(const TopkParams& p, int max_n, size_t smem_limit, bool pdl,
                            cudaStream_t stream) {
  const size_t smem = (static_cast<size_t>((max_n + 3) & ~3) + kHistBins) * sizeof(uint32_t);
  if (smem + 1024 > smem_limit) return cudaErrorInvalidValue;
  cudaError_t e = set_max_smem(reinterpret_cast<const void*>(topk_row_kernel), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_kernel("topk_row_kernel", topk_row_kernel, dim3(p.B * p.S), dim3(kRowThreads), smem, stream, pdl, p);
}

}  // namespace dsa
