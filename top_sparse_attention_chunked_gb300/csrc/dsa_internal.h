// Internal parameter blocks and launcher entry points shared by the library's
// translation units (host API <-> kernels). Not part of the public C ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/dsa.h"

namespace dsa {

// Kernels enqueued by the current public call on this host thread, in order
// (reported by dsa_last_launches). Every launch site records its kernel's name
// once the launch has been accepted.
void note_launch(const char* name);
void reset_launches();

// cudaFuncSetAttribute(kern, MaxDynamicSharedMemorySize, bytes) and
// (NonPortableClusterSizeAllowed, 1), each issued once per kernel, CUDA
// context and value: a driver call per launch costs host time on every call.
cudaError_t set_max_smem(const void* kern, int bytes);
cudaError_t set_nonportable_cluster(const void* kern);

// Launch `kern` (recorded as `name`) on `stream`; with `pdl` the launch may overlap the tail of the
// previous kernel in the stream (the kernel calls pdl_wait() before reading
// what that kernel wrote).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(const char* name, void (*kern)(KArgs...), dim3 grid, dim3 block,
                          size_t smem, cudaStream_t stream, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  if (e == cudaSuccess) note_launch(name);
  return e;
}

constexpr int kChunk = DSA_CHUNK;          // 2,048-key chunks (indexer + top-k)
constexpr int kHistBits = 11;              // first radix digit: top 11 key bits
constexpr int kHistBins = 1 << kHistBits;  // 2,048 bins per query row
constexpr int kKeyTile = 128;              // keys per tcgen05 indexer tile (M)
constexpr uint32_t kDevTimeout = 1u;       // status bit: a bounded wait ran out
constexpr long long kDefaultWaitBudget = 2000000000ll;   // SM cycles before a wait gives up

struct SeqLens {
  int32_t T[DSA_MAX_BATCH];
};

// Where a sequence's cached token lives. Dense: row b * cap + t of a
// [B * cap] array. Paged: the caches are a pool of num_blocks blocks of
// 2^shift tokens and block_table[b * per_seq + t >> shift] names the block
// holding token t; an entry outside [0, num_blocks) is read as block 0 (no
// memory outside the pool is touched) and reported as `bad`.
struct Paging {
  const int32_t* table;   // [B, per_seq] or nullptr (dense)
  int per_seq;            // blocks per sequence (columns of the table)
  int shift;              // log2(block size)
  int num_blocks;         // blocks in the pool
};

constexpr uint32_t kDevBadPage = 2u;   // status bit: a block-table entry outside the pool

__device__ __forceinline__ long long cache_row(const Paging& pg, int b, int cap, int t, bool* bad) {
  if (pg.table == nullptr) return static_cast<long long>(b) * cap + t;
  int blk = __ldg(pg.table + b * pg.per_seq + (t >> pg.shift));
  if (blk < 0 || blk >= pg.num_blocks) {
    *bad = true;
    blk = 0;
  }
  return (static_cast<long long>(blk) << pg.shift) + (t & ((1 << pg.shift) - 1));
}

// ---------------------------------------------------------------- indexer
struct IndexerParams {
  const float* w;        // [B, S, 16]
  float* scores;         // [B, S, cap]
  uint32_t* hist;        // [B*S, 2048] radix histograms (decode) or nullptr
  uint32_t* status;      // device status word
  int B, S, cap;
  int QB;                // query tokens per block (N = 16 * QB)
  int nqb;               // query blocks per sequence, ceil(S / QB)
  long long total_units; // (sequence, query block, key tile) triples
  long long wait_budget; // SM cycles before one of its pipeline waits gives up
  Paging pg;               // cache addressing (dense or paged)
  SeqLens lens;
};

constexpr uint32_t kDevBounds = 4u;    // status bit: a debug bounds check failed

// Debug builds (-DDSA_DEBUG_BOUNDS) check the rows that index-driven gathers
// compute against the extent of the array they read: a row outside it sets
// kDevBounds in the status word and the access is skipped (never a trap).
// Release builds compile the check to `true`.
#ifdef DSA_DEBUG_BOUNDS
__device__ __forceinline__ bool bounds_ok(bool cond, uint32_t* status) {
  if (!cond && status) atomicOr(status, kDevBounds);
  return cond;
}
#else
__device__ __forceinline__ constexpr bool bounds_ok(bool, uint32_t*) { return true; }
#endif

// Kernel kinds for the timing hook (mirror DSA_KERNEL_*).
void timing_before(int kind, cudaStream_t stream);
void timing_after(int kind, cudaStream_t stream);

// grid.y > 1 gives each sequence its own CTAs (required with histograms).
cudaError_t launch_indexer(const IndexerParams& p, const CUtensorMap& tm_kI,
                           const CUtensorMap& tm_qI, dim3 grid, size_t smem_bytes,
                           int stages, cudaStream_t stream);
size_t indexer_smem_bytes(int QB, bool with_hist, int* stages_out, size_t smem_limit);
// Clears `bytes` (a multiple of 16) of scratch; the next kernel may overlap it.
cudaError_t launch_zero_scratch(void* base, size_t bytes, cudaStream_t stream);

// ---------------------------------------------------------------- top-k
struct TopkParams {
  const float* scores;          // [B*S, cap]
  int32_t* idx;                 // [B*S, k]
  uint32_t* hist;               // [B*S, 2048]     zeroed before the first kernel
  uint32_t* ticket;             // [B*S]           zeroed
  uint32_t* cand_count;         // [B*S]           zeroed
  unsigned long long* cands;    // [B*S, cand_stride] candidate composites
  uint32_t* bitmap;             // [B*S, bitmap_stride] selection bits
  long long cand_stride;
  int bitmap_stride;            // words per row
  int B, S, cap, k;
  int nchunks;                  // chunks of the longest row
  int row0, nrows;              // rows handled by this launch (workspace rows are local)
  int hist_ready;               // cluster select: the row histograms are in `hist`
  uint32_t* status;             // device status word (nullptr: none)
  // Decode: as the cluster select emits a key it prefetches that token's K
  // and V rows (all KV heads) and INT8 scales into L2 for the attention that
  // follows. pf_k == nullptr: no prefetch.
  const uint8_t* pf_k;
  const uint8_t* pf_v;
  const float* pf_ks;           // INT8 scales [.., Hkv] or nullptr
  const float* pf_vs;
  int pf_row_bytes;             // bytes of one token's K (or V) over all KV heads
  int pf_heads;                 // KV heads
  Paging pg;                    // cache addressing of the prefetched rows
  SeqLens lens;
};

cudaError_t launch_topk_hist(const TopkParams& p, cudaStream_t stream);
cudaError_t launch_topk_chunk_select(const TopkParams& p, cudaStream_t stream);
// `pdl`: launched right after another kernel of the same call
cudaError_t launch_topk_row(const TopkParams& p, int max_n, size_t smem_limit, bool pdl,
                            cudaStream_t stream);
// Cluster select: up to kTopkClusterMax CTAs per row (16, checked at launch),
// each owning up to 16,384 keys (32 per thread, in registers).
constexpr int kTopkClusterMax = 16;
int topk_cluster_ctas(int max_n);   // 0 if the row is too long for it
cudaError_t launch_topk_cluster_select(const TopkParams& p, int max_n, bool pdl,
                                       cudaStream_t stream);
// Streaming whole-row select (one CTA per row, several rows per SM): rows of
// up to topk_row_stream_max_len() keys; needs no zeroed scratch.
int topk_row_stream_max_len();
cudaError_t launch_topk_row_stream(const TopkParams& p, int max_n, bool pdl, cudaStream_t stream);
// Whole-row select with the keys in registers: keys per thread for rows of
// up to max_n keys (0 if too long).
int topk_row_reg_per(int max_n);
cudaError_t launch_topk_row_reg(const TopkParams& p, int max_n, bool pdl, cudaStream_t stream);
// Longest row the shared-memory whole-row select handles.
int topk_row_max_len(size_t smem_limit);

// ---------------------------------------------------------------- attention
struct AttnParams {
  const void* q;           // [B, S, Hq, 128]
  const void* k;           // [B, cap, Hkv, 128]
  const void* v;
  const float* k_scale;    // [B, cap, Hkv] (INT8 only)
  const float* v_scale;
  const int32_t* idx;      // [B*S, topk]
  // The new tokens' own K / V [B, S, Hkv, 128] in the query dtype, or nullptr.
  // A selected key at or after a sequence's first new token reads these rows
  // (fp32 arithmetic at their own values) instead of the cache.
  const void* k_aux;
  const void* v_aux;
  void* out;               // [B, S, Hq, 128]
  float* partial;          // split-K partial states
  uint32_t* ticket;        // [B*S*Hkv*HG] zeroed when nsplit > 1
  int B, S, Hq, Hkv, G, HG, cap, topk;
  // K / V row (128 values) of (sequence b, token t, KV head g) on a dense
  // cache: b * kv_sb + t * kv_st + g * kv_sh (the paged pool keeps its
  // token-major rows)
  long long kv_sb, kv_st, kv_sh;
  long long kv_rows;       // K / V rows (128 values) the caches span
  long long scale_rows;    // INT8 scale entries the scale arrays hold
  int split_keys, nsplit;
  int cluster;             // nsplit in {2,4,8,16}: splits merged inside a thread-block cluster
  int q_dtype, out_dtype;
  float scale_log2;        // softmax_scale * log2(e)
  uint32_t* status;        // device status word (a bounded wait that ran out)
  Paging pg;               // cache addressing (dense or paged)
  SeqLens lens;
};

constexpr int kAttnRows = 16;                                   // heads per MMA tile
constexpr int kAttnMaxSplits = 128;                             // split-K partial states per row
constexpr int kAttnMaxSplitKeys = 2048;                         // selected keys per split CTA
constexpr int kPartialFloats = 2 * kAttnRows + kAttnRows * DSA_HEAD_DIM;  // m, l, o

// tm_k / tm_v: the caches as [B * cap * Hkv, 128] rows, 128-byte swizzle,
// box of one row (16-bit: 64 columns; INT8: 128 columns)
cudaError_t launch_attention(const AttnParams& p, int q_dtype, int kv_dtype, int out_dtype,
                             const CUtensorMap& tm_k, const CUtensorMap& tm_v, cudaStream_t stream);

// Largest thread-block cluster the split-K attention can use on this device
// (16 if a 16-CTA cluster can be placed, else 8), and whether a split count
// is merged inside a cluster.
int attn_max_cluster();
// Clusters of `size` attention CTAs (2, 4, 8 or 16) resident at once on this
// device (0 if none fits or the size is not one of those).
int attn_cluster_capacity(int size);
inline bool attn_uses_cluster(int nsplit) {
  return (nsplit == 2 || nsplit == 4 || nsplit == 8 || nsplit == 16) && nsplit <= attn_max_cluster();
}
// Whether the cluster top-k can be placed for rows of max_n keys.
bool topk_cluster_feasible(int max_n);

// tcgen05 prefill attention (BF16 / FP16 cache, top_k <= 2048)
bool prefill_tc_supported(const AttnParams& p, int kv_dtype, size_t smem_optin);
cudaError_t launch_prefill_tc(const AttnParams& p, int kv_dtype, int sms, const CUtensorMap& tm_k,
                              const CUtensorMap& tm_v, uint32_t* status, cudaStream_t stream);

// ---------------------------------------------------------------- cache append
struct AppendParams {
  const void* kI_new;      // [B, S, 64] bf16
  const void* k_new;       // [B, S, Hkv, 128] q_dtype
  const void* v_new;
  void* kI;                // [B, cap, 64] bf16
  void* k;                 // [B, cap, Hkv, 128] kv_dtype
  void* v;
  float* k_scale;          // [B, cap, Hkv] (INT8 only)
  float* v_scale;
  int B, S, Hkv, cap;
  int q_dtype, kv_dtype;
  Paging pg;               // cache addressing (dense or paged)
  SeqLens lens;
};

cudaError_t launch_cache_append(const AppendParams& p, int sms, cudaStream_t stream);

}  // namespace dsa
