/*
 * libdsa -- dynamic sparse attention on one NVIDIA GB300 (sm_103a).
 *
 * For each query token the step does three things (pages: ONNX Runtime PR
 * #33802 "[CUDA] Optimize Qwen3.8-Flash-Next DSA, Indexer, HC, and QMoE kernels
 * for SM12x and 256K context", Summary items 1-2, and PR #33997 "[CUDA] Support
 * FP16 KV cache and FP16 query/key in DynamicSparseAttention<BFloat16> ...",
 * Description item 2):
 *
 *   1. indexer   score[t] = sum_h w[h] * max(0, qI[h] . kI[t])   (16 index
 *                heads of dim 64 against one index key per cached token,
 *                fp32 accumulation), streamed in 2,048-key chunks;
 *   2. top-k     the top_k highest-scoring visible keys (ties -> lower index),
 *                a radix select over per-chunk histograms with one final
 *                merge-and-emit;
 *   3. attention softmax GQA attention of every query head over only the
 *                selected K/V rows (BF16, FP16 or INT8 with a per-token
 *                per-head fp32 scale), split over the selected keys with an
 *                online-softmax combine (follow-up PR #33847: the rescale never
 *                flushes the earlier tiles).
 *
 * Around the step: the cache append of the new tokens (with INT8
 * quantise-on-write), fp32 RMSNorm + rotary embedding, both in one launch
 * (dsa_rope_append), and _paged forms of the calls for caches kept in a pool
 * of token blocks with a block table.
 *
 * Conventions (all calls):
 *  - Positions: a sequence's cache holds T_b = total_len[b] rows and its
 *    q_len new query tokens are the LAST q_len rows, so query s sits at
 *    position T_b - q_len + s and sees keys 0 .. T_b - q_len + s (causal,
 *    itself included). Prefill and decode follow the same rule.
 *  - Every tensor argument is a DEVICE pointer owned by the caller, dense
 *    row-major in the layout stated beside it. The library allocates no
 *    device memory and never synchronises the stream: every call enqueues
 *    its kernels on `stream` (a cudaStream_t; NULL = legacy default stream)
 *    and returns. It can be captured in a CUDA graph.
 *  - Arguments are validated on the host before anything is enqueued; on a
 *    bad argument nothing is launched and the call returns the status, with
 *    a message in dsa_last_error_string().
 *  - The workspace is caller-owned device memory of at least
 *    dsa_workspace_size() bytes, 256-byte aligned. Its contents are never
 *    assumed: each call initialises what it uses. Calls that share a
 *    workspace must be ordered on one stream.
 *  - Problems a kernel detects (a bounded wait that ran out) are OR-ed into a
 *    status word at the start of the workspace; read it with
 *    dsa_read_device_status() after the call.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dsa_status {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,   /* shape, length or pointer is wrong          */
  DSA_ERR_UNSUPPORTED = 2,   /* valid but not built (dims, dtype combo)     */
  DSA_ERR_WORKSPACE = 3,     /* workspace missing, misaligned or too small  */
  DSA_ERR_MISALIGNED = 4,    /* a tensor pointer breaks its alignment rule  */
  DSA_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed           */
  DSA_ERR_TIMEOUT = 6,       /* a kernel's bounded wait ran out (device)    */
  DSA_ERR_NO_DEVICE = 7      /* no usable sm_100-class GPU is current       */
} dsa_status;

typedef enum dsa_dtype {
  DSA_BF16 = 0,
  DSA_FP16 = 1,
  DSA_INT8 = 2,              /* KV cache only: codes + fp32 scale per token/head */
  DSA_FP32 = 3               /* output only */
} dsa_dtype;

/* Which call a workspace is sized for. */
typedef enum dsa_op {
  DSA_OP_INDEX_SCORES = 0,
  DSA_OP_TOPK = 1,
  DSA_OP_DECODE = 2,
  DSA_OP_PREFILL = 3
} dsa_op;

/* Built-in limits. */
#define DSA_MAX_BATCH 64          /* sequences per call                          */
#define DSA_HEAD_DIM 128          /* attention head dim                          */
#define DSA_IDX_HEADS 16          /* index heads                                 */
#define DSA_IDX_DIM 64            /* index head dim                              */
#define DSA_CHUNK 2048            /* indexer / top-k chunk (keys)                */
#define DSA_MAX_DECODE_Q_LEN 16   /* query tokens per sequence in decode         */
#define DSA_MAX_CONTEXT (1 << 20) /* visible keys per query row                  */

/*
 * The problem, passed by pointer to every call (read on the host only, so it
 * may live on the stack).
 *
 *   batch            B, 1 .. DSA_MAX_BATCH
 *   q_len            S, new query tokens per sequence (>= 1; <= 16 in decode)
 *   num_q_heads      Hq
 *   num_kv_heads     Hkv, Hq % Hkv == 0; head h reads KV head h / (Hq/Hkv)
 *   head_dim         D, must be 128
 *   idx_heads        must be 16
 *   idx_dim          must be 64
 *   cache_capacity   cap: rows allocated per sequence in kI/K/V/scales; also
 *                    the row stride of the score tensor
 *   top_k            1 .. cap; a query with n < top_k visible keys selects
 *                    all n and pads its index row with -1
 *   total_len[b]     T_b, q_len .. cap (entries >= batch are ignored)
 *   softmax_scale    logits = softmax_scale * q.K; 0 selects 1/sqrt(head_dim)
 *   q_dtype          DSA_BF16 or DSA_FP16
 *   kv_dtype         DSA_BF16, DSA_FP16 or DSA_INT8 (FP16 query with a BF16
 *                    cache is not built)
 *   out_dtype        DSA_BF16, DSA_FP16 or DSA_FP32
 *   attn_split_keys  0 = automatic; otherwise selected keys per split-K
 *                    attention block, a multiple of 16 (a tuning and testing
 *                    knob: results agree for every value)
 */
typedef struct dsa_problem {
  int32_t batch;
  int32_t q_len;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t idx_heads;
  int32_t idx_dim;
  int32_t cache_capacity;
  int32_t top_k;
  int32_t total_len[DSA_MAX_BATCH];
  float softmax_scale;
  int32_t q_dtype;
  int32_t kv_dtype;
  int32_t out_dtype;
  int32_t attn_split_keys;
  /* K / V cache layout, in elements: the strides of the batch, token and KV
   * head dimensions (in this order). All zero: the default token-major
   * layout [B, cap, Hkv, 128] (strides cap*Hkv*128, Hkv*128, 128). Otherwise
   * each (batch, token, head) vector of 128 values must be contiguous, so
   * every stride is a multiple of 128 (the token stride at least 128, the
   * head stride at least 128 when Hkv > 1); a BNSH cache [B, Hkv, cap, 128]
   * is (Hkv*cap*128, 128, cap*128). The same layout holds for K and V (INT8
   * codes included); INT8 scales stay [B, cap, Hkv]. Used by the decode and
   * prefill calls on dense caches; the paged calls, dsa_cache_append and
   * dsa_rope_append take only the default (all zero), else
   * DSA_ERR_UNSUPPORTED. */
  int64_t kv_strides[3];
} dsa_problem;

/*
 * Bytes of workspace the call `op` needs for problem `p` (0 and a message in
 * dsa_last_error_string() if `p` is invalid). Pure host computation.
 */
size_t dsa_workspace_size(const dsa_problem* p, int op);

/*
 * dsa_index_scores -- the indexer alone (step 1). PR #33802 Summary item 2
 * (PackedSparseAttentionIndexer: per-query scoring of every cached index key).
 *
 *   qI      [B, S, 16, 64] bf16, 16-byte aligned
 *   w       [B, S, 16] fp32 head weights
 *   kI      [B, cap, 64] bf16 index keys, 16-byte aligned
 *   scores  [B, S, cap] fp32 out: scores[b,s,t] for t <= T_b - S + s; entries
 *           past a query's visible length are not written. 16-byte aligned.
 * Runs on tcgen05 tensor cores (BF16 x BF16 -> FP32 in tensor memory).
 */
int dsa_index_scores(const dsa_problem* p, const void* qI, const float* w,
                     const void* kI, float* scores, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * dsa_topk -- the selection alone (step 2) on a given fp32 score tensor.
 * PR #33802 Summary item 2 (radix partial top-k per 2,048-key chunk with
 * warp-aggregated histograms, one final merge-and-emit).
 *
 *   scores  [B, S, cap] fp32; only the visible prefix of each row is read.
 *           Values are compared exactly; -0.0 equals +0.0; NaN is not allowed.
 *   idx     [B, S, top_k] int32 out: the selected key indices in ascending
 *           order, then -1 up to top_k.
 * The result is exact (bit-identical to sorting by (-score, index)).
 */
int dsa_topk(const dsa_problem* p, const float* scores, int32_t* idx,
             void* workspace, size_t workspace_bytes, void* stream);

/*
 * dsa_sparse_attn_decode -- the whole step for a few query tokens per
 * sequence (S <= 16): indexer (with the chunk histograms fused in), top-k,
 * then grouped split-K sparse attention. PR #33997 Description item 2
 * (grouped decode over the selected rows), PR #33802 Summary item 1 (INT8
 * cache, split-K decode), PR #33847 (rescale without flushing).
 *
 *   q        [B, S, Hq, 128] q_dtype, 16-byte aligned
 *   qI, w, kI as for dsa_index_scores
 *   k, v     [B, cap, Hkv, 128] kv_dtype (values, or INT8 codes), 16-byte aligned
 *   k_scale, v_scale  [B, cap, Hkv] fp32, required iff kv_dtype == DSA_INT8
 *            (else must be NULL): K^ = code * k_scale
 *   idx_out  [B, S, top_k] int32 (optional, NULL allowed): receives the
 *            selected indices as dsa_topk emits them
 *   out      [B, S, Hq, 128] out_dtype
 */
int dsa_sparse_attn_decode(const dsa_problem* p, const void* q, const void* qI,
                           const float* w, const void* kI, const void* k,
                           const void* v, const float* k_scale,
                           const float* v_scale, int32_t* idx_out, void* out,
                           void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * dsa_sparse_attn_decode_aux -- dsa_sparse_attn_decode with floating
 * auxiliary K/V: the step's new tokens' own key and value rows, given beside
 * the caches in the query's floating type. PR #33997 "[CUDA] Support FP16 KV
 * cache and FP16 query/key in DynamicSparseAttention<BFloat16> ...": its
 * review summary notes that grouped attention can overflow BF16 auxiliary
 * values when converting them to FP16, and its second commit keeps floating
 * auxiliary K/V with FP16 main caches. Reading taken here: a selected key t
 * of sequence b with t >= total_len[b] - q_len (one of the new tokens, whose
 * rows are the last q_len cache rows) takes K and V from
 * k_aux[b][t - (total_len[b] - q_len)] and v_aux[...] at their own values
 * (attended in fp32, never converted to the cache's type; a BF16 value above
 * FP16's 65504 stays finite); every other selected key reads the cache. The
 * indexer and the selection are those of dsa_sparse_attn_decode (the new
 * tokens' index keys are in kI as always).
 *
 *   k_aux, v_aux  [B, S, Hkv, 128] q_dtype, 16-byte aligned, required
 *   all other arguments, the workspace and the errors as for
 *   dsa_sparse_attn_decode (same workspace size).
 */
int dsa_sparse_attn_decode_aux(const dsa_problem* p, const void* q, const void* qI,
                               const float* w, const void* kI, const void* k,
                               const void* v, const float* k_scale,
                               const float* v_scale, const void* k_aux,
                               const void* v_aux, int32_t* idx_out, void* out,
                               void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * dsa_sparse_attn_prefill -- the whole step for a chunk of many new tokens
 * (any S >= 1): the indexer as a dense causal contraction on tcgen05 tensor
 * cores, a per-row top-k held in shared memory, then sparse attention.
 * Same arguments and layouts as dsa_sparse_attn_decode. PR #33997
 * Description item 2 (sparse-attention prefill on tensor cores), PR #33802
 * Summary item 2 (ragged prefill scoring).
 */
int dsa_sparse_attn_prefill(const dsa_problem* p, const void* q, const void* qI,
                            const float* w, const void* kI, const void* k,
                            const void* v, const float* k_scale,
                            const float* v_scale, int32_t* idx_out, void* out,
                            void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * dsa_cache_append -- write the q_len new tokens of every sequence into the
 * caches, the step that comes before the indexer. PR #33997 "[CUDA] Support
 * FP16 KV cache and FP16 query/key in DynamicSparseAttention<BFloat16> ...":
 * its Files changed table puts the cache writes in the implementation file
 * beside the attention kernels, and its description names the quantized
 * (INT8) cache, whose per-token per-head scale this call produces.
 *
 * Token s of sequence b goes to cache row T_b - q_len + s, with
 * T_b = total_len[b] counting the new tokens (the positions rule above), so
 * the same problem then drives dsa_sparse_attn_decode / _prefill. `p` is
 * validated as for dsa_sparse_attn_prefill (top_k and the output fields too).
 *
 *   kI_new        [B, q_len, 64] bf16 new index keys, 16-byte aligned
 *   k_new, v_new  [B, q_len, Hkv, 128] q_dtype new keys / values, 16-byte aligned
 *   kI            [B, cap, 64] bf16 index-key cache (rows T_b-q_len..T_b-1 written)
 *   k, v          [B, cap, Hkv, 128] kv_dtype caches (the same rows written)
 *   k_scale, v_scale  [B, cap, Hkv] fp32, required iff kv_dtype == DSA_INT8
 *                 (else NULL). For an INT8 cache each new (token, KV head) row
 *                 gets scale = absmax/127 and code = round-half-even(x /
 *                 scale) clamped to +-127, both divisions IEEE fp32; an
 *                 all-zero row gets scale 0 and codes 0. A 16-bit cache of the
 *                 other 16-bit type takes x rounded to nearest even.
 * No other row and no other byte is written. The new-token tensors must not
 * overlap any cache (checked, DSA_ERR_INVALID_ARG). Values must be finite. One
 * kernel launch; no workspace.
 */
int dsa_cache_append(const dsa_problem* p, const void* kI_new, const void* k_new,
                     const void* v_new, void* kI, void* k, void* v, float* k_scale,
                     float* v_scale, void* stream);

/*
 * dsa_rmsnorm_rotary -- RMSNorm + rotary position embedding in fp32, the step
 * that produces q, k, qI and kI before the cache append and the attention.
 * PR #33997 Description item 1 (RMSNormRotary computed in exact FP32 with no
 * intermediate BF16 rounding, from a BF16 or FP32 cos/sin cache, to a BF16 or
 * FP16 output). For every head vector x (head_dim D) of token n:
 *     y = x * gamma / sqrt(mean(x^2) + eps)
 *     out_i       = y_i * cos[p, i] - y_{i+r/2} * sin[p, i]    (i < r/2)
 *     out_{i+r/2} = y_{i+r/2} * cos[p, i] + y_i * sin[p, i]
 *     out_i       = y_i                                        (i >= r)
 * with p = positions[n] (clamped to 0 .. max_pos - 1) and r = rotary_dim,
 * every step in fp32 and one round-to-nearest-even conversion at the end.
 * Vectors whose absmax lies outside [2^-60, 2^60] are rescaled by an exact
 * power of two first, so the fp32 sum of squares cannot overflow or vanish.
 * With eps = 0 an all-zero vector gives NaN, as the formula does.
 *
 *   tokens      N >= 0 (0: nothing is launched)
 *   heads       H >= 1
 *   head_dim    D: 64 or 128
 *   rotary_dim  r: even, 0 .. D (0: RMSNorm only)
 *   max_pos     rows of the cos / sin caches (>= 1 when r > 0)
 *   eps         finite, >= 0
 *   x_dtype, y_dtype   DSA_BF16 or DSA_FP16
 *   cos_dtype   DSA_FP32 or DSA_BF16
 *
 *   x           [N, H, D] x_dtype, 16-byte aligned
 *   gamma       [D] fp32 channel weights
 *   cos_cache, sin_cache  [max_pos, r/2] cos_dtype (NULL allowed when r = 0)
 *   positions   [N] int32 (NULL allowed when r = 0)
 *   y           [N, H, D] y_dtype, 16-byte aligned; may be x itself (in
 *               place), must not overlap it otherwise
 * All DEVICE pointers owned by the caller; no workspace; one kernel.
 */
typedef struct dsa_rope_problem {
  int64_t tokens;
  int32_t heads;
  int32_t head_dim;
  int32_t rotary_dim;
  int32_t max_pos;
  float eps;
  int32_t x_dtype;
  int32_t cos_dtype;
  int32_t y_dtype;
} dsa_rope_problem;

int dsa_rmsnorm_rotary(const dsa_rope_problem* rp, const void* x, const float* gamma,
                       const void* cos_cache, const void* sin_cache, const int32_t* positions,
                       void* y, void* stream);

/*
 * dsa_rope_append -- the work before the indexer in one launch: RMSNorm +
 * rotary embedding of the step's new q and qI (in place), of k_new and
 * kI_new, and the cache append of the rotated kI and k and of v_new. Equal,
 * bit for bit, to dsa_rmsnorm_rotary on q (q dtype), qI (BF16), k_new (into
 * the q dtype) and kI_new (into BF16), all at positions total_len[b] - q_len
 * + s, followed by dsa_cache_append. PR #33997 Description item 1 and its
 * Files changed table (the cache writes beside the attention kernels).
 * Dense caches only.
 *
 *   q        [B, S, Hq, 128] q_dtype, rotated in place
 *   qI       [B, S, 16, 64] bf16, rotated in place
 *   k_new, v_new  [B, S, Hkv, 128] q_dtype (not modified)
 *   kI_new   [B, S, 64] bf16 (not modified)
 *   kI, k, v, k_scale, v_scale  the caches, as for dsa_cache_append
 * All 16-byte aligned DEVICE pointers; the new-token tensors must not overlap
 * a cache. The rope parameters:
 *   eps          finite, >= 0 (all four tensors)
 *   max_pos      rows of the cos / sin caches (>= 1 if any rotary width > 0)
 *   cos_dtype    DSA_FP32 or DSA_BF16 (both caches)
 *   rotary_dim, cos, sin              q and k: even width <= 128, caches
 *                                     [max_pos, rotary_dim / 2]
 *   rotary_dim_index, cos_index, sin_index   qI and kI: even width <= 64
 *   gamma_q, gamma_k [128], gamma_qI, gamma_kI [64]   fp32 channel weights
 */
typedef struct dsa_rope_params {
  float eps;
  int32_t max_pos;
  int32_t cos_dtype;
  int32_t rotary_dim;
  int32_t rotary_dim_index;
  const void* cos;
  const void* sin;
  const void* cos_index;
  const void* sin_index;
  const float* gamma_q;
  const float* gamma_k;
  const float* gamma_qI;
  const float* gamma_kI;
} dsa_rope_params;

int dsa_rope_append(const dsa_problem* p, const dsa_rope_params* rope, void* q, void* qI,
                    const void* k_new, const void* kI_new, const void* v_new, void* kI, void* k,
                    void* v, float* k_scale, float* v_scale, void* stream);

/*
 * dsa_topk_noalloc -- dsa_topk for callers that cannot give the library any
 * device memory. Some callers cannot allocate: an operator plugin whose host
 * framework hands it only its input and output tensors, a serving engine that
 * reserves its whole memory budget at start-up and forbids allocations while
 * requests run, or a latency-critical path that cannot take cudaMalloc's
 * implicit device synchronisation. This call takes no workspace: its scratch
 * (radix histograms, tickets, candidates, selection bitmaps) is a static
 * device array of about 8.2 MiB inside libdsa that every GPU loading the
 * library holds until the process exits. The pages have no counterpart of
 * this call.
 *
 *   scores, idx   as for dsa_topk (device pointers owned by the caller)
 *
 * Limits: at most DSA_TOPK_NOALLOC_MAX_ROWS query rows (batch * q_len) of at
 * most DSA_TOPK_NOALLOC_MAX_LEN visible keys; larger problems are rejected
 * with DSA_ERR_UNSUPPORTED before anything is enqueued. The call allocates
 * nothing (no cudaMalloc, no library allocator). Its first call on a device
 * looks up the scratch array's device address for that device
 * (cudaGetSymbolAddress), so make that first call before any stream capture.
 * Every call shares the one array and its contents persist between calls;
 * each call clears the parts that must start at zero. Calls that overlap on
 * the GPU (concurrent streams or host threads) race on the scratch and must
 * be serialised by the caller. The result equals dsa_topk's bit for bit.
 */
#define DSA_TOPK_NOALLOC_MAX_ROWS 8
#define DSA_TOPK_NOALLOC_MAX_LEN 131072
int dsa_topk_noalloc(const dsa_problem* p, const float* scores, int32_t* idx,
                     void* stream);

/*
 * Paged caches. On the page of ONNX Runtime PR #33802, the companion
 * onnxruntime-genai change (#2840), Summary item 1: the KV and indexer caches
 * of a 256K request live in a pool of fixed-size token blocks (block_size 256,
 * num_blocks 1,037, of which 1,024 hold the target's 262,144 tokens); paged
 * attention walks a per-sequence block table (PR #34117, "quantized paged
 * attention"; PR #28200's paged-KV gather on the same page set).
 *
 * With a paged cache, kI, K, V and the INT8 scales are pools of
 * num_blocks * block_size token rows: kI [num_blocks * block_size, 64] bf16,
 * K / V [num_blocks * block_size, Hkv, 128] kv_dtype, k_scale / v_scale
 * [num_blocks * block_size, Hkv] fp32. Token t of sequence b (its logical
 * position, the same one the dense layout uses) lives in pool row
 *     block_table[b * blocks_per_seq + t / block_size] * block_size
 *         + t % block_size.
 * The problem's cache_capacity must equal blocks_per_seq * block_size; it
 * remains the row stride of the score tensor. Every other argument, the
 * workspace size (dsa_workspace_size with the same op) and every result are
 * those of the dense call on the gathered (logical) caches, bit for bit.
 *
 *   block_size      tokens per block: a power of two from 128 to 2^20 (a
 *                   128-key indexer tile never straddles two blocks)
 *   num_blocks      blocks in the pool (num_blocks * block_size * Hkv < 2^31)
 *   blocks_per_seq  columns of the block table
 *   block_table     DEVICE [B, blocks_per_seq] int32, 4-byte aligned, owned by
 *                   the caller. Entries of blocks that hold any of a
 *                   sequence's first total_len[b] tokens must lie in
 *                   [0, num_blocks); the others are never read. An entry
 *                   outside the pool is read as block 0 (no memory outside the
 *                   pool is touched): a gathered key from such a block sets
 *                   bit 1 of the device status word, and dsa_cache_append_paged
 *                   writes nothing through such an entry.
 * Blocks may be shared between sequences (a common prefix); the append must
 * not write a block another sequence reads in the same step.
 */
typedef struct dsa_kv_pages {
  int32_t block_size;
  int32_t num_blocks;
  int32_t blocks_per_seq;
  const int32_t* block_table;
} dsa_kv_pages;

/* dsa_index_scores on a paged index-key pool (kI as described above). */
int dsa_index_scores_paged(const dsa_problem* p, const dsa_kv_pages* pages, const void* qI,
                           const float* w, const void* kI, float* scores, void* workspace,
                           size_t workspace_bytes, void* stream);

/* dsa_sparse_attn_decode on paged kI / K / V / scale pools. */
int dsa_sparse_attn_decode_paged(const dsa_problem* p, const dsa_kv_pages* pages, const void* q,
                                 const void* qI, const float* w, const void* kI, const void* k,
                                 const void* v, const float* k_scale, const float* v_scale,
                                 int32_t* idx_out, void* out, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* dsa_sparse_attn_prefill on paged kI / K / V / scale pools. */
int dsa_sparse_attn_prefill_paged(const dsa_problem* p, const dsa_kv_pages* pages, const void* q,
                                  const void* qI, const float* w, const void* kI, const void* k,
                                  const void* v, const float* k_scale, const float* v_scale,
                                  int32_t* idx_out, void* out, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* dsa_cache_append into paged pools: token s of sequence b goes to the pool
 * row of logical position total_len[b] - q_len + s. */
int dsa_cache_append_paged(const dsa_problem* p, const dsa_kv_pages* pages, const void* kI_new,
                           const void* k_new, const void* v_new, void* kI, void* k, void* v,
                           float* k_scale, float* v_scale, void* stream);

/*
 * Synchronises `stream`, then copies the device status word from the
 * workspace to *status_out (0 = no device-side problem; bit 0 = a bounded
 * wait ran out; bit 1 = a gathered key's block-table entry lay outside the
 * pool). Returns DSA_ERR_TIMEOUT if bit 0 is set, else DSA_ERR_INVALID_ARG if
 * bit 1 is set.
 */
int dsa_read_device_status(const void* workspace, size_t workspace_bytes,
                           void* stream, uint32_t* status_out);

/*
 * dsa_set_wait_budget -- how long the indexer's pipeline waits (TMA loads,
 * tensor-core results, accumulator hand-offs) may run before the kernel gives
 * up, for the calls that this host thread makes afterwards: `cycles` SM clock
 * cycles (0: a wait gives up unless it is complete at its first try), or any
 * negative value for the default of about a second. A kernel whose wait gives
 * up lets every copy and tensor-core operation it issued finish (those drains
 * keep the default budget), frees its tensor memory, sets the timeout bit of
 * the workspace status word (dsa_read_device_status then returns
 * DSA_ERR_TIMEOUT) and leaves the call's outputs undefined; the CUDA context
 * stays usable and the next call with the default budget is correct. A test
 * aid for the failure path: the pages have no counterpart. Returns DSA_OK.
 */
int dsa_set_wait_budget(long long cycles);

/* Message for the last failed call on this host thread ("" if none). */
const char* dsa_last_error_string(void);

/* Name of a status code. */
const char* dsa_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int dsa_version(void);

/*
 * dsa_last_launches -- the kernels that the last dsa_index_scores, dsa_topk,
 * dsa_topk_noalloc, dsa_cache_append, dsa_rmsnorm_rotary, dsa_rope_append,
 * dsa_sparse_attn_decode or
 * dsa_sparse_attn_prefill call (or its _paged form) on
 * this host thread enqueued. Returns how many (0 after a call that failed
 * before launching); when buf is not NULL, writes their names in launch order,
 * comma-separated and NUL-terminated, truncated to fit buflen bytes. No
 * counterpart in the pages: an accounting aid (a benchmark reports how many
 * of the library's kernels one step runs).
 */
int dsa_last_launches(char* buf, size_t buflen);

/*
 * Kernel timing (diagnostics). dsa_timing_select(kind) makes the following
 * calls on this host thread record a pair of CUDA events around every launch
 * of one kernel kind (DSA_KERNEL_*) on the caller's stream (-1 turns it off;
 * the events are recorded as external nodes under stream capture).
 * dsa_timing_read() waits for the most recent pair and returns its elapsed
 * milliseconds. Events are created on first use and kept for the thread.
 */
enum {
  DSA_KERNEL_INDEXER = 0,       /* tcgen05 indexer (decode and prefill)      */
  DSA_KERNEL_TOPK_HIST = 1,     /* chunk histograms (dsa_topk only)           */
  DSA_KERNEL_TOPK_SELECT = 2,   /* chunk select + final merge-and-emit        */
  DSA_KERNEL_TOPK_ROW = 3,      /* whole-row shared-memory select             */
  DSA_KERNEL_ATTENTION = 4,     /* sparse attention (+ split combine)         */
  DSA_KERNEL_APPEND = 5         /* cache append (dsa_cache_append)            */
};
int dsa_timing_select(int kernel_kind);
int dsa_timing_read(float* ms);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
