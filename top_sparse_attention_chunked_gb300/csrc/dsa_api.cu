// Host side of libdsa: argument validation, workspace layout, TMA descriptors
// and kernel dispatch behind the C ABI declared in include/dsa.h.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "dsa_internal.h"

namespace dsa {
namespace {

thread_local std::string g_err;
thread_local long long g_wait_budget = -1;  // < 0: the default budget
thread_local int g_timing_kind = -1;
thread_local cudaEvent_t g_ev[2] = {nullptr, nullptr};
thread_local bool g_ev_recorded = false;
constexpr int kLaunchLog = 16;
thread_local int g_nlaunch = 0;                       // kernels of the current call
thread_local const char* g_launch[kLaunchLog] = {};

}  // namespace

void note_launch(const char* name) {
  if (g_nlaunch < kLaunchLog) g_launch[g_nlaunch] = name;
  ++g_nlaunch;
}

void reset_launches() { g_nlaunch = 0; }

namespace {

int fail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(DSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// ------------------------------------------------------------------ device
struct DeviceInfo {
  int sms = 0;
  size_t smem_optin = 0;
  int major = 0, minor = 0;
};

int device_info(DeviceInfo* info) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  static bool have[64] = {};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DSA_ERR_NO_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 64) return fail(DSA_ERR_NO_DEVICE, "device ordinal %d out of range", dev);
  if (!have[dev]) {
    DeviceInfo d;
    int v = 0;
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(shared memory)");
    d.smem_optin = static_cast<size_t>(v);
    cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
    cache[dev] = d;
    have[dev] = true;
  }
  *info = cache[dev];
  if (info->major != 10)
    return fail(DSA_ERR_NO_DEVICE, "libdsa is built for sm_103a (Blackwell); device is sm_%d%d",
                info->major, info->minor);
  return DSA_OK;
}

// ------------------------------------------------------------------ TMA maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Encoded maps of this thread's recent calls: an encoding is a pure function
// of (kind, base, rows, box rows), and the same caches and query buffers come
// back call after call, so a hit skips the driver call.
struct MapCacheEntry {
  int kind;
  const void* base;
  long long rows;
  int box_rows;
  CUtensorMap map;
};
constexpr int kMapCache = 16;
thread_local MapCacheEntry g_map_cache[kMapCache];
thread_local int g_map_cache_n = 0, g_map_cache_next = 0;

bool map_cached(int kind, const void* base, long long rows, int box_rows, CUtensorMap* m) {
  for (int i = 0; i < g_map_cache_n; ++i) {
    const MapCacheEntry& e = g_map_cache[i];
    if (e.kind == kind && e.base == base && e.rows == rows && e.box_rows == box_rows) {
      *m = e.map;
      return true;
    }
  }
  return false;
}
void map_remember(int kind, const void* base, long long rows, int box_rows, const CUtensorMap& m) {
  MapCacheEntry& e = g_map_cache[g_map_cache_next];
  e = MapCacheEntry{kind, base, rows, box_rows, m};
  g_map_cache_next = (g_map_cache_next + 1) % kMapCache;
  if (g_map_cache_n < kMapCache) ++g_map_cache_n;
}

// rows x 64 bf16 matrix, box of box_rows x 64, 128-byte swizzle
int make_map_rows64(CUtensorMap* m, const void* base, long long rows, int box_rows) {
  if (map_cached(0, base, rows, box_rows, m)) return DSA_OK;
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(DSA_IDX_DIM), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(DSA_IDX_DIM) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(DSA_IDX_DIM), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  map_remember(0, base, rows, box_rows, *m);
  return DSA_OK;
}

// rows x 128 16-bit matrix (one KV head of one token per row), box 64 x 1,
// 128-byte swizzle: the source of TMA row gathers
int make_map_kv_rows(CUtensorMap* m, const void* base, long long rows) {
  if (map_cached(1, base, rows, 1, m)) return DSA_OK;
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(DSA_HEAD_DIM), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(DSA_HEAD_DIM) * 2};
  cuuint32_t box[2] = {64, 1};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled (KV rows) failed (%d)", (int)r);
  map_remember(1, base, rows, 1, *m);
  return DSA_OK;
}

// ------------------------------------------------------------------ problem checks
struct Derived {
  int rows = 0;        // B * S
  int max_n = 0;       // longest visible row
  int kmax = 0;        // largest k_eff
  int G = 0, HG = 0;   // group size, head groups per KV head
  int bm_words = 0;    // bitmap words per row
  long long kv_sb = 0, kv_st = 0, kv_sh = 0;   // K / V row strides (rows of 128 values)
  bool kv_default = true;                      // the token-major layout
};

int check_problem(const dsa_problem* p, int op, Derived* d) {
  if (!p) return fail(DSA_ERR_INVALID_ARG, "problem is NULL");
  if (p->batch < 1 || p->batch > DSA_MAX_BATCH)
    return fail(DSA_ERR_INVALID_ARG, "batch %d outside 1..%d", p->batch, DSA_MAX_BATCH);
  if (p->q_len < 1) return fail(DSA_ERR_INVALID_ARG, "q_len %d < 1", p->q_len);
  if (p->cache_capacity < 1 || p->cache_capacity > (1 << 30))
    return fail(DSA_ERR_INVALID_ARG, "cache_capacity %d invalid", p->cache_capacity);
  if (p->idx_heads != DSA_IDX_HEADS || p->idx_dim != DSA_IDX_DIM)
    return fail(DSA_ERR_UNSUPPORTED, "index heads x dim must be %dx%d (got %dx%d)",
                DSA_IDX_HEADS, DSA_IDX_DIM, p->idx_heads, p->idx_dim);
  if (p->top_k < 1 || p->top_k > p->cache_capacity)
    return fail(DSA_ERR_INVALID_ARG, "top_k %d outside 1..cache_capacity (%d)", p->top_k,
                p->cache_capacity);
  d->rows = p->batch * p->q_len;
  d->max_n = 0;
  for (int b = 0; b < p->batch; ++b) {
    const int T = p->total_len[b];
    if (T < p->q_len || T > p->cache_capacity)
      return fail(DSA_ERR_INVALID_ARG,
                  "total_len[%d] = %d outside q_len..cache_capacity (%d..%d)", b, T, p->q_len,
                  p->cache_capacity);
    if (T > d->max_n) d->max_n = T;
  }
  if (d->max_n > DSA_MAX_CONTEXT)
    return fail(DSA_ERR_UNSUPPORTED, "visible length %d above %d", d->max_n, DSA_MAX_CONTEXT);
  d->kmax = p->top_k < d->max_n ? p->top_k : d->max_n;
  d->bm_words = ceil_div(p->cache_capacity, 32);
  if (op == DSA_OP_DECODE || op == DSA_OP_PREFILL) {
    if (p->head_dim != DSA_HEAD_DIM)
      return fail(DSA_ERR_UNSUPPORTED, "head_dim must be %d (got %d)", DSA_HEAD_DIM, p->head_dim);
    if (p->num_q_heads < 1 || p->num_kv_heads < 1 || p->num_q_heads % p->num_kv_heads != 0)
      return fail(DSA_ERR_INVALID_ARG, "num_q_heads %d must be a multiple of num_kv_heads %d",
                  p->num_q_heads, p->num_kv_heads);
    if (p->q_dtype != DSA_BF16 && p->q_dtype != DSA_FP16)
      return fail(DSA_ERR_UNSUPPORTED, "q_dtype must be BF16 or FP16");
    if (p->kv_dtype != DSA_BF16 && p->kv_dtype != DSA_FP16 && p->kv_dtype != DSA_INT8)
      return fail(DSA_ERR_UNSUPPORTED, "kv_dtype must be BF16, FP16 or INT8");
    if (p->q_dtype == DSA_FP16 && p->kv_dtype == DSA_BF16)
      return fail(DSA_ERR_UNSUPPORTED, "FP16 query with a BF16 cache is not built");
    if (p->out_dtype != DSA_BF16 && p->out_dtype != DSA_FP16 && p->out_dtype != DSA_FP32)
      return fail(DSA_ERR_UNSUPPORTED, "out_dtype must be BF16, FP16 or FP32");
    if (p->attn_split_keys < 0 || p->attn_split_keys % 16 != 0 ||
        p->attn_split_keys > kAttnMaxSplitKeys)
      return fail(DSA_ERR_INVALID_ARG, "attn_split_keys %d must be 0 or a multiple of 16 up to %d",
                  p->attn_split_keys, kAttnMaxSplitKeys);
    if (!(p->softmax_scale >= 0.0f) || std::isinf(p->softmax_scale))
      return fail(DSA_ERR_INVALID_ARG, "softmax_scale must be finite and >= 0");
    d->G = p->num_q_heads / p->num_kv_heads;
    d->HG = ceil_div(d->G, kAttnRows);
  }
  if (op == DSA_OP_DECODE || op == DSA_OP_PREFILL) {
    const int64_t* ks = p->kv_strides;
    d->kv_default = (ks[0] == 0 && ks[1] == 0 && ks[2] == 0);
    if (d->kv_default) {
      d->kv_sb = static_cast<long long>(p->cache_capacity) * p->num_kv_heads;
      d->kv_st = p->num_kv_heads;
      d->kv_sh = 1;
    } else {
      for (int i = 0; i < 3; ++i)
        if (ks[i] < 0 || ks[i] % DSA_HEAD_DIM != 0)
          return fail(DSA_ERR_INVALID_ARG, "kv_strides[%d] = %lld must be a non-negative multiple of %d",
                      i, static_cast<long long>(ks[i]), DSA_HEAD_DIM);
      if (ks[1] < DSA_HEAD_DIM || (p->num_kv_heads > 1 && ks[2] < DSA_HEAD_DIM))
        return fail(DSA_ERR_INVALID_ARG, "kv_strides: the token stride (and, with several KV heads, "
                    "the head stride) must be at least %d", DSA_HEAD_DIM);
      d->kv_sb = ks[0] / DSA_HEAD_DIM;
      d->kv_st = ks[1] / DSA_HEAD_DIM;
      d->kv_sh = ks[2] / DSA_HEAD_DIM;
    }
  } else if (p->kv_strides[0] || p->kv_strides[1] || p->kv_strides[2]) {
    return fail(DSA_ERR_UNSUPPORTED, "kv_strides apply to the decode and prefill calls only");
  }
  if (op == DSA_OP_DECODE && p->q_len > DSA_MAX_DECODE_Q_LEN)
    return fail(DSA_ERR_UNSUPPORTED, "decode takes at most %d query tokens per sequence (got %d)",
                DSA_MAX_DECODE_Q_LEN, p->q_len);
  return DSA_OK;
}

// Automatic split count before rounding: enough CTAs for two per SM, and,
// while the grid stays within one wave of three CTAs per SM, at most 128 keys
// (two 16-key tiles per warp) per split; up to the 16 CTAs a cluster merges,
// never splits of fewer than 16 keys.
int auto_splits(const Derived& d, int units, int sms) {
  int s = std::max(ceil_div(2 * sms, units), std::min(ceil_div(d.kmax, 128), 3 * sms / units));
  s = std::min(s, 16);
  s = std::min(s, ceil_div(d.kmax, 16));
  return s < 1 ? 1 : s;
}

// Upper bound of the automatic split count (any GPU with <= 256 SMs).
int splits_bound(const dsa_problem* p, const Derived& d) {
  if (p->attn_split_keys > 0) return ceil_div(d.kmax, p->attn_split_keys);
  if (ceil_div(d.kmax, kAttnMaxSplitKeys) > 16) return kAttnMaxSplits;
  const int units = d.rows * p->num_kv_heads * d.HG;
  return auto_splits(d, units, 256);
}

// Actual split of the selected keys for the attention kernel.
void choose_split(const dsa_problem* p, const Derived& d, int sms, int* split_keys, int* nsplit) {
  int sk;
  if (p->attn_split_keys > 0) {
    sk = p->attn_split_keys;
  } else {
    const int units = d.rows * p->num_kv_heads * d.HG;
    int s = auto_splits(d, units, sms);
    if (s > attn_max_cluster()) s = attn_max_cluster();
    // a power of two (so the cluster combine splits the 128 columns evenly),
    // and no split longer than kAttnMaxSplitKeys
    const int s_min = ceil_div(d.kmax, kAttnMaxSplitKeys);
    int s2 = 1;
    while (s2 * 2 <= s) s2 *= 2;
    // clusters that do not all fit at once would run in a second wave:
    // halve the split count while the units need more clusters than fit
    while (s2 > 2 && s2 / 2 >= s_min && attn_uses_cluster(s2) && units > attn_cluster_capacity(s2))
      s2 /= 2;
    while (s2 < s_min) s2 *= 2;
    s = s2;
    sk = ceil_div(ceil_div(d.kmax, s), 16) * 16;
    const int sk_min = ceil_div(ceil_div(d.kmax, kAttnMaxSplits), 16) * 16;
    if (sk < sk_min) sk = sk_min;
  }
  *split_keys = sk;
  *nsplit = ceil_div(d.kmax, sk);
}

// ------------------------------------------------------------------ workspace
constexpr int kPrefillTopkGroup = 128;   // rows per chunked top-k round in prefill

struct Layout {
  size_t status = 0;
  size_t zero_begin = 0, zero_end = 0;
  size_t hist = 0, topk_ticket = 0, cand_count = 0, topk_zero_end = 0, attn_ticket = 0;
  size_t scores = 0, cands = 0, bitmap = 0, idx = 0, partial = 0;
  long long cand_stride = 0;
  int topk_rows = 0;   // rows the top-k scratch covers
  size_t total = 0;
};

Layout layout(const dsa_problem* p, int op, const Derived& d) {
  Layout L;
  size_t o = 256;   // status word
  const bool attn = (op == DSA_OP_DECODE || op == DSA_OP_PREFILL);
  const bool topk = (op != DSA_OP_INDEX_SCORES);
  L.topk_rows = (op == DSA_OP_PREFILL && d.rows > kPrefillTopkGroup) ? kPrefillTopkGroup : d.rows;
  const int units = attn ? d.rows * p->num_kv_heads * d.HG : 0;
  L.zero_begin = o;
  if (topk) {
    L.hist = o;        o = up256(o + static_cast<size_t>(L.topk_rows) * kHistBins * 4);
    L.topk_ticket = o; o = up256(o + static_cast<size_t>(L.topk_rows) * 4);
    L.cand_count = o;  o = up256(o + static_cast<size_t>(L.topk_rows) * 4);
    L.topk_zero_end = o;
  }
  if (attn) {
    L.attn_ticket = o; o = up256(o + static_cast<size_t>(units) * 4);
  }
  L.zero_end = o;
  if (attn) {
    L.scores = o; o = up256(o + static_cast<size_t>(d.rows) * p->cache_capacity * 4);
  }
  if (topk) {
    L.cand_stride = d.max_n;
    L.cands = o;  o = up256(o + static_cast<size_t>(L.topk_rows) * d.max_n * 8);
    L.bitmap = o; o = up256(o + static_cast<size_t>(L.topk_rows) * d.bm_words * 4);
  }
  if (attn) {
    L.idx = o;     o = up256(o + static_cast<size_t>(d.rows) * p->top_k * 4);
    const int ns = splits_bound(p, d);
    if (ns > 1) {
      L.partial = o;
      o = up256(o + static_cast<size_t>(units) * ns * kPartialFloats * 4);
    }
  }
  L.total = o;
  return L;
}

int check_ws(void* ws, size_t bytes, const Layout& L) {
  if (!ws) return fail(DSA_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(ws, 256)) return fail(DSA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (bytes < L.total)
    return fail(DSA_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", bytes, L.total);
  return DSA_OK;
}

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

SeqLens lens_of(const dsa_problem* p) {
  SeqLens s;
  memset(&s, 0, sizeof(s));
  for (int b = 0; b < p->batch; ++b) s.T[b] = p->total_len[b];
  return s;
}

// Cache rows (tokens) the kI / K / V arrays hold: the dense [B, cap] layout or
// the paged pool.
long long pool_tokens(const dsa_problem* p, const Paging& pg) {
  return pg.table ? (static_cast<long long>(pg.num_blocks) << pg.shift)
                  : static_cast<long long>(p->batch) * p->cache_capacity;
}

const Paging kDense = {nullptr, 0, 0, 0};

// Calls that take only the token-major K / V layout.
int check_default_layout(const dsa_problem* p) {
  if (p->kv_strides[0] || p->kv_strides[1] || p->kv_strides[2])
    return fail(DSA_ERR_UNSUPPORTED, "paged caches and cache writes take only the default kv_strides");
  return DSA_OK;
}

// Validates a paged-cache descriptor against the problem and fills *pg.
int check_pages(const dsa_problem* p, const dsa_kv_pages* pages, Paging* pg) {
  if (!pages) return fail(DSA_ERR_INVALID_ARG, "pages is NULL");
  if (int rc = check_default_layout(p)) return rc;
  const int bs = pages->block_size;
  if (bs < 128 || bs > (1 << 20) || (bs & (bs - 1)) != 0)
    return fail(DSA_ERR_UNSUPPORTED, "block_size %d must be a power of two from 128 to 2^20", bs);
  if (pages->num_blocks < 1) return fail(DSA_ERR_INVALID_ARG, "num_blocks %d < 1", pages->num_blocks);
  if (pages->blocks_per_seq < 1)
    return fail(DSA_ERR_INVALID_ARG, "blocks_per_seq %d < 1", pages->blocks_per_seq);
  if (static_cast<long long>(pages->blocks_per_seq) * bs != p->cache_capacity)
    return fail(DSA_ERR_INVALID_ARG, "cache_capacity %d must equal blocks_per_seq * block_size (%lld)",
                p->cache_capacity, static_cast<long long>(pages->blocks_per_seq) * bs);
  if (!pages->block_table) return fail(DSA_ERR_INVALID_ARG, "block_table is NULL");
  if (!aligned(pages->block_table, 4)) return fail(DSA_ERR_MISALIGNED, "block_table must be 4-byte aligned");
  if ((static_cast<long long>(pages->num_blocks) * bs) * std::max(1, p->num_kv_heads) >= (1LL << 31))
    return fail(DSA_ERR_UNSUPPORTED, "num_blocks * block_size * num_kv_heads must be below 2^31");
  int shift = 0;
  while ((1 << shift) < bs) ++shift;
  *pg = Paging{pages->block_table, pages->blocks_per_seq, shift, pages->num_blocks};
  return DSA_OK;
}

int pow2_at_least(int x) {
  int v = 1;
  while (v < x) v <<= 1;
  return v;
}

// ------------------------------------------------------------------ stages
int run_indexer(const dsa_problem* p, const Derived& d, const DeviceInfo& di, const Paging& pg,
                const void* qI, const float* w, const void* kI, float* scores, uint32_t* hist,
                uint32_t* status, cudaStream_t st) {
  IndexerParams ip{};
  ip.pg = pg;
  ip.w = w;
  ip.scores = scores;
  ip.hist = hist;
  ip.status = status;
  ip.B = p->batch;
  ip.S = p->q_len;
  ip.cap = p->cache_capacity;
  ip.QB = p->q_len <= 16 ? pow2_at_least(p->q_len) : 16;
  ip.nqb = ceil_div(p->q_len, ip.QB);
  ip.lens = lens_of(p);
  long long total = 0;
  long long per_seq_max = 0;
  for (int b = 0; b < p->batch; ++b) {
    long long nb = 0;
    for (int qb = 0; qb < ip.nqb; ++qb) {
      const int last_s = std::min(p->q_len, (qb + 1) * ip.QB) - 1;
      const int n = p->total_len[b] - p->q_len + last_s + 1;
      nb += ceil_div(n, kKeyTile);
    }
    total += nb;
    if (nb > per_seq_max) per_seq_max = nb;
  }
  ip.total_units = total;
  ip.wait_budget = g_wait_budget >= 0 ? g_wait_budget : kDefaultWaitBudget;
  CUtensorMap tm_kI, tm_qI;
  int rc = make_map_rows64(&tm_kI, kI, pool_tokens(p, pg), kKeyTile);
  if (rc) return rc;
  rc = make_map_rows64(&tm_qI, qI, static_cast<long long>(d.rows) * DSA_IDX_HEADS, ip.QB * 16);
  if (rc) return rc;
  int stages = 0;
  const size_t smem = indexer_smem_bytes(ip.QB, hist != nullptr, &stages, di.smem_optin);
  if (smem > di.smem_optin) return fail(DSA_ERR_UNSUPPORTED, "indexer needs %zu B of shared memory", smem);
  dim3 grid;
  if (hist) {
    // CTAs per sequence, so each CTA's histograms belong to one sequence
    long long per = ceil_div(di.sms, p->batch);
    if (per > per_seq_max) per = per_seq_max;
    if (per < 1) per = 1;
    grid = dim3(static_cast<unsigned>(per), static_cast<unsigned>(p->batch));
    if (p->batch == 1) grid.y = 1;   // one sequence: the flat split is the same
  } else {
    grid = dim3(static_cast<unsigned>(total < di.sms ? total : di.sms));
  }
  timing_before(DSA_KERNEL_INDEXER, st);
  cudaError_t e = launch_indexer(ip, tm_kI, tm_qI, grid, smem, stages, st);
  timing_after(DSA_KERNEL_INDEXER, st);
  if (e != cudaSuccess) return cuda_fail(e, "indexer launch");
  return DSA_OK;
}

// The decode's caches, for the top-k's L2 prefetch of the selected rows.
struct KvPrefetch {
  const void* k;
  const void* v;
  const float* ks;
  const float* vs;
  Paging pg;
};

int run_topk(const dsa_problem* p, const Derived& d, const DeviceInfo& di, const Layout& L,
             const float* scores, int32_t* idx, void* ws, bool hist_ready, bool prefer_rows,
             bool after_kernel, cudaStream_t st, const KvPrefetch* pf = nullptr) {
  TopkParams tp{};
  tp.status = at<uint32_t>(ws, 0);
  if (pf) {
    const int elem = p->kv_dtype == DSA_INT8 ? 1 : 2;
    tp.pf_k = static_cast<const uint8_t*>(pf->k);
    tp.pf_v = static_cast<const uint8_t*>(pf->v);
    tp.pf_ks = pf->ks;
    tp.pf_vs = pf->vs;
    tp.pf_row_bytes = p->num_kv_heads * DSA_HEAD_DIM * elem;
    tp.pf_heads = p->num_kv_heads;
    tp.pg = pf->pg;
  }
  tp.scores = scores;
  tp.idx = idx;
  tp.hist = at<uint32_t>(ws, L.hist);
  tp.ticket = at<uint32_t>(ws, L.topk_ticket);
  tp.cand_count = at<uint32_t>(ws, L.cand_count);
  tp.cands = at<unsigned long long>(ws, L.cands);
  tp.bitmap = at<uint32_t>(ws, L.bitmap);
  tp.cand_stride = L.cand_stride;
  tp.bitmap_stride = d.bm_words;
  tp.B = p->batch;
  tp.S = p->q_len;
  tp.cap = p->cache_capacity;
  tp.k = p->top_k;
  tp.nchunks = ceil_div(d.max_n, kChunk);
  tp.lens = lens_of(p);
  tp.row0 = 0;
  tp.nrows = d.rows;
  cudaError_t e;
  const int row_max = topk_row_max_len(di.smem_optin);
  if (!hist_ready && prefer_rows && d.max_n <= topk_row_stream_max_len()) {
    timing_before(DSA_KERNEL_TOPK_ROW, st);
    e = launch_topk_row_stream(tp, d.max_n, after_kernel, st);
    timing_after(DSA_KERNEL_TOPK_ROW, st);
    if (e != cudaSuccess) return cuda_fail(e, "top-k row launch");
    return DSA_OK;
  }
  if (!hist_ready && prefer_rows && d.max_n <= row_max) {
    timing_before(DSA_KERNEL_TOPK_ROW, st);
    if (topk_row_reg_per(d.max_n) > 0)
      e = launch_topk_row_reg(tp, d.max_n, after_kernel, st);
    else
      e = launch_topk_row(tp, d.max_n, di.smem_optin, after_kernel, st);
    timing_after(DSA_KERNEL_TOPK_ROW, st);
    if (e != cudaSuccess) return cuda_fail(e, "top-k row launch");
    return DSA_OK;
  }
  tp.hist_ready = hist_ready ? 1 : 0;
  if (topk_cluster_ctas(d.max_n) > 0 && topk_cluster_feasible(d.max_n)) {
    // one cluster per row (it builds the row histogram itself unless the
    // indexer did); no other scratch
    timing_before(DSA_KERNEL_TOPK_SELECT, st);
    e = launch_topk_cluster_select(tp, d.max_n, after_kernel, st);
    timing_after(DSA_KERNEL_TOPK_SELECT, st);
    if (e == cudaSuccess) return DSA_OK;
    if (e != cudaErrorNotSupported) return cuda_fail(e, "top-k cluster launch");
  }
  // chunked path, in rounds of at most L.topk_rows rows
  for (int r0 = 0; r0 < d.rows; r0 += L.topk_rows) {
    tp.row0 = r0;
    tp.nrows = std::min(L.topk_rows, d.rows - r0);
    if (!hist_ready) {
      e = cudaMemsetAsync(static_cast<uint8_t*>(ws) + L.hist, 0, L.topk_zero_end - L.hist, st);
      if (e != cudaSuccess) return cuda_fail(e, "workspace clear");
      timing_before(DSA_KERNEL_TOPK_HIST, st);
      e = launch_topk_hist(tp, st);
      timing_after(DSA_KERNEL_TOPK_HIST, st);
      if (e != cudaSuccess) return cuda_fail(e, "top-k histogram launch");
    }
    timing_before(DSA_KERNEL_TOPK_SELECT, st);
    e = launch_topk_chunk_select(tp, st);
    timing_after(DSA_KERNEL_TOPK_SELECT, st);
    if (e != cudaSuccess) return cuda_fail(e, "top-k select launch");
  }
  return DSA_OK;
}

int run_attention(const dsa_problem* p, const Derived& d, const DeviceInfo& di, const Layout& L,
                  const Paging& pg, const void* q, const void* k, const void* v, const float* ks,
                  const float* vs, const int32_t* idx, void* out, void* ws, bool prefill,
                  cudaStream_t st, const void* k_aux = nullptr, const void* v_aux = nullptr) {
  AttnParams ap{};
  ap.k_aux = k_aux;
  ap.v_aux = v_aux;
  ap.pg = pg;
  ap.q = q;
  ap.k = k;
  ap.v = v;
  ap.k_scale = ks;
  ap.v_scale = vs;
  ap.idx = idx;
  ap.out = out;
  ap.partial = L.partial ? at<float>(ws, L.partial) : nullptr;
  ap.ticket = at<uint32_t>(ws, L.attn_ticket);
  ap.B = p->batch;
  ap.S = p->q_len;
  ap.Hq = p->num_q_heads;
  ap.Hkv = p->num_kv_heads;
  ap.G = d.G;
  ap.HG = d.HG;
  ap.cap = p->cache_capacity;
  ap.topk = p->top_k;
  ap.kv_sb = d.kv_sb;
  ap.kv_st = d.kv_st;
  ap.kv_sh = d.kv_sh;
  ap.scale_rows = pool_tokens(p, pg) * p->num_kv_heads;
  choose_split(p, d, di.sms, &ap.split_keys, &ap.nsplit);
  if (ap.nsplit > kAttnMaxSplits)
    return fail(DSA_ERR_UNSUPPORTED, "attn_split_keys %d gives %d splits (max %d)",
                p->attn_split_keys, ap.nsplit, kAttnMaxSplits);
  if (ap.nsplit > splits_bound(p, d))
    return fail(DSA_ERR_UNSUPPORTED, "device has more SMs than the workspace bound assumes");
  const float scale = p->softmax_scale > 0.0f ? p->softmax_scale
                                              : 1.0f / std::sqrt(static_cast<float>(p->head_dim));
  ap.scale_log2 = scale * 1.4426950408889634f;
  ap.lens = lens_of(p);
  ap.q_dtype = p->q_dtype;
  ap.out_dtype = p->out_dtype;
  ap.cluster = attn_uses_cluster(ap.nsplit) ? 1 : 0;
  ap.status = at<uint32_t>(ws, 0);
  cudaError_t e;
  timing_before(DSA_KERNEL_ATTENTION, st);
  // K / V rows the caches span (the row maps' extent): the pool's, or the
  // last (batch, token, head) row of the strided layout plus one
  const long long kv_rows =
      pg.table ? pool_tokens(p, pg) * p->num_kv_heads
               : (p->batch - 1) * d.kv_sb + (p->cache_capacity - 1LL) * d.kv_st +
                     (p->num_kv_heads - 1LL) * d.kv_sh + 1;
  ap.kv_rows = kv_rows;
  if (prefill && p->attn_split_keys == 0 && prefill_tc_supported(ap, p->kv_dtype, di.smem_optin)) {
    CUtensorMap tm_k, tm_v;
    const long long rows = kv_rows;
    if (rows >= (1LL << 31)) {
      timing_after(DSA_KERNEL_ATTENTION, st);
      return fail(DSA_ERR_UNSUPPORTED, "the K / V caches must span fewer than 2^31 rows");
    }
    int rc = make_map_kv_rows(&tm_k, k, rows);
    if (rc == DSA_OK) rc = make_map_kv_rows(&tm_v, v, rows);
    if (rc != DSA_OK) {
      timing_after(DSA_KERNEL_ATTENTION, st);
      return rc;
    }
    e = launch_prefill_tc(ap, p->kv_dtype, di.sms, tm_k, tm_v, at<uint32_t>(ws, 0), st);
  } else {
    // row gathers (16-bit caches) address rows with signed 32-bit coordinates
    const long long rows = kv_rows;
    if (p->kv_dtype != DSA_INT8 && rows >= (1LL << 31)) {
      timing_after(DSA_KERNEL_ATTENTION, st);
      return fail(DSA_ERR_UNSUPPORTED, "cache rows * num_kv_heads must be below 2^31");
    }
    CUtensorMap tm_k{}, tm_v{};   // INT8 caches are gathered with cp.async
    int rc = DSA_OK;
    if (p->kv_dtype != DSA_INT8) {
      rc = make_map_kv_rows(&tm_k, k, rows);
      if (rc == DSA_OK) rc = make_map_kv_rows(&tm_v, v, rows);
    }
    if (rc != DSA_OK) {
      timing_after(DSA_KERNEL_ATTENTION, st);
      return rc;
    }
    e = launch_attention(ap, p->q_dtype, p->kv_dtype, p->out_dtype, tm_k, tm_v, st);
  }
  timing_after(DSA_KERNEL_ATTENTION, st);
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return DSA_OK;
}

bool prefill_tc_ok(const dsa_problem* p, const Derived& d, const DeviceInfo& di, const Paging& pg) {
  AttnParams ap{};
  ap.pg = pg;
  ap.topk = p->top_k;
  ap.B = p->batch;
  ap.cap = p->cache_capacity;
  ap.Hkv = p->num_kv_heads;
  (void)d;
  return prefill_tc_supported(ap, p->kv_dtype, di.smem_optin);
}

int check_attn_ptrs(const dsa_problem* p, const void* q, const void* qI, const float* w,
                    const void* kI, const void* k, const void* v, const float* ks,
                    const float* vs, const int32_t* idx_out, const void* out) {
  if (!q || !qI || !w || !kI || !k || !v || !out)
    return fail(DSA_ERR_INVALID_ARG, "a required tensor pointer is NULL");
  if (p->kv_dtype == DSA_INT8) {
    if (!ks || !vs) return fail(DSA_ERR_INVALID_ARG, "INT8 cache needs k_scale and v_scale");
    if (!aligned(ks, 4) || !aligned(vs, 4)) return fail(DSA_ERR_MISALIGNED, "scales must be 4-byte aligned");
  } else if (ks || vs) {
    return fail(DSA_ERR_INVALID_ARG, "k_scale/v_scale must be NULL unless the cache is INT8");
  }
  if (!aligned(q, 16) || !aligned(qI, 16) || !aligned(kI, 16) || !aligned(k, 16) ||
      !aligned(v, 16))
    return fail(DSA_ERR_MISALIGNED, "q, qI, kI, k and v must be 16-byte aligned");
  if (!aligned(w, 4) || !aligned(out, 4) || (idx_out && !aligned(idx_out, 4)))
    return fail(DSA_ERR_MISALIGNED, "w, out and idx_out must be 4-byte aligned");
  return DSA_OK;
}

int attn_call(const dsa_problem* p, int op, const Paging& pg, const void* q, const void* qI, const float* w,
              const void* kI, const void* k, const void* v, const float* ks, const float* vs,
              int32_t* idx_out, void* out, void* ws, size_t ws_bytes, void* stream,
              const void* k_aux = nullptr, const void* v_aux = nullptr) {
  reset_launches();
  Derived d;
  int rc = check_problem(p, op, &d);
  if (rc) return rc;
  rc = check_attn_ptrs(p, q, qI, w, kI, k, v, ks, vs, idx_out, out);
  if (rc) return rc;
  const Layout L = layout(p, op, d);
  rc = check_ws(ws, ws_bytes, L);
  if (rc) return rc;
  DeviceInfo di;
  rc = device_info(&di);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool decode = (op == DSA_OP_DECODE);
  // Which kernels run decides what scratch must start at zero: the chunked
  // top-k needs its histograms, tickets and counters cleared, the split-K
  // attention outside a cluster its tickets. Otherwise nothing is cleared
  // (the indexer resets the status word itself).
  const bool topk_rows = !decode && (d.max_n <= topk_row_stream_max_len() ||
                                     d.max_n <= topk_row_max_len(di.smem_optin));
  // decode: the indexer epilogue builds the top-k's row histograms
  const bool hist_in_indexer = decode;
  int split_keys = 0, nsplit = 1;
  choose_split(p, d, di.sms, &split_keys, &nsplit);
  const bool tc_prefill = !decode && p->attn_split_keys == 0 && prefill_tc_ok(p, d, di, pg);
  const bool attn_tickets = !tc_prefill && nsplit > 1 && !attn_uses_cluster(nsplit);
  if (hist_in_indexer || attn_tickets) {
    // histograms, tickets and counters start at zero; the clearing kernel
    // overlaps the indexer, which waits for it only before its final flush
    cudaError_t e = launch_zero_scratch(at<uint8_t>(ws, L.zero_begin), L.zero_end - L.zero_begin, st);
    if (e != cudaSuccess) return cuda_fail(e, "workspace clear");
  }
  float* scores = at<float>(ws, L.scores);
  int32_t* idx = idx_out ? idx_out : at<int32_t>(ws, L.idx);
  uint32_t* status = at<uint32_t>(ws, 0);
  rc = run_indexer(p, d, di, pg, qI, w, kI, scores, hist_in_indexer ? at<uint32_t>(ws, L.hist) : nullptr,
                   status, st);
  if (rc) return rc;
  const KvPrefetch pf{k, v, ks, vs, pg};
  // the prefetch takes a token's rows of all KV heads as one span
  rc = run_topk(p, d, di, L, scores, idx, ws, hist_in_indexer, topk_rows, true, st,
                decode && d.kv_default ? &pf : nullptr);
  if (rc) return rc;
  return run_attention(p, d, di, L, pg, q, k, v, ks, vs, idx, out, ws, !decode, st, k_aux, v_aux);
}

int index_call(const dsa_problem* p, const dsa_kv_pages* pages, const void* qI, const float* w,
               const void* kI, float* scores, void* ws, size_t ws_bytes, void* stream) {
  reset_launches();
  Derived d;
  int rc = check_problem(p, DSA_OP_INDEX_SCORES, &d);
  if (rc) return rc;
  Paging pg = kDense;
  if (pages && (rc = check_pages(p, pages, &pg))) return rc;
  if (!qI || !w || !kI || !scores) return fail(DSA_ERR_INVALID_ARG, "a tensor pointer is NULL");
  if (!aligned(qI, 16) || !aligned(kI, 16) || !aligned(scores, 16) || !aligned(w, 4))
    return fail(DSA_ERR_MISALIGNED, "qI, kI and scores must be 16-byte aligned, w 4-byte");
  const Layout L = layout(p, DSA_OP_INDEX_SCORES, d);
  rc = check_ws(ws, ws_bytes, L);
  if (rc) return rc;
  DeviceInfo di;
  rc = device_info(&di);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws, 0, 256, st);
  if (e != cudaSuccess) return cuda_fail(e, "workspace clear");
  return run_indexer(p, d, di, pg, qI, w, kI, scores, nullptr, at<uint32_t>(ws, 0), st);
}

int attn_entry(const dsa_problem* p, int op, const dsa_kv_pages* pages, const void* q,
               const void* qI, const float* w, const void* kI, const void* k, const void* v,
               const float* ks, const float* vs, int32_t* idx_out, void* out, void* ws,
               size_t ws_bytes, void* stream) {
  Paging pg = kDense;
  if (pages) {
    reset_launches();
    Derived d;
    int rc = check_problem(p, op, &d);
    if (rc) return rc;
    if ((rc = check_pages(p, pages, &pg))) return rc;
  }
  return attn_call(p, op, pg, q, qI, w, kI, k, v, ks, vs, idx_out, out, ws, ws_bytes, stream);
}

}  // namespace

// ------------------------------------------------------------------ kernel attributes
namespace {
using CtxGetCurrentFn2 = int (*)(void**);   // cuCtxGetCurrent(CUcontext*)
CtxGetCurrentFn2 ctx_current_fn() {
  static CtxGetCurrentFn2 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn2>(f);
  });
  return fn;
}
struct AttrEntry {
  const void* kern;
  void* ctx;
  int attr, value;
};
std::mutex g_attr_mu;
AttrEntry g_attr[256];
int g_attr_n = 0;

cudaError_t set_attr_once(const void* kern, cudaFuncAttribute attr, int value) {
  void* ctx = nullptr;
  CtxGetCurrentFn2 fn = ctx_current_fn();
  if (!fn || fn(&ctx) != 0 || !ctx) return cudaFuncSetAttribute(kern, attr, value);
  std::lock_guard<std::mutex> lock(g_attr_mu);
  for (int i = 0; i < g_attr_n; ++i) {
    AttrEntry& e = g_attr[i];
    if (e.kern == kern && e.ctx == ctx && e.attr == static_cast<int>(attr)) {
      if (e.value == value) return cudaSuccess;
      const cudaError_t r = cudaFuncSetAttribute(kern, attr, value);
      if (r == cudaSuccess) e.value = value;
      return r;
    }
  }
  const cudaError_t r = cudaFuncSetAttribute(kern, attr, value);
  if (r == cudaSuccess && g_attr_n < 256) g_attr[g_attr_n++] = AttrEntry{kern, ctx, static_cast<int>(attr), value};
  return r;
}
}  // namespace

cudaError_t set_max_smem(const void* kern, int bytes) {
  return set_attr_once(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}
cudaError_t set_nonportable_cluster(const void* kern) {
  return set_attr_once(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

// ------------------------------------------------------------------ no-alloc top-k helpers
int noalloc_fail(int status, const char* msg) { return fail(status, "%s", msg); }

// Records a failure of a call implemented in another translation unit.
int report_error(int status, const char* msg) { return fail(status, "%s", msg); }

// Problem validation for calls that write caches (any q_len, as for prefill).
int problem_check_for_append(const dsa_problem* p) {
  Derived d;
  if (int rc = check_problem(p, DSA_OP_PREFILL, &d)) return rc;
  return check_default_layout(p);
}

int noalloc_check_topk(const dsa_problem* p, int* rows, int* max_n) {
  reset_launches();
  Derived d;
  const int rc = check_problem(p, DSA_OP_TOPK, &d);
  if (rc) return rc;
  *rows = d.rows;
  *max_n = d.max_n;
  return DSA_OK;
}

// ------------------------------------------------------------------ timing hook
void timing_before(int kind, cudaStream_t st) {
  if (kind != g_timing_kind) return;
  if (!g_ev[0]) {
    cudaEventCreate(&g_ev[0]);
    cudaEventCreate(&g_ev[1]);
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(st, &cs);
  if (cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(g_ev[0], st, cudaEventRecordExternal);
  else
    cudaEventRecord(g_ev[0], st);
}

void timing_after(int kind, cudaStream_t st) {
  if (kind != g_timing_kind || !g_ev[1]) return;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(st, &cs);
  if (cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(g_ev[1], st, cudaEventRecordExternal);
  else
    cudaEventRecord(g_ev[1], st);
  g_ev_recorded = true;
}

}  // namespace dsa

// ====================================================================== C ABI
using namespace dsa;

extern "C" {

size_t dsa_workspace_size(const dsa_problem* p, int op) {
  if (op < DSA_OP_INDEX_SCORES || op > DSA_OP_PREFILL) {
    fail(DSA_ERR_INVALID_ARG, "unknown op %d", op);
    return 0;
  }
  Derived d;
  if (check_problem(p, op, &d)) return 0;
  return layout(p, op, d).total;
}

int dsa_index_scores(const dsa_problem* p, const void* qI, const float* w, const void* kI,
                     float* scores, void* ws, size_t ws_bytes, void* stream) {
  return index_call(p, nullptr, qI, w, kI, scores, ws, ws_bytes, stream);
}

int dsa_index_scores_paged(const dsa_problem* p, const dsa_kv_pages* pages, const void* qI,
                           const float* w, const void* kI, float* scores, void* ws,
                           size_t ws_bytes, void* stream) {
  if (!pages) {
    reset_launches();
    return fail(DSA_ERR_INVALID_ARG, "pages is NULL");
  }
  return index_call(p, pages, qI, w, kI, scores, ws, ws_bytes, stream);
}

int dsa_topk(const dsa_problem* p, const float* scores, int32_t* idx, void* ws, size_t ws_bytes,
             void* stream) {
  reset_launches();
  Derived d;
  int rc = check_problem(p, DSA_OP_TOPK, &d);
  if (rc) return rc;
  if (!scores || !idx) return fail(DSA_ERR_INVALID_ARG, "a tensor pointer is NULL");
  if (!aligned(scores, 4) || !aligned(idx, 4))
    return fail(DSA_ERR_MISALIGNED, "scores and idx must be 4-byte aligned");
  const Layout L = layout(p, DSA_OP_TOPK, d);
  rc = check_ws(ws, ws_bytes, L);
  if (rc) return rc;
  DeviceInfo di;
  rc = device_info(&di);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws, 0, 256, st);
  if (e != cudaSuccess) return cuda_fail(e, "workspace clear");
  // few rows: spread each row over its chunks; many short rows: one CTA per row
  const bool prefer_rows = d.rows >= 2 * di.sms;
  return run_topk(p, d, di, L, scores, idx, ws, false, prefer_rows, false, st);
}

int dsa_sparse_attn_decode_aux(const dsa_problem* p, const void* q, const void* qI, const float* w,
                               const void* kI, const void* k, const void* v, const float* k_scale,
                               const float* v_scale, const void* k_aux, const void* v_aux,
                               int32_t* idx_out, void* out, void* ws, size_t ws_bytes,
                               void* stream) {
  reset_launches();
  if (!k_aux || !v_aux) return fail(DSA_ERR_INVALID_ARG, "k_aux and v_aux are required");
  if (!aligned(k_aux, 16) || !aligned(v_aux, 16))
    return fail(DSA_ERR_MISALIGNED, "k_aux and v_aux must be 16-byte aligned");
  return attn_call(p, DSA_OP_DECODE, kDense, q, qI, w, kI, k, v, k_scale, v_scale, idx_out, out, ws,
                   ws_bytes, stream, k_aux, v_aux);
}

int dsa_sparse_attn_decode(const dsa_problem* p, const void* q, const void* qI, const float* w,
                           const void* kI, const void* k, const void* v, const float* k_scale,
                           const float* v_scale, int32_t* idx_out, void* out, void* ws,
                           size_t ws_bytes, void* stream) {
  return attn_entry(p, DSA_OP_DECODE, nullptr, q, qI, w, kI, k, v, k_scale, v_scale, idx_out, out, ws,
                   ws_bytes, stream);
}

int dsa_sparse_attn_prefill(const dsa_problem* p, const void* q, const void* qI, const float* w,
                            const void* kI, const void* k, const void* v, const float* k_scale,
                            const float* v_scale, int32_t* idx_out, void* out, void* ws,
                            size_t ws_bytes, void* stream) {
  return attn_entry(p, DSA_OP_PREFILL, nullptr, q, qI, w, kI, k, v, k_scale, v_scale, idx_out, out, ws,
                   ws_bytes, stream);
}

static int append_call(const dsa_problem* p, const dsa_kv_pages* pages, const void* kI_new,
                       const void* k_new, const void* v_new, void* kI, void* k, void* v,
                       float* k_scale, float* v_scale, void* stream) {
  reset_launches();
  Derived d;
  int rc = check_problem(p, DSA_OP_PREFILL, &d);
  if (rc) return rc;
  if ((rc = check_default_layout(p))) return rc;
  Paging pg = kDense;
  if (pages && (rc = check_pages(p, pages, &pg))) return rc;
  if (!kI_new || !k_new || !v_new || !kI || !k || !v)
    return fail(DSA_ERR_INVALID_ARG, "a required tensor pointer is NULL");
  const bool int8 = (p->kv_dtype == DSA_INT8);
  if (int8) {
    if (!k_scale || !v_scale) return fail(DSA_ERR_INVALID_ARG, "INT8 cache needs k_scale and v_scale");
    if (!aligned(k_scale, 4) || !aligned(v_scale, 4))
      return fail(DSA_ERR_MISALIGNED, "scales must be 4-byte aligned");
  } else if (k_scale || v_scale) {
    return fail(DSA_ERR_INVALID_ARG, "k_scale/v_scale must be NULL unless the cache is INT8");
  }
  if (!aligned(kI_new, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(kI, 16) ||
      !aligned(k, 16) || !aligned(v, 16))
    return fail(DSA_ERR_MISALIGNED, "kI_new, k_new, v_new, kI, k and v must be 16-byte aligned");
  // the new tokens are read while the caches are written: no input may overlap an output
  const long long B = p->batch, S = p->q_len, H = p->num_kv_heads;
  const long long rows = pool_tokens(p, pg);   // cache rows (dense or the pool)
  struct Span { const void* p; long long n; };
  const Span in[3] = {{kI_new, B * S * DSA_IDX_DIM * 2}, {k_new, B * S * H * DSA_HEAD_DIM * 2},
                      {v_new, B * S * H * DSA_HEAD_DIM * 2}};
  const long long row_bytes = int8 ? DSA_HEAD_DIM : DSA_HEAD_DIM * 2;
  const Span out[5] = {{kI, rows * DSA_IDX_DIM * 2}, {k, rows * H * row_bytes},
                       {v, rows * H * row_bytes}, {k_scale, int8 ? rows * H * 4 : 0},
                       {v_scale, int8 ? rows * H * 4 : 0}};
  for (const Span& a : in)
    for (const Span& o : out) {
      const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), o0 = reinterpret_cast<uintptr_t>(o.p);
      if (o.n > 0 && a0 < o0 + static_cast<uintptr_t>(o.n) && o0 < a0 + static_cast<uintptr_t>(a.n))
        return fail(DSA_ERR_INVALID_ARG, "a new-token tensor overlaps a cache");
    }
  DeviceInfo di;
  rc = device_info(&di);
  if (rc) return rc;
  AppendParams ap{};
  ap.kI_new = kI_new;
  ap.k_new = k_new;
  ap.v_new = v_new;
  ap.kI = kI;
  ap.k = k;
  ap.v = v;
  ap.k_scale = k_scale;
  ap.v_scale = v_scale;
  ap.B = p->batch;
  ap.S = p->q_len;
  ap.Hkv = p->num_kv_heads;
  ap.cap = p->cache_capacity;
  ap.q_dtype = p->q_dtype;
  ap.kv_dtype = p->kv_dtype;
  ap.pg = pg;
  for (int b = 0; b < p->batch; ++b) ap.lens.T[b] = p->total_len[b];
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  timing_before(DSA_KERNEL_APPEND, st);
  const cudaError_t e = launch_cache_append(ap, di.sms, st);
  if (e != cudaSuccess) return cuda_fail(e, "cache append launch");
  timing_after(DSA_KERNEL_APPEND, st);
  return DSA_OK;
}

int dsa_cache_append(const dsa_problem* p, const void* kI_new, const void* k_new,
                     const void* v_new, void* kI, void* k, void* v, float* k_scale,
                     float* v_scale, void* stream) {
  return append_call(p, nullptr, kI_new, k_new, v_new, kI, k, v, k_scale, v_scale, stream);
}

int dsa_cache_append_paged(const dsa_problem* p, const dsa_kv_pages* pages, const void* kI_new,
                           const void* k_new, const void* v_new, void* kI, void* k, void* v,
                           float* k_scale, float* v_scale, void* stream) {
  if (!pages) {
    reset_launches();
    return fail(DSA_ERR_INVALID_ARG, "pages is NULL");
  }
  return append_call(p, pages, kI_new, k_new, v_new, kI, k, v, k_scale, v_scale, stream);
}

int dsa_sparse_attn_decode_paged(const dsa_problem* p, const dsa_kv_pages* pages, const void* q,
                                 const void* qI, const float* w, const void* kI, const void* k,
                                 const void* v, const float* k_scale, const float* v_scale,
                                 int32_t* idx_out, void* out, void* ws, size_t ws_bytes,
                                 void* stream) {
  if (!pages) {
    reset_launches();
    return fail(DSA_ERR_INVALID_ARG, "pages is NULL");
  }
  return attn_entry(p, DSA_OP_DECODE, pages, q, qI, w, kI, k, v, k_scale, v_scale, idx_out, out,
                    ws, ws_bytes, stream);
}

int dsa_sparse_attn_prefill_paged(const dsa_problem* p, const dsa_kv_pages* pages, const void* q,
                                  const void* qI, const float* w, const void* kI, const void* k,
                                  const void* v, const float* k_scale, const float* v_scale,
                                  int32_t* idx_out, void* out, void* ws, size_t ws_bytes,
                                  void* stream) {
  if (!pages) {
    reset_launches();
    return fail(DSA_ERR_INVALID_ARG, "pages is NULL");
  }
  return attn_entry(p, DSA_OP_PREFILL, pages, q, qI, w, kI, k, v, k_scale, v_scale, idx_out, out,
                    ws, ws_bytes, stream);
}

int dsa_read_device_status(const void* ws, size_t ws_bytes, void* stream, uint32_t* status_out) {
  if (!ws || ws_bytes < 256 || !status_out)
    return fail(DSA_ERR_INVALID_ARG, "workspace or status_out invalid");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  uint32_t v = 0;
  e = cudaMemcpy(&v, ws, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  *status_out = v;
  if (v & kDevTimeout) return fail(DSA_ERR_TIMEOUT, "a kernel's bounded wait ran out");
  if (v & kDevBadPage)
    return fail(DSA_ERR_INVALID_ARG, "a gathered key's block-table entry lies outside the pool");
  if (v & kDevBounds)
    return fail(DSA_ERR_INVALID_ARG, "a debug bounds check failed (a row outside its array)");
  return DSA_OK;
}

const char* dsa_last_error_string(void) { return g_err.c_str(); }

int dsa_set_wait_budget(long long cycles) {
  g_wait_budget = cycles;
  return DSA_OK;
}

const char* dsa_status_string(int s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE";
    case DSA_ERR_MISALIGNED: return "DSA_ERR_MISALIGNED";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT";
    case DSA_ERR_NO_DEVICE: return "DSA_ERR_NO_DEVICE";
    default: return "unknown status";
  }
}

int dsa_version(void) { return 200; }

int dsa_last_launches(char* buf, size_t buflen) {
  if (buf && buflen > 0) {
    size_t o = 0;
    buf[0] = '\0';
    const int n = g_nlaunch < kLaunchLog ? g_nlaunch : kLaunchLog;
    for (int i = 0; i < n; ++i) {
      const int w = snprintf(buf + o, buflen - o, "%s%s", i ? "," : "", g_launch[i]);
      if (w < 0 || static_cast<size_t>(w) >= buflen - o) break;
      o += static_cast<size_t>(w);
    }
  }
  return g_nlaunch;
}

int dsa_timing_select(int kind) {
  if (kind < -1 || kind > DSA_KERNEL_APPEND) return fail(DSA_ERR_INVALID_ARG, "unknown kernel kind %d", kind);
  g_timing_kind = kind;
  g_ev_recorded = false;
  return DSA_OK;
}

int dsa_timing_read(float* ms) {
  if (!ms) return fail(DSA_ERR_INVALID_ARG, "ms is NULL");
  if (!g_ev_recorded || !g_ev[1]) return fail(DSA_ERR_INVALID_ARG, "no timed launch recorded");
  cudaError_t e = cudaEventSynchronize(g_ev[1]);
  if (e != cudaSuccess) return cuda_fail(e, "event synchronize");
  e = cudaEventElapsedTime(ms, g_ev[0], g_ev[1]);
  if (e != cudaSuccess) return cuda_fail(e, "event elapsed time");
  return DSA_OK;
}

}  // extern "C"
