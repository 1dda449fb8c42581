// dsa_topk_noalloc: the exact top-k of dsa_topk with its scratch in a static
// device array inside libdsa instead of a caller-provided workspace.
//
// Some callers cannot hand the library device memory: an operator plugin whose
// host framework passes only input and output tensors, a serving engine that
// reserves its whole memory budget at start-up and forbids allocation while
// requests run, or a latency-critical path that cannot afford cudaMalloc's
// implicit device synchronisation. For them this entry point keeps its radix
// histograms, tickets, candidate list and selection bitmaps in
// `g_topk_scratch` below (about 8.2 MiB), which every GPU that loads the
// library holds until the process exits. The call itself allocates nothing.
#include <cstdio>
#include <mutex>

#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kNaRows = DSA_TOPK_NOALLOC_MAX_ROWS;
constexpr int kNaLen = DSA_TOPK_NOALLOC_MAX_LEN;
constexpr size_t kNaHist = 0;                                                  // rows x 2048 u32
constexpr size_t kNaTicket = kNaHist + static_cast<size_t>(kNaRows) * kHistBins * 4;
constexpr size_t kNaCount = kNaTicket + 256;
constexpr size_t kNaZeroEnd = kNaCount + 256;                                  // cleared per call
constexpr size_t kNaBitmap = kNaZeroEnd;                                       // rows x len/32 u32
constexpr size_t kNaCands = kNaBitmap + static_cast<size_t>(kNaRows) * (kNaLen / 32) * 4;
constexpr size_t kNaBytes = kNaCands + static_cast<size_t>(kNaRows) * kNaLen * 8;

// The scratch. In host code this name is only a host-side stand-in; kernels get
// its device address from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_topk_scratch[kNaBytes];

std::mutex g_na_mu;
// Device address of g_topk_scratch per device ordinal, with the CUDA context
// it was looked up in: a new context on that device (after a device reset the
// module is loaded again and the array may move) looks it up again.
uint8_t* g_na_ptr[64] = {};
void* g_na_ctx[64] = {};

using CtxGetCurrentFn = int (*)(void**);   // cuCtxGetCurrent(CUcontext*)
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(f);
  });
  return fn;
}

}  // namespace

int noalloc_fail(int status, const char* msg);   // sets dsa_last_error_string()
int noalloc_check_topk(const dsa_problem* p, int* rows, int* max_n);

}  // namespace dsa

using namespace dsa;

extern "C" int dsa_topk_noalloc(const dsa_problem* p, const float* scores, int32_t* idx,
                                void* stream) {
  int rows = 0, max_n = 0;
  int rc = noalloc_check_topk(p, &rows, &max_n);
  if (rc) return rc;
  if (rows > kNaRows || max_n > kNaLen) {
    char buf[200];
    snprintf(buf, sizeof(buf),
             "dsa_topk_noalloc handles at most %d query rows of at most %d visible keys "
             "(got %d rows, longest %d); use dsa_topk with a workspace",
             kNaRows, kNaLen, rows, max_n);
    return noalloc_fail(DSA_ERR_UNSUPPORTED, buf);
  }
  if (!scores || !idx) return noalloc_fail(DSA_ERR_INVALID_ARG, "a tensor pointer is NULL");
  if ((reinterpret_cast<uintptr_t>(scores) & 3) || (reinterpret_cast<uintptr_t>(idx) & 3))
    return noalloc_fail(DSA_ERR_MISALIGNED, "scores and idx must be 4-byte aligned");

  // once per device and context, with that device current: the array's
  // device address (the first call on a device does this set-up, so make it
  // before capturing calls in a CUDA graph)
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return noalloc_fail(DSA_ERR_NO_DEVICE, "no CUDA device is current");
  CtxGetCurrentFn ctx_fn = ctx_get_current();
  void* ctx = nullptr;
  if (ctx_fn) ctx_fn(&ctx);
  uint8_t* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_na_mu);
    if (!g_na_ptr[dev] || ctx == nullptr || g_na_ctx[dev] != ctx) {
      void* ptr = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&ptr, g_topk_scratch);
      if (e != cudaSuccess || !ptr) {
        char buf[200];
        snprintf(buf, sizeof(buf), "cudaGetSymbolAddress(top-k scratch) failed: %s",
                 cudaGetErrorString(e));
        return noalloc_fail(DSA_ERR_CUDA, buf);
      }
      g_na_ptr[dev] = static_cast<uint8_t*>(ptr);
      // the lookup made the device's context current if none was
      if (ctx_fn) ctx_fn(&ctx);
      g_na_ctx[dev] = ctx;
    }
    base = g_na_ptr[dev];
  }

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // histograms, tickets and candidate counters start at zero on every call
  cudaError_t e = cudaMemsetAsync(base, 0, kNaZeroEnd, st);
  if (e != cudaSuccess) return noalloc_fail(DSA_ERR_CUDA, "clearing the top-k scratch failed");

  TopkParams tp{};
  tp.scores = scores;
  tp.idx = idx;
  tp.hist = reinterpret_cast<uint32_t*>(base + kNaHist);
  tp.ticket = reinterpret_cast<uint32_t*>(base + kNaTicket);
  tp.cand_count = reinterpret_cast<uint32_t*>(base + kNaCount);
  tp.cands = reinterpret_cast<unsigned long long*>(base + kNaCands);
  tp.bitmap = reinterpret_cast<uint32_t*>(base + kNaBitmap);
  tp.cand_stride = kNaLen;
  tp.bitmap_stride = kNaLen / 32;
  tp.B = p->batch;
  tp.S = p->q_len;
  tp.cap = p->cache_capacity;
  tp.k = p->top_k;
  tp.nchunks = (max_n + kChunk - 1) / kChunk;
  tp.row0 = 0;
  tp.nrows = rows;
  for (int b = 0; b < DSA_MAX_BATCH; ++b) tp.lens.T[b] = b < p->batch ? p->total_len[b] : 0;
  e = launch_topk_hist(tp, st);
  if (e == cudaSuccess) e = launch_topk_chunk_select(tp, st);
  if (e != cudaSuccess) return noalloc_fail(DSA_ERR_CUDA, cudaGetErrorString(e));
  return DSA_OK;
}
