// qsa_noalloc.cu -- qsa_sparse_decode_noalloc: split-K sparse decode attention
// whose fp32 partials and split counters live in a fixed scratch array owned
// by this library, so that the caller hands over no workspace at all.
//
// The scratch is one file-scope __device__ array per GPU: the driver places it
// when this module is loaded into a context, and nothing here calls an
// allocator.  The first call in a context looks up the array's device address
// and clears the counter region on the caller's stream; later calls in the
// same context reuse that address.  The cache is keyed on the context's
// unique id, so a call after cudaDeviceReset (a new primary context, where the
// module and its array are loaded afresh) or from another context on the same
// GPU looks the address up and clears the counters again.  The kernels are
// the ones qsa_sparse_decode launches: this entry point fills the three
// workspace fields of a copy of the params and calls it.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "qsa_internal.h"

namespace {

// Capacity: 256 (sequence, KV head) pairs at headDim 128.  The regions sit at
// fixed offsets, so every call finds its counters at the same place, and all
// counters are zero between calls (each combine resets the one it used).
constexpr int kScratchPairs = 256;
constexpr int kScratchD = 128;
constexpr size_t kCounterBytes = 1024;                                                // int32 [256]
constexpr size_t kStatsBytes = static_cast<size_t>(kScratchPairs) * 8 * 2 * 16 * 4;   // fp32 [256*8, 2, 16]
constexpr size_t kPartialOBytes = static_cast<size_t>(kScratchPairs) * 8 * 16 * kScratchD * 4;  // fp32 [256*8, 16, 128]
constexpr size_t kScratchBytes = kCounterBytes + kStatsBytes + kPartialOBytes;          // 16.25 MiB
static_assert(kScratchPairs * 4 <= static_cast<int>(kCounterBytes), "counter region");
static_assert(kCounterBytes % 256 == 0 && kStatsBytes % 256 == 0, "regions stay 256-byte aligned");

__device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
struct ContextScratch {
  unsigned long long ctx_id;  // 0: not set up yet (driver context ids start at 1)
  unsigned char* base;
};
ContextScratch g_scratch[kMaxDevices];

qsa_status_t failf(qsa_status_t s, const char* fmt, ...) {
  char buf[320];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  return qsa::record_error(s, buf);
}

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <class Fn>
Fn driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(p);
}

// Unique id of the calling thread's current context, or 0 when there is none yet.
unsigned long long current_context_id() {
  static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch in the current context; looked up (and its
// counters cleared on `stream`) by the first call made in that context.
qsa_status_t scratch_for_current_context(cudaStream_t stream, unsigned char** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return failf(QSA_ERR_CUDA, "qsa_sparse_decode_noalloc: cudaGetDevice failed (%s)", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return failf(QSA_ERR_UNSUPPORTED, "qsa_sparse_decode_noalloc: device ordinal %d >= %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  const unsigned long long id = current_context_id();
  if (id != 0 && g_scratch[dev].ctx_id == id) {
    *out = g_scratch[dev].base;
    return QSA_OK;
  }
  void* addr = nullptr;
  e = cudaGetSymbolAddress(&addr, g_decode_scratch);  // also makes the device's primary context current
  if (e != cudaSuccess || !addr)
    return failf(QSA_ERR_CUDA, "qsa_sparse_decode_noalloc: looking up the scratch on device %d failed (%s)", dev,
                 cudaGetErrorString(e));
  e = cudaMemsetAsync(addr, 0, kCounterBytes, stream);
  if (e != cudaSuccess)
    return failf(QSA_ERR_CUDA, "qsa_sparse_decode_noalloc: clearing the split counters on device %d failed (%s)",
                 dev, cudaGetErrorString(e));
  g_scratch[dev].ctx_id = current_context_id();  // 0 (driver entry points unavailable): look up on every call
  g_scratch[dev].base = static_cast<unsigned char*>(addr);
  *out = g_scratch[dev].base;
  return QSA_OK;
}

}  // namespace

extern "C" {

qsa_status_t qsa_sparse_decode_noalloc(const QsaSparseDecodeParams* p) {
  if (!p) return qsa::record_error(QSA_ERR_INVALID_ARG, "qsa_sparse_decode_noalloc: params is NULL");
  if (p->partialO || p->partialStats || p->splitCounters)
    return qsa::record_error(QSA_ERR_INVALID_ARG,
                             "qsa_sparse_decode_noalloc: partialO, partialStats and splitCounters must be NULL "
                             "(this entry point uses its own scratch)");
  const long long pairs = static_cast<long long>(p->batchSize) * p->numKVHeads;
  if (p->batchSize >= 1 && p->numKVHeads >= 1 && pairs > kScratchPairs)
    return failf(QSA_ERR_UNSUPPORTED,
                 "qsa_sparse_decode_noalloc: batchSize * numKVHeads = %lld exceeds the %lld (sequence, KV head) "
                 "pairs its fixed scratch holds; call qsa_sparse_decode with a workspace instead",
                 pairs, static_cast<long long>(kScratchPairs));
  if (p->headDim > kScratchD)
    return failf(QSA_ERR_UNSUPPORTED, "qsa_sparse_decode_noalloc: headDim %d > %d", p->headDim, kScratchD);
  unsigned char* base = nullptr;
  const qsa_status_t s = scratch_for_current_context(static_cast<cudaStream_t>(p->stream), &base);
  if (s != QSA_OK) return s;
  QsaSparseDecodeParams q = *p;
  q.splitCounters = reinterpret_cast<int32_t*>(base);
  q.partialStats = reinterpret_cast<float*>(base + kCounterBytes);
  q.partialO = reinterpret_cast<float*>(base + kCounterBytes + kStatsBytes);
  return qsa_sparse_decode(&q);
}

}  // extern "C"
