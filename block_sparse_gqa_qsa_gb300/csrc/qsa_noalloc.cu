// qsa_noalloc.cu -- qsa_sparse_decode_noalloc: split-K sparse decode attention
// whose fp32 partials and split counters live in a fixed scratch array owned
// by this library, so that the caller hands over no workspace at all.
//
// The scratch is one file-scope __device__ array per GPU: the driver places it
// when this module is loaded, and nothing here calls an allocator.  The first
// call on a device looks up the array's device address once and clears the
// counter region on the caller's stream; later calls reuse that address.  The
// kernels are the ones qsa_sparse_decode launches: this entry point fills the
// three workspace fields of a copy of the params and calls it.
#include <atomic>
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
std::atomic<unsigned char*> g_scratch_ptr[kMaxDevices];

qsa_status_t failf(qsa_status_t s, const char* fmt, ...) {
  char buf[320];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  return qsa::record_error(s, buf);
}

// Device address of this GPU's scratch; looked up (and its counters cleared on
// `stream`) by the first call that runs with that GPU current.
qsa_status_t scratch_for_current_device(cudaStream_t stream, unsigned char** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return failf(QSA_ERR_CUDA, "qsa_sparse_decode_noalloc: cudaGetDevice failed (%s)", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return failf(QSA_ERR_UNSUPPORTED, "qsa_sparse_decode_noalloc: device ordinal %d >= %d", dev, kMaxDevices);
  unsigned char* base = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (base) {
    *out = base;
    return QSA_OK;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  base = g_scratch_ptr[dev].load(std::memory_order_relaxed);
  if (!base) {
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_decode_scratch);
    if (e != cudaSuccess || !addr)
      return failf(QSA_ERR_CUDA, "qsa_sparse_decode_noalloc: looking up the scratch on device %d failed (%s)", dev,
                   cudaGetErrorString(e));
    e = cudaMemsetAsync(addr, 0, kCounterBytes, stream);
    if (e != cudaSuccess)
      return failf(QSA_ERR_CUDA, "qsa_sparse_decode_noalloc: clearing the split counters on device %d failed (%s)",
                   dev, cudaGetErrorString(e));
    base = static_cast<unsigned char*>(addr);
    g_scratch_ptr[dev].store(base, std::memory_order_release);
  }
  *out = base;
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
  const qsa_status_t s = scratch_for_current_device(static_cast<cudaStream_t>(p->stream), &base);
  if (s != QSA_OK) return s;
  QsaSparseDecodeParams q = *p;
  q.splitCounters = reinterpret_cast<int32_t*>(base);
  q.partialStats = reinterpret_cast<float*>(base + kCounterBytes);
  q.partialO = reinterpret_cast<float*>(base + kCounterBytes + kStatsBytes);
  return qsa_sparse_decode(&q);
}

}  // extern "C"
