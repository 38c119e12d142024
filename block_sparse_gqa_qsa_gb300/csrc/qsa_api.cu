// qsa_api.cu -- the C ABI of libqsa.so (declared in include/qsa.h): host-side
// validation, workspace arithmetic, RoPE frequency tables, the TMA tensor map
// of the decode indexer, and the kernel launches.  Nothing here allocates or
// synchronises; a failed check returns before anything is enqueued.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "qsa_internal.h"

namespace {

thread_local std::string g_last_error;

qsa_status_t fail(qsa_status_t s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

qsa_status_t ok() {
  g_last_error.clear();
  return QSA_OK;
}

qsa_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(QSA_ERR_CUDA, "%s: CUDA error %d (%s)", what, static_cast<int>(e), cudaGetErrorString(e));
}

}  // namespace

qsa_status_t qsa::record_error(qsa_status_t s, const char* msg) { return fail(s, "%s", msg); }

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

qsa::RopeFreqs rope_freqs(float theta, int rot) {
  qsa::RopeFreqs r;
  std::memset(&r, 0, sizeof(r));
  for (int i = 0; i < rot / 2; ++i) {
    r.inv_freq[i] = std::pow(static_cast<double>(theta), -2.0 * i / rot);
    double x = r.inv_freq[i] / 6.283185307179586;
    x -= std::floor(x);
    r.turn[i] = static_cast<unsigned long long>(std::ldexp(x, 64));  // x < 1, so this stays below 2^64
  }
  const double pi = 3.14159265358979323846;
  for (int j = 0; j <= 32; ++j) {  // cos(pi j / 64); past pi / 4 as sin of the complement, so j = 32 is exactly 0
    const double c = j <= 16 ? std::cos(pi * j / 64.0) : std::sin(pi * (32 - j) / 64.0);
    r.qcos_hi[j] = static_cast<float>(c);
    r.qcos_lo[j] = static_cast<float>(c - static_cast<double>(r.qcos_hi[j]));
  }
  return r;
}

constexpr int kMaxAttnListWidth = 16384;  // attention stages one list (or slice) in shared memory

// Indexer arguments shared by both indexers ("Qsa Attention Plugin" constructor
// attributes: indexerNumHeads, indexerHeadDim, indexerBudget, indexerCompressRatio).
qsa_status_t check_indexer_shape(int Hi, int di, int rot, int ratio, int budget, int topK, float theta,
                                 float eps) {
  if (Hi < 1 || di < 1 || rot < 0 || rot > di || (rot & 1) || ratio < 1 || budget < 1 || !(theta > 0.f) ||
      !(eps >= 0.f))
    return fail(QSA_ERR_INVALID_ARG, "indexer: invalid numHeads/headDim/rotDim/compressRatio/budget/theta/eps");
  if (static_cast<long long>(topK) < static_cast<long long>(budget) * ratio + ratio - 1)
    return fail(QSA_ERR_INVALID_ARG, "indexer: topK %d < budget*ratio + ratio - 1 = %lld", topK,
                static_cast<long long>(budget) * ratio + ratio - 1);
  if (Hi > 8) return fail(QSA_ERR_UNSUPPORTED, "indexer: numHeads %d > 8", Hi);
  if (di != 64 && di != 128) return fail(QSA_ERR_UNSUPPORTED, "indexer: headDim %d not 64 or 128", di);
  if (rot > 128) return fail(QSA_ERR_UNSUPPORTED, "indexer: rotDim %d > 128", rot);
  return QSA_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

}  // namespace

namespace {

// The attention entry points share their checks; fn names the caller in messages.
qsa_status_t sparse_prefill_entry(const QsaSparsePrefillParams* p, const char* fn, bool bf16, bool tcgen05 = false) {
  if (!p) return fail(QSA_ERR_INVALID_ARG, "%s: params is NULL", fn);
  if (!p->qPtr || !p->kPtr || !p->vPtr || !p->oPtr || !p->indices || !p->contextLengths)
    return fail(QSA_ERR_INVALID_ARG, "%s: a tensor pointer is NULL", fn);
  if (p->batchSize < 1 || p->seqLen < 1 || p->numQHeads < 1 || p->numKVHeads < 1 || p->headDim < 1 || p->topK < 1)
    return fail(QSA_ERR_INVALID_ARG, "%s: sizes must be >= 1", fn);
  if (p->numQHeads % p->numKVHeads)
    return fail(QSA_ERR_INVALID_ARG, "%s: numQHeads %% numKVHeads != 0", fn);
  if (!qsa_sparse_prefill_can_implement(p->numQHeads, p->numKVHeads, p->headDim))
    return fail(QSA_ERR_UNSUPPORTED, "%s: needs headDim 128 and a GQA group of at most 16", fn);
  if (p->topK > kMaxAttnListWidth)
    return fail(QSA_ERR_UNSUPPORTED, "%s: topK > %d", fn, kMaxAttnListWidth);
  if (static_cast<long long>(p->batchSize) * p->seqLen * p->numKVHeads > 0x7fffffffLL)
    return fail(QSA_ERR_UNSUPPORTED, "%s: batchSize*seqLen*numKVHeads exceeds the grid", fn);
  if (!aligned(p->qPtr, 16) || !aligned(p->kPtr, 16) || !aligned(p->vPtr, 16) || !aligned(p->oPtr, 16))
    return fail(QSA_ERR_INVALID_ARG, "%s: Q/K/V/O must be 16-byte aligned", fn);
  const cudaError_t e = tcgen05 ? qsa::launch_sparse_prefill_tc(*p, bf16) : qsa::launch_sparse_prefill(*p, bf16);
  return e == cudaSuccess ? ok() : cuda_fail(e, fn);
}


qsa_status_t sparse_decode_entry(const QsaSparseDecodeParams* p, const char* fn, bool bf16) {
  if (!p) return fail(QSA_ERR_INVALID_ARG, "%s: params is NULL", fn);
  if (!p->qPtr || !p->kvPoolPtr || !p->pageTable || !p->indices || !p->contextLengths || !p->oPtr)
    return fail(QSA_ERR_INVALID_ARG, "%s: a tensor pointer is NULL", fn);
  if (!p->partialO || !p->partialStats || !p->splitCounters)
    return fail(QSA_ERR_WORKSPACE, "%s: partialO/partialStats/splitCounters is NULL", fn);
  if (p->batchSize < 1 || p->numQHeads < 1 || p->numKVHeads < 1 || p->headDim < 1 || p->topK < 1 ||
      p->numFlatPages < 1 || p->maxPagesPerSeq < 1)
    return fail(QSA_ERR_INVALID_ARG, "%s: sizes must be >= 1", fn);
  if (p->numQHeads % p->numKVHeads)
    return fail(QSA_ERR_INVALID_ARG, "%s: numQHeads %% numKVHeads != 0", fn);
  if (p->poolHeadDim < p->headDim) return fail(QSA_ERR_INVALID_ARG, "%s: poolHeadDim < headDim", fn);
  if (!qsa_sparse_decode_can_implement(p->numQHeads, p->numKVHeads, p->headDim, p->poolHeadDim))
    return fail(QSA_ERR_UNSUPPORTED,
                "%s: needs headDim 128, a GQA group of at most 16, poolHeadDim a multiple of 8", fn);
  if (p->topK > kMaxAttnListWidth) return fail(QSA_ERR_UNSUPPORTED, "%s: topK > %d", fn, kMaxAttnListWidth);
  if (p->batchSize > 65535 || p->numKVHeads > 65535)
    return fail(QSA_ERR_UNSUPPORTED, "%s: batchSize/numKVHeads > 65535", fn);
  if (static_cast<long long>(p->maxPagesPerSeq) * 128 > 0x7fffffffLL)
    return fail(QSA_ERR_UNSUPPORTED, "%s: maxPagesPerSeq too large", fn);
  if (!aligned(p->qPtr, 16) || !aligned(p->kvPoolPtr, 16) || !aligned(p->oPtr, 16) || !aligned(p->partialO, 16) ||
      !aligned(p->partialStats, 4) || !aligned(p->splitCounters, 4))
    return fail(QSA_ERR_INVALID_ARG, "%s: q/pool/o/partialO must be 16-byte aligned", fn);
  const cudaError_t e = qsa::launch_sparse_decode(*p, bf16);
  return e == cudaSuccess ? ok() : cuda_fail(e, fn);
}

}  // namespace

extern "C" {

const char* qsa_status_string(qsa_status_t s) {
  switch (s) {
    case QSA_OK: return "QSA_OK";
    case QSA_ERR_INVALID_ARG: return "QSA_ERR_INVALID_ARG";
    case QSA_ERR_UNSUPPORTED: return "QSA_ERR_UNSUPPORTED";
    case QSA_ERR_WORKSPACE: return "QSA_ERR_WORKSPACE";
    case QSA_ERR_CUDA: return "QSA_ERR_CUDA";
  }
  return "QSA_ERR_UNKNOWN";
}

const char* qsa_last_error_message(void) { return g_last_error.c_str(); }

qsa_status_t qsa_last_device_error(const void* workspace, void* stream, int32_t* out) {
  if (!workspace || !out) return fail(QSA_ERR_INVALID_ARG, "qsa_last_device_error: workspace or out is NULL");
  const cudaError_t e = cudaMemcpyAsync(out, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost,
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "qsa_last_device_error");
}

void qsa_debug_set_wait_limit_ns(uint64_t ns) { qsa::set_decode_wait_limit_ns(ns); }

int32_t qsa_indexer_prefill_max_blocks(void) { return qsa::kPrefillMaxSeqLen; }
int32_t qsa_indexer_prefill_max_seq_len(void) { return qsa::kPrefillMaxSeqLen; }

size_t qsa_indexer_prefill_workspace_size(int32_t B, int32_t S, int32_t di, int32_t ratio) {
  if (B < 1 || S < 1 || di < 1 || ratio < 1) return 0;
  return qsa::indexer_prefill_workspace_bytes(B, S, di, ratio);
}

size_t qsa_indexer_decode_workspace_size(int32_t B, int32_t maxPagesPerSeq, int32_t ratio, int32_t budget) {
  if (B < 1 || maxPagesPerSeq < 1 || ratio < 1 || qsa::kTokensPerPageHost % ratio != 0 || budget < 1) return 0;
  return qsa::indexer_decode_workspace_bytes(B, maxPagesPerSeq, ratio, budget);
}

size_t qsa_sparse_decode_partial_o_elems(int32_t B, int32_t Hkv, int32_t D) {
  if (B < 1 || Hkv < 1 || D < 1) return 0;
  return static_cast<size_t>(B) * Hkv * 8 * 16 * D;
}
size_t qsa_sparse_decode_partial_stats_elems(int32_t B, int32_t Hkv) {
  if (B < 1 || Hkv < 1) return 0;
  return static_cast<size_t>(B) * Hkv * 8 * 2 * 16;
}
size_t qsa_sparse_decode_counter_elems(int32_t B, int32_t Hkv) {
  if (B < 1 || Hkv < 1) return 0;
  return static_cast<size_t>(B) * Hkv;
}
int32_t qsa_sparse_decode_max_splits(void) { return 8; }
int32_t qsa_sparse_decode_partial_rows(void) { return 16; }

int32_t qsa_sparse_prefill_can_implement(int32_t Hq, int32_t Hkv, int32_t D) {
  return Hq >= 1 && Hkv >= 1 && Hq % Hkv == 0 && Hq / Hkv <= 16 && D == 128;
}
int32_t qsa_sparse_decode_can_implement(int32_t Hq, int32_t Hkv, int32_t D, int32_t poolHeadDim) {
  return qsa_sparse_prefill_can_implement(Hq, Hkv, D) && poolHeadDim >= D && poolHeadDim % 8 == 0;
}

qsa_status_t qsa_indexer_prefill(const QsaIndexerPrefillParams* p) {
  if (!p) return fail(QSA_ERR_INVALID_ARG, "qsa_indexer_prefill: params is NULL");
  if (!p->idxQ || !p->idxK || !p->qNormW || !p->kNormW || !p->contextLengths || !p->indices)
    return fail(QSA_ERR_INVALID_ARG, "qsa_indexer_prefill: a tensor pointer is NULL");
  if (p->batchSize < 1 || p->seqLen < 1)
    return fail(QSA_ERR_INVALID_ARG, "qsa_indexer_prefill: batchSize/seqLen must be >= 1");
  qsa_status_t s = check_indexer_shape(p->numHeads, p->headDim, p->rotDim, p->compressRatio, p->budget, p->topK,
                                       p->ropeTheta, p->rmsNormEps);
  if (s != QSA_OK) return s;
  if (p->batchSize > 65535) return fail(QSA_ERR_UNSUPPORTED, "qsa_indexer_prefill: batchSize > 65535");
  if (p->seqLen > qsa::kPrefillMaxSeqLen)
    return fail(QSA_ERR_UNSUPPORTED, "qsa_indexer_prefill: seqLen %d > %d", p->seqLen, qsa::kPrefillMaxSeqLen);
  if (static_cast<long long>(p->batchSize) * p->seqLen > 0x7fffffffLL)
    return fail(QSA_ERR_UNSUPPORTED, "qsa_indexer_prefill: batchSize*seqLen exceeds 2^31 - 1 rows");
  const size_t need = qsa::indexer_prefill_workspace_bytes(p->batchSize, p->seqLen, p->headDim, p->compressRatio);
  if (!p->workspace || p->workspaceBytes < need || !aligned(p->workspace, 256))
    return fail(QSA_ERR_WORKSPACE, "qsa_indexer_prefill: workspace needs %zu bytes, 256-byte aligned", need);
  const cudaError_t e = qsa::launch_indexer_prefill(*p, rope_freqs(p->ropeTheta, p->rotDim));
  return e == cudaSuccess ? ok() : cuda_fail(e, "qsa_indexer_prefill");
}

qsa_status_t qsa_indexer_decode(const QsaIndexerDecodeParams* p) {
  if (!p) return fail(QSA_ERR_INVALID_ARG, "qsa_indexer_decode: params is NULL");
  if (!p->idxQ || !p->idxK || !p->qNormW || !p->kNormW || !p->kvPool || !p->pageTable || !p->contextLengths ||
      !p->indices)
    return fail(QSA_ERR_INVALID_ARG, "qsa_indexer_decode: a tensor pointer is NULL");
  if (p->batchSize < 1 || p->numKVHeads < 1 || p->kvHeadDim < 1 || p->numFlatPages < 1 || p->maxPagesPerSeq < 1)
    return fail(QSA_ERR_INVALID_ARG, "qsa_indexer_decode: batchSize/numKVHeads/kvHeadDim/numFlatPages/"
                                     "maxPagesPerSeq must be >= 1");
  if (p->poolHeadDim < p->kvHeadDim + p->headDim)
    return fail(QSA_ERR_INVALID_ARG, "qsa_indexer_decode: poolHeadDim %d < kvHeadDim + headDim", p->poolHeadDim);
  qsa_status_t s = check_indexer_shape(p->numHeads, p->headDim, p->rotDim, p->compressRatio, p->budget, p->topK,
                                       p->ropeTheta, p->rmsNormEps);
  if (s != QSA_OK) return s;
  if (qsa::kTokensPerPageHost % p->compressRatio != 0)
    return fail(QSA_ERR_INVALID_ARG, "qsa_indexer_decode: compressRatio %d does not divide the 128-token page",
                p->compressRatio);
  if (p->compressRatio < 4 || p->compressRatio > 16)
    return fail(QSA_ERR_UNSUPPORTED, "qsa_indexer_decode: compressRatio %d outside 4..16 (a page's key tails are "
                                     "one swizzled TMA tile of 8..32 rows)", p->compressRatio);
  if (p->budget > 4096)
    return fail(QSA_ERR_UNSUPPORTED, "qsa_indexer_decode: budget %d > 4096", p->budget);
  if (p->batchSize > qsa::kDecodeMaxBatch)
    return fail(QSA_ERR_UNSUPPORTED, "qsa_indexer_decode: batchSize > %d", qsa::kDecodeMaxBatch);
  if (p->kvHeadDim % 8 || p->poolHeadDim % 8 || !aligned(p->kvPool, 16))
    return fail(QSA_ERR_UNSUPPORTED, "qsa_indexer_decode: kvHeadDim and poolHeadDim must be multiples of 8 and "
                                     "kvPool 16-byte aligned (TMA rows)");
  if (static_cast<long long>(p->maxPagesPerSeq) * 128 > 0x7fffffffLL)
    return fail(QSA_ERR_UNSUPPORTED, "qsa_indexer_decode: maxPagesPerSeq too large");
  if (static_cast<long long>(p->maxPagesPerSeq) * (qsa::kTokensPerPageHost / p->compressRatio) > (1LL << 21))
    return fail(QSA_ERR_UNSUPPORTED, "qsa_indexer_decode: more than 2097152 blocks per sequence");
  const size_t need = qsa::indexer_decode_workspace_bytes(p->batchSize, p->maxPagesPerSeq, p->compressRatio, p->budget);
  if (!p->workspace || p->workspaceBytes < need || !aligned(p->workspace, 256))
    return fail(QSA_ERR_WORKSPACE, "qsa_indexer_decode: workspace needs %zu bytes, 256-byte aligned", need);
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return fail(QSA_ERR_CUDA, "qsa_indexer_decode: cuTensorMapEncodeTiled is unavailable");
  // Strided view of the key tails: [numFlatPages][128/r block-start rows][headDim] starting at column kvHeadDim
  // of head 0 ("KV pool contract": block g's key in the V-row tail of token r*g).
  const int bpp = qsa::kTokensPerPageHost / p->compressRatio;
  const size_t row_bytes = static_cast<size_t>(p->numKVHeads) * p->poolHeadDim * 2;
  CUtensorMap map;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(p->headDim), static_cast<cuuint64_t>(bpp),
                        static_cast<cuuint64_t>(p->numFlatPages)};
  cuuint64_t strides[2] = {row_bytes * p->compressRatio, row_bytes * qsa::kTokensPerPageHost};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(bpp), 1};  // one 128-byte swizzled half per copy
  cuuint32_t estr[3] = {1, 1, 1};
  void* base = static_cast<char*>(p->kvPool) + static_cast<size_t>(p->kvHeadDim) * 2;
  const CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(QSA_ERR_UNSUPPORTED, "qsa_indexer_decode: tensor map rejected (CUresult %d)", r);
  const cudaError_t e = qsa::launch_indexer_decode(*p, rope_freqs(p->ropeTheta, p->rotDim), map);
  return e == cudaSuccess ? ok() : cuda_fail(e, "qsa_indexer_decode");
}

qsa_status_t qsa_sparse_prefill(const QsaSparsePrefillParams* p) {
  return sparse_prefill_entry(p, "qsa_sparse_prefill", false);
}
qsa_status_t qsa_sparse_prefill_bf16(const QsaSparsePrefillParams* p) {
  return sparse_prefill_entry(p, "qsa_sparse_prefill_bf16", true);
}
qsa_status_t qsa_sparse_prefill_tcgen05(const QsaSparsePrefillParams* p) {
  return sparse_prefill_entry(p, "qsa_sparse_prefill_tcgen05", false, true);
}
qsa_status_t qsa_sparse_prefill_tcgen05_bf16(const QsaSparsePrefillParams* p) {
  return sparse_prefill_entry(p, "qsa_sparse_prefill_tcgen05_bf16", true, true);
}

qsa_status_t qsa_rope_qkv(const QsaRopeQkvParams* p) {
  if (!p) return fail(QSA_ERR_INVALID_ARG, "qsa_rope_qkv: params is NULL");
  if (!p->qkv || !p->qNormW || !p->kNormW || !p->contextLengths || !p->qOut)
    return fail(QSA_ERR_INVALID_ARG, "qsa_rope_qkv: a required pointer is NULL");
  if (p->batchSize < 1 || p->seqLen < 1 || p->numQHeads < 1 || p->numKVHeads < 1)
    return fail(QSA_ERR_INVALID_ARG, "qsa_rope_qkv: sizes must be >= 1");
  if (p->headDim != 64 && p->headDim != 128)
    return fail(QSA_ERR_UNSUPPORTED, "qsa_rope_qkv: headDim %d not 64 or 128", p->headDim);
  if (p->rotDim < 0 || p->rotDim > p->headDim || (p->rotDim & 1) || !(p->ropeTheta > 0.f) || !(p->rmsNormEps >= 0.f))
    return fail(QSA_ERR_INVALID_ARG, "qsa_rope_qkv: rotDim must be even and <= headDim; theta > 0, eps >= 0");
  if (static_cast<long long>(p->numQHeads + 2LL * p->numKVHeads) * p->headDim * 2 > qsa::kRopeMaxRowBytes)
    return fail(QSA_ERR_UNSUPPORTED, "qsa_rope_qkv: (numQHeads + 2 numKVHeads) * headDim * 2 exceeds %d bytes",
                qsa::kRopeMaxRowBytes);
  if (p->rotDim % 16)
    return fail(QSA_ERR_UNSUPPORTED, "qsa_rope_qkv: rotDim %d is not a multiple of 16 (rotation partners are "
                                     "exchanged as whole 8-element chunks)", p->rotDim);
  if (!aligned(p->qkv, 16) || !aligned(p->qOut, 16) || !aligned(p->kOut, 16) || !aligned(p->vOut, 16) ||
      !aligned(p->kvPool, 16))
    return fail(QSA_ERR_UNSUPPORTED, "qsa_rope_qkv: qkv, qOut, kOut, vOut and kvPool must be 16-byte aligned");
  if (static_cast<long long>(p->batchSize) * p->seqLen > 0x7fffffffLL)
    return fail(QSA_ERR_UNSUPPORTED, "qsa_rope_qkv: batchSize*seqLen exceeds the grid");
  if (p->kvPool) {
    if (!p->pageTable || p->poolHeadDim < p->headDim || p->numFlatPages < 1 || p->maxPagesPerSeq < 1)
      return fail(QSA_ERR_INVALID_ARG, "qsa_rope_qkv: kvPool needs pageTable, poolHeadDim >= headDim and page counts");
    if (p->poolHeadDim % 8)
      return fail(QSA_ERR_UNSUPPORTED, "qsa_rope_qkv: poolHeadDim %d is not a multiple of 8 (16-byte row writes)",
                  p->poolHeadDim);
    if (static_cast<long long>(p->maxPagesPerSeq) * qsa::kTokensPerPageHost > 0x7fffffffLL)
      return fail(QSA_ERR_UNSUPPORTED, "qsa_rope_qkv: maxPagesPerSeq too large");
  }
  const cudaError_t e = qsa::launch_rope_qkv(*p, rope_freqs(p->ropeTheta, p->rotDim));
  return e == cudaSuccess ? ok() : cuda_fail(e, "qsa_rope_qkv");
}

qsa_status_t qsa_indexer_prefill_handoff(const QsaIndexerHandoffParams* p) {
  if (!p) return fail(QSA_ERR_INVALID_ARG, "qsa_indexer_prefill_handoff: params is NULL");
  if (!p->idxK || !p->contextLengths || !p->workspace || !p->kvPool || !p->pageTable)
    return fail(QSA_ERR_INVALID_ARG, "qsa_indexer_prefill_handoff: a pointer is NULL");
  if (p->batchSize < 1 || p->seqLen < 1 || p->compressRatio < 1 || p->numKVHeads < 1 || p->kvHeadDim < 1 ||
      p->numFlatPages < 1 || p->maxPagesPerSeq < 1)
    return fail(QSA_ERR_INVALID_ARG, "qsa_indexer_prefill_handoff: sizes must be >= 1");
  if (p->headDim != 64 && p->headDim != 128)
    return fail(QSA_ERR_UNSUPPORTED, "qsa_indexer_prefill_handoff: headDim %d not 64 or 128", p->headDim);
  if (p->poolHeadDim < p->kvHeadDim + p->headDim)
    return fail(QSA_ERR_INVALID_ARG, "qsa_indexer_prefill_handoff: poolHeadDim %d < kvHeadDim + headDim",
                p->poolHeadDim);
  if (p->kvHeadDim % 8 || p->poolHeadDim % 8 || !aligned(p->kvPool, 16) || !aligned(p->idxK, 16))
    return fail(QSA_ERR_UNSUPPORTED, "qsa_indexer_prefill_handoff: kvHeadDim and poolHeadDim must be multiples of 8 "
                                     "and idxK / kvPool 16-byte aligned (16-byte copies)");
  if (static_cast<long long>(p->maxPagesPerSeq) * qsa::kTokensPerPageHost < p->seqLen ||
      static_cast<long long>(p->maxPagesPerSeq) * qsa::kTokensPerPageHost > 0x7fffffffLL)
    return fail(QSA_ERR_INVALID_ARG, "qsa_indexer_prefill_handoff: maxPagesPerSeq must cover seqLen");
  const size_t need = qsa::indexer_prefill_workspace_bytes(p->batchSize, p->seqLen, p->headDim, p->compressRatio);
  if (p->workspaceBytes < need || !aligned(p->workspace, 256))
    return fail(QSA_ERR_WORKSPACE, "qsa_indexer_prefill_handoff: the prefill workspace has %zu bytes, 256-byte "
                                   "aligned, for this shape", need);
  const cudaError_t e = qsa::launch_indexer_handoff(*p);
  return e == cudaSuccess ? ok() : cuda_fail(e, "qsa_indexer_prefill_handoff");
}

int32_t qsa_gather_scratch_pages(int32_t topK) { return topK < 1 ? 0 : qsa::gather_scratch_pages(topK); }

size_t qsa_gather_scratch_elems(int32_t B, int32_t Hkv, int32_t D, int32_t topK) {
  if (B < 1 || Hkv < 1 || D < 1 || topK < 1) return 0;
  return 2 * static_cast<size_t>(B) * qsa::gather_scratch_pages(topK) * qsa::kTokensPerPageHost * Hkv * D;
}

qsa_status_t qsa_gather_selected(const QsaGatherParams* p) {
  if (!p) return fail(QSA_ERR_INVALID_ARG, "qsa_gather_selected: params is NULL");
  if (!p->kvPool || !p->pageTable || !p->indices || !p->contextLengths || !p->scratch || !p->scratchPageTable ||
      !p->scratchIndices || !p->scratchLengths)
    return fail(QSA_ERR_INVALID_ARG, "qsa_gather_selected: a pointer is NULL");
  if (p->batchSize < 1 || p->numKVHeads < 1 || p->headDim < 1 || p->poolHeadDim < 1 || p->numFlatPages < 1 ||
      p->maxPagesPerSeq < 1 || p->topK < 1)
    return fail(QSA_ERR_INVALID_ARG, "qsa_gather_selected: sizes must be >= 1");
  if (p->poolHeadDim < p->headDim) return fail(QSA_ERR_INVALID_ARG, "qsa_gather_selected: poolHeadDim < headDim");
  if (p->headDim % 8 || p->poolHeadDim % 8 || p->numKVHeads * (p->headDim / 8) > qsa::gather_max_row_chunks())
    return fail(QSA_ERR_UNSUPPORTED, "qsa_gather_selected: headDim and poolHeadDim must be multiples of 8 and "
                                     "numKVHeads * headDim at most %d", qsa::gather_max_row_chunks() * 8);
  if (!aligned(p->kvPool, 16) || !aligned(p->scratch, 16))
    return fail(QSA_ERR_UNSUPPORTED, "qsa_gather_selected: kvPool and scratch must be 16-byte aligned");
  if (static_cast<long long>(p->maxPagesPerSeq) * qsa::kTokensPerPageHost > 0x7fffffffLL ||
      static_cast<long long>(p->batchSize) * p->topK > 0x7fffffffLL)
    return fail(QSA_ERR_UNSUPPORTED, "qsa_gather_selected: maxPagesPerSeq or batchSize * topK too large");
  const cudaError_t e = qsa::launch_gather(*p);
  return e == cudaSuccess ? ok() : cuda_fail(e, "qsa_gather_selected");
}

qsa_status_t qsa_sparse_decode(const QsaSparseDecodeParams* p) {
  return sparse_decode_entry(p, "qsa_sparse_decode", false);
}
qsa_status_t qsa_sparse_decode_bf16(const QsaSparseDecodeParams* p) {
  return sparse_decode_entry(p, "qsa_sparse_decode_bf16", true);
}

}  // extern "C"
