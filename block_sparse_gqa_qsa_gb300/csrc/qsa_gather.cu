// qsa_gather.cu -- gather-to-scratch form of the split-K decode (qsa.rs,
// "qsa_gather" and the scratch-as-paged-cache note): the K and V rows of the
// tokens a decode list names are copied out of the paged pool into contiguous
// scratch, and the scratch is described as a paged pool of its own (page
// table, identity list, lengths), so that the unchanged split-K decode
// consumes it.  It is the A/B counterpart of the decode kernel's in-kernel
// page-table gathers.
//
// Slot n of a sequence's scratch holds list entry n; an entry that names no
// token (negative, or >= contextLengths[b], or on a page outside the pool)
// leaves its slot unwritten and is -1 in the scratch list.  The scratch list
// keeps every entry at its list position, so each decode split sees the same
// keys in the same order as on the pool and the two outputs agree bit for bit.
//
// One warp per list entry, eight per CTA: the warp loads the entry's K row
// and V row (numKVHeads x headDim halves each, 16 bytes per lane per copy)
// into registers, then stores both into the entry's scratch slot.
#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr int kGatherWarps = 8;
constexpr int kGatherMaxChunks = 4;  // 16-byte chunks per lane per row: numKVHeads * headDim <= 32 * 8 * 4

struct GatherArgs {
  const __half* pool;
  const int32_t* pageTable;
  const int32_t* indices;
  const int32_t* ctx;
  __half* scratch;
  int32_t* spt;
  int32_t* sidx;
  int32_t* slen;
  int B, Hkv, D, poolHeadDim, numFlatPages, maxPagesPerSeq, topK, P;
};

__global__ void __launch_bounds__(kGatherWarps * 32) gather_kernel(const GatherArgs a) {
  const int lane = threadIdx.x & 31;
  const long long e = static_cast<long long>(blockIdx.x) * kGatherWarps + (threadIdx.x >> 5);
  if (e >= static_cast<long long>(a.B) * a.topK) return;
  const int b = static_cast<int>(e / a.topK), n = static_cast<int>(e % a.topK);
  if (lane == 0) {
    if ((n & (kTokensPerPageHost - 1)) == 0) {  // scratch page n / 128 of sequence b: K pages, then V pages
      const int p = n / kTokensPerPageHost;
      a.spt[(static_cast<size_t>(b) * 2) * a.P + p] = b * a.P + p;
      a.spt[(static_cast<size_t>(b) * 2 + 1) * a.P + p] = (a.B + b) * a.P + p;
    }
    if (n == 0) a.slen[b] = a.topK;
  }
  const int L = max(0, min(a.ctx[b], a.maxPagesPerSeq * kTokensPerPageHost));
  const int j = __ldg(a.indices + e);
  bool ok = static_cast<unsigned>(j) < static_cast<unsigned>(L);
  int kp = 0, vp = 0;
  if (ok) {
    const int32_t* pt = a.pageTable + static_cast<size_t>(b) * 2 * a.maxPagesPerSeq;
    kp = __ldg(pt + (j >> 7));
    vp = __ldg(pt + a.maxPagesPerSeq + (j >> 7));
    ok = static_cast<unsigned>(kp) < static_cast<unsigned>(a.numFlatPages) &&
         static_cast<unsigned>(vp) < static_cast<unsigned>(a.numFlatPages);
  }
  if (lane == 0) a.sidx[e] = ok ? n : -1;
  if (!ok) return;  // warp-uniform
  const int cpr = a.D / 8, nch = a.Hkv * cpr;  // 16-byte chunks per head and per row
  const __half* krow = a.pool + (static_cast<size_t>(kp) * kTokensPerPageHost + (j & 127)) * a.Hkv * a.poolHeadDim;
  const __half* vrow = a.pool + (static_cast<size_t>(vp) * kTokensPerPageHost + (j & 127)) * a.Hkv * a.poolHeadDim;
  uint4 kv[2][kGatherMaxChunks];
#pragma unroll
  for (int u = 0; u < kGatherMaxChunks; ++u) {
    const int c = lane + 32 * u;
    if (c < nch) {
      const int off = (c / cpr) * a.poolHeadDim + (c % cpr) * 8;
      kv[0][u] = __ldg(reinterpret_cast<const uint4*>(krow + off));
      kv[1][u] = __ldg(reinterpret_cast<const uint4*>(vrow + off));
    }
  }
  const size_t rowElems = static_cast<size_t>(a.Hkv) * a.D;
  uint4* kdst = reinterpret_cast<uint4*>(a.scratch + (static_cast<size_t>(b) * a.P * kTokensPerPageHost + n) * rowElems);
  uint4* vdst = reinterpret_cast<uint4*>(a.scratch +
                                         (static_cast<size_t>(a.B + b) * a.P * kTokensPerPageHost + n) * rowElems);
#pragma unroll
  for (int u = 0; u < kGatherMaxChunks; ++u) {
    const int c = lane + 32 * u;
    if (c < nch) {
      kdst[c] = kv[0][u];
      vdst[c] = kv[1][u];
    }
  }
}

}  // namespace

int gather_scratch_pages(int topK) { return (topK + kTokensPerPageHost - 1) / kTokensPerPageHost; }

int gather_max_row_chunks() { return 32 * kGatherMaxChunks; }

cudaError_t launch_gather(const QsaGatherParams& p) {
  GatherArgs a;
  a.pool = static_cast<const __half*>(p.kvPool);
  a.pageTable = p.pageTable;
  a.indices = p.indices;
  a.ctx = p.contextLengths;
  a.scratch = static_cast<__half*>(p.scratch);
  a.spt = p.scratchPageTable;
  a.sidx = p.scratchIndices;
  a.slen = p.scratchLengths;
  a.B = p.batchSize;
  a.Hkv = p.numKVHeads;
  a.D = p.headDim;
  a.poolHeadDim = p.poolHeadDim;
  a.numFlatPages = p.numFlatPages;
  a.maxPagesPerSeq = p.maxPagesPerSeq;
  a.topK = p.topK;
  a.P = gather_scratch_pages(p.topK);
  const long long entries = static_cast<long long>(p.batchSize) * p.topK;
  const unsigned grid = static_cast<unsigned>((entries + kGatherWarps - 1) / kGatherWarps);
  gather_kernel<<<grid, kGatherWarps * 32, 0, static_cast<cudaStream_t>(p.stream)>>>(a);
  return cudaGetLastError();
}

}  // namespace qsa
