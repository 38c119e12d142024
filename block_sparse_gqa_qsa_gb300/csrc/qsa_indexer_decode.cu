// qsa_indexer_decode.cu -- the QSA indexer for one new token per sequence over
// the paged KV pool ("Qsa Attention Plugin", step 3: B1 fused q-prep +
// predicated tail write / compress, B2 block scores from the kbar tails, B3
// deterministic top-512 + expand; "KV pool contract" for where the state lives).
//
// One launch.  A sequence's complete blocks are cut into chunks of
// `pagesPerChunk` pages; one CTA per (chunk, sequence):
//   B1  index-query prep at t = L-1 (fp32, f64 angles), redundantly per CTA;
//       chunk 0 stores the new raw key in token t's K-row tail when t leaves
//       its block incomplete; the CTA owning the page of a block that t
//       completes forms that block's key in f64 (from the K-row tails of its
//       first r-1 tokens and the new key), stores it in the V-row tail of the
//       block's first token and scores it from shared memory.
//   B2  streams the chunk's block keys: one 3-D TMA copy fetches the 128/r
//       key tails of a page (box {di, 128/r, 1} over a strided view of the
//       pool) into a 4-stage ring; each key is scored by di/8 lanes of a warp
//       (8 dims x 8 heads each), reduced with transposing warp shuffles.
//   B3  keeps the chunk's top-`budget` (key desc, id asc) as candidates; the
//       last CTA of each group of 8 (an atomic ticket, no waiting) merges the
//       group's candidates, up a tree, and the root writes the index list.
// Every wait on a TMA barrier is bounded; on expiry the CTA records
// kErrWaitTimeout in the workspace status word and stops.
#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr size_t kStatusBytes = 256;
constexpr int kThreads = 256;
constexpr int kStages = 4;
constexpr int kVPT = 16;         // selection elements per thread (4096 per CTA)
constexpr int kFanIn = 8;        // children merged per tree node
constexpr int kMaxChunkBlocks = kThreads * kVPT;
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;  // 0.2 s
constexpr int kMaxDynSmem = 227 * 1024;

struct DecIdxArgs {
  const __half* idxQ;
  const __half* idxK;
  const float* wq;
  const float* wk;
  __half* pool;
  const int32_t* pageTable;
  const int32_t* ctx;
  int32_t* indices;
  uint32_t* candKey;  // [B][slotsPerSeq][budget]
  int32_t* candId;    // [B][slotsPerSeq][budget]
  int32_t* candCnt;   // [B][slotsPerSeq]
  int32_t* counters;  // [B][countersPerSeq]
  int32_t* status;
  int Hkv, D, poolHeadDim, numFlatPages, maxPagesPerSeq, Hi, rot, ratio, budget, topK;
  int pagesPerChunk, chunksMax, slotsPerSeq, countersPerSeq;
  float eps;
  RopeFreqs rf;
};

__device__ __forceinline__ size_t pool_row(int page, int tok_in_page, int Hkv, int poolHeadDim) {
  return (static_cast<size_t>(page) * kTokensPerPage + tok_in_page) * Hkv * poolHeadDim;  // head 0
}

// Writes the selected (ascending-id) elements either as the candidates of a
// tree slot or, at the root, as the sequence's expanded index list.
template <int VPT>
__device__ __forceinline__ void emit(const DecIdxArgs& a, int b, const uint32_t (&key)[VPT],
                                     const int (&id)[VPT], const bool (&sel)[VPT], bool root, int slot,
                                     int n_c, int t, int* scan) {
  int ns = 0;
#pragma unroll
  for (int v = 0; v < VPT; ++v) ns += sel[v] ? 1 : 0;
  int tot;
  int pos = cta_exclusive_scan<kThreads>(ns, scan, tot);
  if (!root) {
    const size_t base = (static_cast<size_t>(b) * a.slotsPerSeq + slot) * a.budget;
#pragma unroll
    for (int v = 0; v < VPT; ++v)
      if (sel[v]) {
        a.candKey[base + pos] = key[v];
        a.candId[base + pos] = id[v];
        ++pos;
      }
    if (threadIdx.x == 0) a.candCnt[static_cast<size_t>(b) * a.slotsPerSeq + slot] = tot;
    return;
  }
  int32_t* out = a.indices + static_cast<size_t>(b) * a.topK;
#pragma unroll
  for (int v = 0; v < VPT; ++v)
    if (sel[v]) {
      for (int j = 0; j < a.ratio; ++j) out[pos * a.ratio + j] = id[v] * a.ratio + j;
      ++pos;
    }
  const int head = tot * a.ratio;
  for (int i = head + threadIdx.x; i < a.topK; i += kThreads) {
    const int j = n_c * a.ratio + (i - head);
    out[i] = j <= t ? j : -1;
  }
}

__host__ __device__ __forceinline__ int align_up(int x, int a) { return (x + a - 1) / a * a; }

// Shared-memory carve-up of the decode indexer (byte offsets), used by host and device.
struct DecSmem {
  int bars, q, sc, m, y, knew, red, total;
};
__host__ __device__ __forceinline__ DecSmem dec_smem_layout(int di, int ratio, int pagesPerChunk) {
  const int bpp = kTokensPerPage / ratio;
  DecSmem l;
  int off = kStages * bpp * di * 2;  // the TMA ring starts at offset 0
  l.bars = off = align_up(off, 16);
  off += kStages * 8;
  l.q = off = align_up(off, 16);
  off += 8 * di * 4;
  l.sc = off = align_up(off, 16);
  off += pagesPerChunk * bpp * 4;
  l.m = off = align_up(off, 16);
  off += di * 8;
  l.y = off;
  off += di * 8;
  l.knew = off = align_up(off, 16);
  off += di * 2;
  l.red = off = align_up(off, 16);
  off += 32 * 4;
  l.total = off;
  return l;
}

template <int DI>
__global__ void __launch_bounds__(kThreads) decode_indexer_kernel(const DecIdxArgs a,
                                                                  const __grid_constant__ CUtensorMap kmap) {
  constexpr int LPB = DI / 8;    // lanes per block key (8 dims each)
  constexpr int BPW = 32 / LPB;  // block keys per warp pass
  extern __shared__ __align__(1024) uint8_t smem[];
  const int bpp = kTokensPerPage / a.ratio;       // block keys per page
  const int stage_bytes = bpp * DI * 2;
  const DecSmem lay = dec_smem_layout(DI, a.ratio, a.pagesPerChunk);
  uint8_t* ring = smem;                                            // [kStages][bpp][DI] fp16
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);
  float* q_s = reinterpret_cast<float*>(smem + lay.q);             // [8][DI]
  float* sc_s = reinterpret_cast<float*>(smem + lay.sc);           // [pagesPerChunk * bpp]
  double* m_s = reinterpret_cast<double*>(smem + lay.m);           // [DI] f64 scratch
  double* y_s = reinterpret_cast<double*>(smem + lay.y);           // [DI]
  __half* knew_s = reinterpret_cast<__half*>(smem + lay.knew);     // [DI]
  int* red = reinterpret_cast<int*>(smem + lay.red);               // 16 + 8 + 8 ints
  int* scan = red + 16;
  int* misc = scan + 8;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, b = blockIdx.y;
  const int L = max(0, min(a.ctx[b], a.maxPagesPerSeq * kTokensPerPage));
  if (L == 0) {  // no token: empty list, no state change
    if (c == 0)
      for (int i = tid; i < a.topK; i += kThreads) a.indices[static_cast<size_t>(b) * a.topK + i] = -1;
    return;
  }
  const int t = L - 1;
  const int n_c = L / a.ratio;
  const bool completes = (L % a.ratio) == 0;
  const int npg = (n_c + bpp - 1) / bpp;  // pages holding complete blocks
  const int nch = max(1, (npg + a.pagesPerChunk - 1) / a.pagesPerChunk);
  if (c >= nch) return;
  const int p0 = c * a.pagesPerChunk, p1 = min(p0 + a.pagesPerChunk, npg);
  const int npages = max(0, p1 - p0);
  const int g0 = p0 * bpp;
  const int nloc = max(0, min(p1 * bpp, n_c) - g0);
  const int32_t* ptK = a.pageTable + static_cast<size_t>(b) * 2 * a.maxPagesPerSeq;
  const int32_t* ptV = ptK + a.maxPagesPerSeq;

  // ---- start the key stream early
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    for (int s = 0; s < kStages && s < npages; ++s) {
      int vp = __ldg(ptV + p0 + s);
      if (static_cast<unsigned>(vp) >= static_cast<unsigned>(a.numFlatPages)) {
        atomicOr(a.status, kErrBadPage);
        vp = 0;
      }
      mbar_arrive_expect_tx(&bars[s], stage_bytes);
      tma_load_3d(ring + s * stage_bytes, &kmap, 0, 0, vp, &bars[s]);
    }
  }

  // ---- B1: index-query prep at pos t (warp h -> head h)
  {
    constexpr int PER = DI / 32;
    const int h = warp;
    if (h < a.Hi) {
      const __half* x = a.idxQ + (static_cast<size_t>(b) * a.Hi + h) * DI;
      float y[PER];
      float ss = 0.f;
#pragma unroll
      for (int p = 0; p < PER; ++p) {
        y[p] = __half2float(x[lane + 32 * p]);
        ss = fmaf(y[p], y[p], ss);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
      const float inv = 1.0f / sqrtf(ss / DI + a.eps);
#pragma unroll
      for (int p = 0; p < PER; ++p) {
        const int i = lane + 32 * p;
        y[p] = y[p] * inv * (1.0f + a.wq[i]);
        q_s[h * DI + i] = y[p];
      }
      __syncwarp();
      const int half = a.rot >> 1;
      float v[PER];
#pragma unroll
      for (int p = 0; p < PER; ++p) {
        const int i = lane + 32 * p;
        v[p] = y[p];
        if (i < half) {
          float cs, sn;
          rope_cos_sin_f32(static_cast<double>(t), a.rf.inv_freq[i], cs, sn);
          v[p] = y[p] * cs - q_s[h * DI + i + half] * sn;
        } else if (i < a.rot) {
          const int k = i - half;
          float cs, sn;
          rope_cos_sin_f32(static_cast<double>(t), a.rf.inv_freq[k], cs, sn);
          v[p] = y[p] * cs + q_s[h * DI + k] * sn;
        }
      }
      __syncwarp();
#pragma unroll
      for (int p = 0; p < PER; ++p) q_s[h * DI + lane + 32 * p] = v[p];
    } else {
#pragma unroll
      for (int p = 0; p < PER; ++p) q_s[h * DI + lane + 32 * p] = 0.f;
    }
  }

  // ---- B1: predicated tail write / compress
  int g_new = -1;
  if (!completes) {
    if (c == 0 && tid < DI) {
      const int kp = __ldg(ptK + (t >> 7));
      if (static_cast<unsigned>(kp) < static_cast<unsigned>(a.numFlatPages))
        a.pool[pool_row(kp, t & 127, a.Hkv, a.poolHeadDim) + a.D + tid] = a.idxK[static_cast<size_t>(b) * DI + tid];
      else if (tid == 0)
        atomicOr(a.status, kErrBadPage);
    }
  } else {
    const int gn = n_c - 1;
    const int first = gn * a.ratio;  // block's first token; all r tokens share its page
    if ((first >> 7) / a.pagesPerChunk == c) {
      g_new = gn;
      if (warp == 0) {
        const int kp = __ldg(ptK + (first >> 7));
        const int vp = __ldg(ptV + (first >> 7));
        const bool okp = static_cast<unsigned>(kp) < static_cast<unsigned>(a.numFlatPages) &&
                         static_cast<unsigned>(vp) < static_cast<unsigned>(a.numFlatPages);
        if (!okp && lane == 0) atomicOr(a.status, kErrBadPage);
        for (int i = lane; i < DI; i += 32) {
          double acc = 0.0;
          for (int j = 0; j < a.ratio; ++j) {
            const int tok = first + j;
            const __half hv = (tok == t || !okp)
                                  ? a.idxK[static_cast<size_t>(b) * DI + i]
                                  : a.pool[pool_row(kp, tok & 127, a.Hkv, a.poolHeadDim) + a.D + i];
            acc = __dadd_rn(acc, static_cast<double>(__half2float(hv)));
          }
          m_s[i] = __ddiv_rn(acc, static_cast<double>(a.ratio));
        }
        __syncwarp();
        double inv = 0.0;
        if (lane == 0) {
          double ss = 0.0;
          for (int i = 0; i < DI; ++i) ss = __dadd_rn(ss, __dmul_rn(m_s[i], m_s[i]));
          inv = __ddiv_rn(1.0, __dsqrt_rn(__dadd_rn(__ddiv_rn(ss, static_cast<double>(DI)), static_cast<double>(a.eps))));
        }
        inv = __shfl_sync(kFull, inv, 0);
        for (int i = lane; i < DI; i += 32)
          y_s[i] = __dmul_rn(__dmul_rn(m_s[i], inv), __dadd_rn(1.0, static_cast<double>(a.wk[i])));
        __syncwarp();
        const int half = a.rot >> 1;
        const double pos = static_cast<double>(first);
        for (int i = lane; i < DI; i += 32) {
          double r = y_s[i];
          if (i < half) {
            double s, cc;
            sincos(__dmul_rn(pos, a.rf.inv_freq[i]), &s, &cc);
            r = __dsub_rn(__dmul_rn(y_s[i], cc), __dmul_rn(y_s[i + half], s));
          } else if (i < a.rot) {
            const int k = i - half;
            double s, cc;
            sincos(__dmul_rn(pos, a.rf.inv_freq[k]), &s, &cc);
            r = __dadd_rn(__dmul_rn(y_s[i], cc), __dmul_rn(y_s[k], s));
          }
          const __half hk = __double2half(r);
          knew_s[i] = hk;
          if (okp) a.pool[pool_row(vp, first & 127, a.Hkv, a.poolHeadDim) + a.D + i] = hk;
        }
      }
    }
  }
  __syncthreads();

  // ---- B2: stream and score the chunk's block keys
  const int sub = lane % LPB;
  float qr[8][8];
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    const float4 x0 = *reinterpret_cast<const float4*>(q_s + h * DI + sub * 8);
    const float4 x1 = *reinterpret_cast<const float4*>(q_s + h * DI + sub * 8 + 4);
    qr[h][0] = x0.x; qr[h][1] = x0.y; qr[h][2] = x0.z; qr[h][3] = x0.w;
    qr[h][4] = x1.x; qr[h][5] = x1.y; qr[h][6] = x1.z; qr[h][7] = x1.w;
  }
  bool alive = true;
  int failed_at = npages;
  for (int pi = 0; pi < npages; ++pi) {
    const int s = pi % kStages;
    const bool ok = mbar_wait_bounded(&bars[s], (pi / kStages) & 1, kWaitLimitNs);
    if (!__syncthreads_and(ok)) {
      alive = false;
      failed_at = pi;
      break;
    }
    const __half* tile = reinterpret_cast<const __half*>(ring + s * stage_bytes);
    for (int blk0 = warp * BPW; blk0 < bpp; blk0 += 8 * BPW) {
      const int blk = blk0 + lane / LPB;
      const int g = (p0 + pi) * bpp + blk;
      const bool valid = blk < bpp && g < n_c;
      const __half* src = g == g_new ? knew_s : tile + (valid ? blk : 0) * DI;
      const uint4 raw = *reinterpret_cast<const uint4*>(src + sub * 8);
      const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
      float kv[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(h2[i]);
        kv[2 * i] = f.x;
        kv[2 * i + 1] = f.y;
      }
      float d[8];
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        float acc = qr[h][0] * kv[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) acc = fmaf(qr[h][i], kv[i], acc);
        d[h] = acc;
      }
      // Transposing reduction over the LPB lanes of this key: after three
      // halvings each lane holds one head's partial; LPB = 16 needs one more
      // exchange to complete the sum.
      int n = 8;
#pragma unroll
      for (int o = LPB / 2; o >= LPB / 8; o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (i < n / 2) {
            const float send = upper ? d[i] : d[i + n / 2];
            const float keep = upper ? d[i + n / 2] : d[i];
            d[i] = keep + __shfl_xor_sync(kFull, send, o);
          }
        }
        n >>= 1;
      }
      float dot = d[0];
      if (LPB == 16) dot += __shfl_xor_sync(kFull, dot, 1);
      float sc = dot > 0.f ? dot : 0.f;
#pragma unroll
      for (int o = LPB / 8; o < LPB; o <<= 1) sc += __shfl_xor_sync(kFull, sc, o);
      if (valid && sub == 0) sc_s[pi * bpp + blk] = sc;
    }
    __syncthreads();  // stage s fully read
    if (tid == 0 && pi + kStages < npages) {
      int vp = __ldg(ptV + p0 + pi + kStages);
      if (static_cast<unsigned>(vp) >= static_cast<unsigned>(a.numFlatPages)) {
        atomicOr(a.status, kErrBadPage);
        vp = 0;
      }
      fence_proxy_async();
      mbar_arrive_expect_tx(&bars[s], stage_bytes);
      tma_load_3d(ring + s * stage_bytes, &kmap, 0, 0, vp, &bars[s]);
    }
  }
  if (!alive) {
    // Pages failed_at .. failed_at + kStages - 1 may still be in flight: let
    // each land (bounded) before the CTA exits.
    if (tid == 0) {
      atomicOr(a.status, kErrWaitTimeout);
      const int issued = min(npages, failed_at + kStages);
      for (int pi = failed_at; pi < issued; ++pi)
        mbar_wait_bounded(&bars[pi % kStages], (pi / kStages) & 1, kWaitLimitNs);
    }
    return;
  }

  // ---- B3: chunk top-k, then the merge tree
  uint32_t key[kVPT];
  int id[kVPT];
  bool sel[kVPT];
  {
    const int base = tid * kVPT;
    const int nv = max(0, min(kVPT, nloc - base));
#pragma unroll
    for (int v = 0; v < kVPT; ++v) {
      key[v] = v < nv ? __float_as_uint(sc_s[base + v]) : 0u;
      id[v] = g0 + base + v;
      sel[v] = v < nv;
    }
    if (nloc > a.budget) cta_topk<kThreads, kVPT>(key, nv, a.budget, sel, red, scan);
  }
  int cnt = nch, lvl_off = 0, lvl_n = a.chunksMax, node = c;
  bool root = cnt == 1;
  emit<kVPT>(a, b, key, id, sel, root, lvl_off + node, n_c, t, scan);
  while (!root) {
    const int parent = node / kFanIn;
    const int nsib = min(kFanIn, cnt - parent * kFanIn);
    const int next_off = lvl_off + lvl_n;
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      int32_t* ctr = a.counters + static_cast<size_t>(b) * a.countersPerSeq + (next_off - a.chunksMax) + parent;
      const bool last = atomicAdd(ctr, 1) == nsib - 1;
      if (last) *ctr = 0;  // re-armed for the next call
      misc[0] = last;
    }
    __syncthreads();
    if (!misc[0]) return;
    __threadfence();
    // Children's candidates, concatenated in child order (ascending ids).
    const size_t slot0 = static_cast<size_t>(b) * a.slotsPerSeq + lvl_off + parent * kFanIn;
    int offs[kFanIn + 1];
    offs[0] = 0;
#pragma unroll
    for (int k = 0; k < kFanIn; ++k) offs[k + 1] = offs[k] + (k < nsib ? __ldcg(a.candCnt + slot0 + k) : 0);
    const int total = offs[kFanIn];
    const int base = tid * kVPT;
    const int nv = max(0, min(kVPT, total - base));
#pragma unroll
    for (int v = 0; v < kVPT; ++v) {
      const int e = base + v;
      key[v] = 0u;
      id[v] = 0;
      sel[v] = v < nv;
      if (v < nv) {
        int k = 0;
        while (e >= offs[k + 1]) ++k;
        const size_t at = (slot0 + k) * a.budget + (e - offs[k]);
        key[v] = __ldcg(a.candKey + at);
        id[v] = __ldcg(a.candId + at);
      }
    }
    if (total > a.budget) cta_topk<kThreads, kVPT>(key, nv, a.budget, sel, red, scan);
    node = parent;
    cnt = (cnt + kFanIn - 1) / kFanIn;
    lvl_off = next_off;
    lvl_n = (lvl_n + kFanIn - 1) / kFanIn;
    root = cnt == 1;
    emit<kVPT>(a, b, key, id, sel, root, lvl_off + node, n_c, t, scan);
  }
}

size_t decode_smem_bytes(int di, int ratio, int pagesPerChunk) {
  return static_cast<size_t>(dec_smem_layout(di, ratio, pagesPerChunk).total);
}

}  // namespace

DecodePlan plan_indexer_decode(int B, int maxPagesPerSeq, int ratio) {
  DecodePlan pl;
  const int bpp = kTokensPerPage / ratio;
  const long long total_pages = static_cast<long long>(B) * maxPagesPerSeq;
  const int target_ctas = 640;  // ~4 resident CTAs on each of the 152 SMs
  long long cp = (total_pages + target_ctas - 1) / target_ctas;
  cp = cp < 1 ? 1 : cp;
  const int cap = kMaxChunkBlocks / bpp;  // chunk scores must fit one selection pass
  pl.pagesPerChunk = static_cast<int>(cp > cap ? cap : cp);
  pl.chunksMax = (maxPagesPerSeq + pl.pagesPerChunk - 1) / pl.pagesPerChunk;
  pl.levels = 0;
  pl.slotsPerSeq = pl.chunksMax;
  for (int n = pl.chunksMax; n > 1;) {
    n = (n + kFanIn - 1) / kFanIn;
    pl.slotsPerSeq += n;
    ++pl.levels;
  }
  pl.countersPerSeq = pl.slotsPerSeq - pl.chunksMax;
  return pl;
}

size_t indexer_decode_workspace_bytes(int B, int maxPagesPerSeq, int ratio, int budget) {
  const DecodePlan pl = plan_indexer_decode(B, maxPagesPerSeq, ratio);
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t slots = static_cast<size_t>(B) * pl.slotsPerSeq;
  return kStatusBytes + up(slots * budget * 4) * 2 + up(slots * 4) + up(static_cast<size_t>(B) * pl.countersPerSeq * 4);
}

cudaError_t launch_indexer_decode(const QsaIndexerDecodeParams& p, const RopeFreqs& rf,
                                  const CUtensorMap& kbarMap) {
  const DecodePlan pl = plan_indexer_decode(p.batchSize, p.maxPagesPerSeq, p.compressRatio);
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t slots = static_cast<size_t>(p.batchSize) * pl.slotsPerSeq;
  uint8_t* ws = static_cast<uint8_t*>(p.workspace);
  DecIdxArgs a;
  a.status = reinterpret_cast<int32_t*>(ws);
  a.candKey = reinterpret_cast<uint32_t*>(ws + kStatusBytes);
  a.candId = reinterpret_cast<int32_t*>(ws + kStatusBytes + up(slots * p.budget * 4));
  a.candCnt = reinterpret_cast<int32_t*>(ws + kStatusBytes + 2 * up(slots * p.budget * 4));
  a.counters = reinterpret_cast<int32_t*>(ws + kStatusBytes + 2 * up(slots * p.budget * 4) + up(slots * 4));
  a.idxQ = static_cast<const __half*>(p.idxQ);
  a.idxK = static_cast<const __half*>(p.idxK);
  a.wq = p.qNormW;
  a.wk = p.kNormW;
  a.pool = static_cast<__half*>(p.kvPool);
  a.pageTable = p.pageTable;
  a.ctx = p.contextLengths;
  a.indices = p.indices;
  a.Hkv = p.numKVHeads;
  a.D = p.kvHeadDim;
  a.poolHeadDim = p.poolHeadDim;
  a.numFlatPages = p.numFlatPages;
  a.maxPagesPerSeq = p.maxPagesPerSeq;
  a.Hi = p.numHeads;
  a.rot = p.rotDim;
  a.ratio = p.compressRatio;
  a.budget = p.budget;
  a.topK = p.topK;
  a.pagesPerChunk = pl.pagesPerChunk;
  a.chunksMax = pl.chunksMax;
  a.slotsPerSeq = pl.slotsPerSeq;
  a.countersPerSeq = pl.countersPerSeq;
  a.eps = p.rmsNormEps;
  a.rf = rf;
  const size_t smem = decode_smem_bytes(p.headDim, p.compressRatio, pl.pagesPerChunk);
  if (smem > static_cast<size_t>(kMaxDynSmem)) return cudaErrorInvalidValue;
  dim3 grid(pl.chunksMax, p.batchSize);
  cudaStream_t st = static_cast<cudaStream_t>(p.stream);
  if (p.headDim == 64) {
    static const cudaError_t attr = cudaFuncSetAttribute(
        decode_indexer_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
    if (attr != cudaSuccess) return attr;
    decode_indexer_kernel<64><<<grid, kThreads, smem, st>>>(a, kbarMap);
  } else {
    static const cudaError_t attr = cudaFuncSetAttribute(
        decode_indexer_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
    if (attr != cudaSuccess) return attr;
    decode_indexer_kernel<128><<<grid, kThreads, smem, st>>>(a, kbarMap);
  }
  return cudaGetLastError();
}

}  // namespace qsa
