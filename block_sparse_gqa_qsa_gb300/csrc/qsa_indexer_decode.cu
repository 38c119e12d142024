// qsa_indexer_decode.cu -- the QSA indexer for one new token per sequence over
// the paged KV pool ("Qsa Attention Plugin", step 3: B1 fused q-prep +
// predicated tail write / compress, B2 block scores from the kbar tails, B3
// deterministic top-512 + expand; "KV pool contract" for where the state lives).
//
// Three launches on the caller's stream:
//   decode_prep_kernel    (B1) one CTA per sequence: index-query prep at
//       t = L-1 (fp32, f64 angles) into the workspace; then the state update:
//       the new raw key into token t's K-row tail when t leaves its block
//       incomplete, else the block t completes is pooled in f64 (from the
//       K-row tails of its first r-1 tokens and the new key) and its key is
//       stored in the V-row tail of the block's first token.
//   decode_score_kernel   (B2) persistent, one CTA per SM, warp-specialised:
//       a producer warp streams the key tails of every page that holds
//       complete blocks (3-D TMA copies, box {64, 128/r, 1} with the 128-byte
//       swizzle over a strided view of the pool, page ids fetched 32 at a time)
//       into a 24-stage ring; 15 consumer warps score one page each: 16 lanes
//       per key, 8 dims x 8 heads per lane (dims paired in fp32x2 FMAs), then
//       a transposing shuffle reduction whose head order is pre-permuted per
//       lane (h ^ m) so that every step is one add of one shuffle; they write
//       the scores and add them to a 4096-bin histogram of the score bits per
//       sequence.  Pages are split evenly over the CTAs.
//   decode_select_kernel  (B3) per sequence: the histogram gives the bin that
//       holds the budget-th largest score; CTAs over 2048-block slices collect
//       the blocks above that bin and the blocks inside it (gathered in shared
//       memory, one global reservation per CTA); the last CTA to finish keeps
//       the top of the tie bin by (score desc, id asc), sorts the kept ids
//       (bitonic, in shared memory), expands them with the causal tail, and
//       re-arms the histogram and counters.
// Waits on TMA barriers are bounded; on expiry the kernel records
// kErrWaitTimeout in the workspace status word and stops.
#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr size_t kStatusBytes = 256;
constexpr int kNumBins = 4096;       // histogram of (score bits >> 19): exponent + 4 mantissa bits
constexpr int kBinShift = 19;
constexpr int kSliceBlocks = 2048;   // blocks one select CTA filters (8 per thread, one round of loads)
constexpr int kMaxSelect = 4096;     // budget cap: the final CTA sorts the kept block ids in shared memory
constexpr int kConsumerWarps = 15;  // + 1 producer warp = 16 warps, up to 128 registers each
constexpr int kScoreThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 24;
constexpr int kSelThreads = 256;
constexpr int kTieVPT = 16;          // tie candidates per thread held in registers
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;  // 0.2 s
constexpr int kMaxDynSmem = 227 * 1024;

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

struct WsLayout {
  size_t q, scores, hist, sureId, tieKey, tieId, counters, total;
};
WsLayout ws_layout(int B, int nbmax, int budget) {
  WsLayout l;
  size_t off = kStatusBytes;
  l.q = off;
  off += up256(static_cast<size_t>(B) * 8 * 128 * 4);  // prepared queries fp32 [B][8][128]
  l.scores = off;
  off += up256(static_cast<size_t>(B) * nbmax * 4);     // block scores fp32 [B][nbmax]
  l.hist = off;
  off += up256(static_cast<size_t>(B) * kNumBins * 4);  // int32 [B][kNumBins], zero between calls
  l.sureId = off;
  off += up256(static_cast<size_t>(B) * budget * 4);    // blocks above the threshold bin [B][budget]
  l.tieKey = off;
  off += up256(static_cast<size_t>(B) * nbmax * 4);     // blocks inside it [B][nbmax]
  l.tieId = off;
  off += up256(static_cast<size_t>(B) * nbmax * 4);
  l.counters = off;
  off += up256(static_cast<size_t>(B) * 3 * 4);         // sure count, tie count, ticket: zero between calls
  l.total = off;
  return l;
}

__device__ __forceinline__ size_t pool_row(int page, int tok_in_page, int Hkv, int poolHeadDim) {
  return (static_cast<size_t>(page) * kTokensPerPage + tok_in_page) * Hkv * poolHeadDim;  // head 0
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_addr(bar)) : "memory");
}

// ------------------------------------------------------------------ B1
struct PrepArgs {
  const __half* idxQ;
  const __half* idxK;
  const float* wq;
  const float* wk;
  __half* pool;
  const int32_t* pageTable;
  const int32_t* ctx;
  float* q;
  int32_t* status;
  int Hi, Hkv, D, poolHeadDim, numFlatPages, maxPagesPerSeq, rot, ratio;
  float eps;
  RopeFreqs rf;
};

template <int DI>
__global__ void __launch_bounds__(256) decode_prep_kernel(const PrepArgs a) {
  constexpr int PER = DI / 32;
  __shared__ float y_s[8][DI];
  __shared__ double m_s[DI];
  __shared__ double y2_s[DI];
  __shared__ double part_s[8];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x;
  const int L = max(0, min(a.ctx[b], a.maxPagesPerSeq * kTokensPerPage));
  if (L == 0) return;
  const int t = L - 1;
  const int n_c = L / a.ratio;
  const bool completes = (L % a.ratio) == 0;
  const int32_t* ptK = a.pageTable + static_cast<size_t>(b) * 2 * a.maxPagesPerSeq;
  const int32_t* ptV = ptK + a.maxPagesPerSeq;

  // index-query prep: warp h -> head h (heads >= Hi are zero)
  {
    const int h = warp;
    float* qo = a.q + (static_cast<size_t>(b) * 8 + h) * 128;
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
        y_s[h][i] = y[p];
      }
      __syncwarp();
      const int half = a.rot >> 1;
#pragma unroll
      for (int p = 0; p < PER; ++p) {
        const int i = lane + 32 * p;
        float v = y[p];
        if (i < half) {
          float cs, sn;
          rope_cos_sin_f32(static_cast<double>(t), a.rf.inv_freq[i], cs, sn);
          v = y[p] * cs - y_s[h][i + half] * sn;
        } else if (i < a.rot) {
          const int k = i - half;
          float cs, sn;
          rope_cos_sin_f32(static_cast<double>(t), a.rf.inv_freq[k], cs, sn);
          v = y[p] * cs + y_s[h][k] * sn;
        }
        qo[i] = v;
      }
    } else {
#pragma unroll
      for (int p = 0; p < PER; ++p) qo[lane + 32 * p] = 0.f;
    }
  }

  // state update
  if (!completes) {
    if (tid < DI) {
      const int kp = __ldg(ptK + (t >> 7));
      if (static_cast<unsigned>(kp) < static_cast<unsigned>(a.numFlatPages))
        a.pool[pool_row(kp, t & 127, a.Hkv, a.poolHeadDim) + a.D + tid] = a.idxK[static_cast<size_t>(b) * DI + tid];
      else if (tid == 0)
        atomicOr(a.status, kErrBadPage);
    }
    return;
  }
  const int first = (n_c - 1) * a.ratio;  // all r tokens of the block share this page
  const int kp = __ldg(ptK + (first >> 7)), vp = __ldg(ptV + (first >> 7));
  const bool okp = static_cast<unsigned>(kp) < static_cast<unsigned>(a.numFlatPages) &&
                   static_cast<unsigned>(vp) < static_cast<unsigned>(a.numFlatPages);
  if (!okp) {
    if (tid == 0) atomicOr(a.status, kErrBadPage);
    return;
  }
  double sq = 0.0;
  if (tid < DI) {
    double acc = 0.0;
    for (int j = 0; j < a.ratio; ++j) {
      const int tok = first + j;
      const __half hv = tok == t ? a.idxK[static_cast<size_t>(b) * DI + tid]
                                 : a.pool[pool_row(kp, tok & 127, a.Hkv, a.poolHeadDim) + a.D + tid];
      acc = __dadd_rn(acc, static_cast<double>(__half2float(hv)));
    }
    const double m = __ddiv_rn(acc, static_cast<double>(a.ratio));
    m_s[tid] = m;
    sq = __dmul_rn(m, m);
  }
  if (warp < DI / 32) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq = __dadd_rn(sq, __shfl_xor_sync(kFull, sq, o));
    if (lane == 0) part_s[warp] = sq;
  }
  __syncthreads();
  if (tid < DI) {
    double ss = 0.0;
    for (int w = 0; w < DI / 32; ++w) ss = __dadd_rn(ss, part_s[w]);
    const double inv = __ddiv_rn(1.0, __dsqrt_rn(__dadd_rn(__ddiv_rn(ss, static_cast<double>(DI)),
                                                           static_cast<double>(a.eps))));
    y2_s[tid] = __dmul_rn(__dmul_rn(m_s[tid], inv), __dadd_rn(1.0, static_cast<double>(a.wk[tid])));
  }
  __syncthreads();
  if (tid < DI) {
    const int i = tid, half = a.rot >> 1;
    const double pos = static_cast<double>(first);
    double r = y2_s[i];
    if (i < half) {
      double s, c;
      rope_cos_sin_f64(pos, a.rf.inv_freq[i], c, s);
      r = __dsub_rn(__dmul_rn(y2_s[i], c), __dmul_rn(y2_s[i + half], s));
    } else if (i < a.rot) {
      const int k = i - half;
      double s, c;
      rope_cos_sin_f64(pos, a.rf.inv_freq[k], c, s);
      r = __dadd_rn(__dmul_rn(y2_s[i], c), __dmul_rn(y2_s[k], s));
    }
    a.pool[pool_row(vp, first & 127, a.Hkv, a.poolHeadDim) + a.D + i] = __double2half(r);
  }
}

// ------------------------------------------------------------------ B2
struct ScoreArgs {
  const int32_t* ctx;
  const int32_t* pageTable;
  const float* q;
  float* scores;
  int32_t* hist;
  int32_t* status;
  int B, maxPagesPerSeq, numFlatPages, ratio, nbmax;
};

__host__ __device__ __forceinline__ int score_smem_bytes(int di, int ratio, int B) {
  const int stage = (kTokensPerPage / ratio) * di * 2;
  return kStages * stage + 2 * kStages * 8 + ((B + 1 + 3) / 4) * 16 + kConsumerWarps * 128 * 4;
}

// One lane per key row: byte offset of 16-byte chunk c (dims 8c..8c+7 of a
// 64-dim half) of row r in a TMA tile written with the 128-byte swizzle.
__device__ __forceinline__ int swz128(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

// Writes one page's scores (lane j = block j of the page) and adds them to the
// sequence's histogram, one atomic per distinct bin of the warp.
__device__ __forceinline__ void page_epilogue(const ScoreArgs& a, int b, int p, int n_c, int bpp, float sc) {
  const int lane = threadIdx.x & 31;
  const int g = p * bpp + lane;
  const bool valid = lane < bpp && g < n_c;
  const int bin = static_cast<int>(__float_as_uint(sc) >> kBinShift);
  if (valid) a.scores[static_cast<size_t>(b) * a.nbmax + g] = sc;
  const unsigned act = __ballot_sync(kFull, valid);
  if (valid) {
    const unsigned peers = __match_any_sync(act, bin);
    if (lane == __ffs(peers) - 1) atomicAdd(a.hist + static_cast<size_t>(b) * kNumBins + bin, __popc(peers));
  }
}

template <int DI>
__global__ void __launch_bounds__(kScoreThreads, 1) decode_score_kernel(const ScoreArgs a,
                                                                        const __grid_constant__ CUtensorMap kmap) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int bpp = kTokensPerPage / a.ratio;
  const int stage_bytes = bpp * DI * 2;
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * stage_bytes);
  uint64_t* empty = full + kStages;
  int* pref = reinterpret_cast<int*>(empty + kStages);  // pages of complete blocks, exclusive prefix [B+1]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int MAXL = a.maxPagesPerSeq * kTokensPerPage;

  for (int b = tid; b < a.B; b += blockDim.x) {
    const int L = max(0, min(a.ctx[b], MAXL));
    pref[b + 1] = (L / a.ratio + bpp - 1) / bpp;
  }
  if (tid == 0) {
    pref[0] = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < a.B; base += 32) {
      const int i = base + lane;
      int v = i < a.B ? pref[i + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += y;
      }
      if (i < a.B) pref[i + 1] = v + carry;
      carry += __shfl_sync(kFull, v, 31);
    }
  }
  __syncthreads();
  const long long W = pref[a.B];
  const long long lo = W * blockIdx.x / gridDim.x, hi = W * (blockIdx.x + 1) / gridDim.x;
  if (lo >= hi) return;

  if (warp == kConsumerWarps) {  // ---- producer: page ids 32 at a time, one TMA per 64-dim half
    int bw = 0;  // sequence of the batch's first page
    bool alive = true;
    for (long long base = lo; base < hi && alive; base += 32) {
      while (base >= pref[bw + 1]) ++bw;
      const long long i = base + lane;
      int vp = 0;
      if (i < hi) {
        int bl = bw;
        while (i >= pref[bl + 1]) ++bl;
        vp = __ldg(a.pageTable + (static_cast<size_t>(bl) * 2 + 1) * a.maxPagesPerSeq + (i - pref[bl]));
        if (static_cast<unsigned>(vp) >= static_cast<unsigned>(a.numFlatPages)) {
          atomicOr(a.status, kErrBadPage);
          vp = 0;
        }
      }
      const int cnt = static_cast<int>(hi - base < 32 ? hi - base : 32);
      for (int k = 0; k < cnt; ++k) {
        const int vpk = __shfl_sync(kFull, vp, k);
        int ok = 1;
        if (lane == 0) {
          const int jdx = static_cast<int>(base + k - lo), s = jdx % kStages, n = jdx / kStages;
          if (!mbar_wait_bounded(&empty[s], (n & 1) ^ 1, kWaitLimitNs)) {
            atomicOr(a.status, kErrWaitTimeout);
            ok = 0;
          } else {
            mbar_arrive_expect_tx(&full[s], stage_bytes);
#pragma unroll
            for (int hh = 0; hh < DI / 64; ++hh)
              tma_load_3d(ring + s * stage_bytes + hh * bpp * 128, &kmap, 64 * hh, 0, vpk, &full[s]);
          }
        }
        if (!__shfl_sync(kFull, ok, 0)) {
          alive = false;
          break;
        }
      }
    }
    return;
  }

  // ---- consumers: warp w takes pages lo + w, lo + w + kConsumerWarps, ...; 16 lanes per key
  constexpr int LPB = DI / 8, BPW = 32 / LPB, LOGL = LPB == 16 ? 4 : 3;
  const int sub = lane % LPB;
  const int m = (sub >> (LOGL - 3)) & 7;
  uint64_t q2[8][4];
  int cached_b = -1, n_c = 0;
  int b = 0;
  float* myscr = reinterpret_cast<float*>(pref + (a.B + 1 + 3) / 4 * 4) + warp * 128;
  for (long long i = lo + warp; i < hi; i += kConsumerWarps) {
    while (i >= pref[b + 1]) ++b;
    const int p = static_cast<int>(i - pref[b]);
    const int jx = static_cast<int>(i - lo), s = jx % kStages, n = jx / kStages;
    if (b != cached_b) {
      const float* qb = a.q + static_cast<size_t>(b) * 8 * 128;
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float4 x0 = *reinterpret_cast<const float4*>(qb + (h ^ m) * 128 + sub * 8);
        const float4 x1 = *reinterpret_cast<const float4*>(qb + (h ^ m) * 128 + sub * 8 + 4);
        q2[h][0] = pack_f2(x0.x, x0.y);
        q2[h][1] = pack_f2(x0.z, x0.w);
        q2[h][2] = pack_f2(x1.x, x1.y);
        q2[h][3] = pack_f2(x1.z, x1.w);
      }
      n_c = max(0, min(a.ctx[b], MAXL)) / a.ratio;
      cached_b = b;
    }
    if (!mbar_wait_bounded(&full[s], n & 1, kWaitLimitNs)) {
      if (lane == 0) atomicOr(a.status, kErrWaitTimeout);
      break;
    }
    const uint8_t* tile = ring + s * stage_bytes;
#pragma unroll 2
    for (int pass = 0; pass < bpp / BPW; ++pass) {
      const int blk = pass * BPW + lane / LPB;
      const uint4 raw = *reinterpret_cast<const uint4*>(tile + (sub >> 3) * bpp * 128 + swz128(blk, sub & 7));
      const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
      uint64_t kp[4];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const float2 f = __half22float2(h2[jj]);
        kp[jj] = pack_f2(f.x, f.y);
      }
      float d[8];
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        uint64_t acc = ffma2(q2[h][0], kp[0], 0ull);
        acc = ffma2(q2[h][1], kp[1], acc);
        acc = ffma2(q2[h][2], kp[2], acc);
        acc = ffma2(q2[h][3], kp[3], acc);
        d[h] = lo_f2(acc) + hi_f2(acc);
      }
#pragma unroll
      for (int i2 = 0; i2 < 4; ++i2) d[i2] += __shfl_xor_sync(kFull, d[i2 + 4], LPB / 2);
#pragma unroll
      for (int i2 = 0; i2 < 2; ++i2) d[i2] += __shfl_xor_sync(kFull, d[i2 + 2], LPB / 4);
      d[0] += __shfl_xor_sync(kFull, d[1], LPB / 8);
      if (LPB == 16) d[0] += __shfl_xor_sync(kFull, d[0], 1);
      float sc = d[0] > 0.f ? d[0] : 0.f;
      sc += __shfl_xor_sync(kFull, sc, LPB / 8);
      sc += __shfl_xor_sync(kFull, sc, LPB / 4);
      sc += __shfl_xor_sync(kFull, sc, LPB / 2);
      if (sub == 0) myscr[blk] = sc;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    page_epilogue(a, b, p, n_c, bpp, myscr[lane < bpp ? lane : 0]);
    __syncwarp();
  }
}

// ------------------------------------------------------------------ B3
struct SelectArgs {
  const int32_t* ctx;
  const float* scores;
  int32_t* hist;
  int32_t* sureId;
  uint32_t* tieKey;
  int32_t* tieId;
  int32_t* counters;  // [B][3]: sure count, tie count, ticket
  int32_t* indices;
  int maxPagesPerSeq, ratio, budget, topK, nbmax;
};

__global__ void __launch_bounds__(kSelThreads) decode_select_kernel(const SelectArgs a) {
  __shared__ int red[2 * kSelThreads / 32];
  __shared__ int scan[kSelThreads / 32];
  __shared__ int info[8];
  __shared__ int buf_s[kMaxSelect];            // filter: sure ids | final: kept ids to sort
  __shared__ uint32_t tkey_s[kSliceBlocks];    // filter: this slice's ties
  __shared__ int tid_s[kSliceBlocks];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s = blockIdx.x, b = blockIdx.y;
  const int L = max(0, min(a.ctx[b], a.maxPagesPerSeq * kTokensPerPage));
  const int t = L - 1;
  const int n_c = L / a.ratio;
  int32_t* out = a.indices + static_cast<size_t>(b) * a.topK;
  int32_t* hrow = a.hist + static_cast<size_t>(b) * kNumBins;
  int32_t* ctr = a.counters + static_cast<size_t>(b) * 3;
  if (L == 0) {
    if (s == 0)
      for (int i = tid; i < a.topK; i += kSelThreads) out[i] = -1;
    return;
  }
  if (n_c <= a.budget) {  // every block kept: the list is 0..t
    if (s == 0) {
      for (int i = tid; i < a.topK; i += kSelThreads) out[i] = i <= t ? i : -1;
      for (int i = tid; i < kNumBins; i += kSelThreads) hrow[i] = 0;
    }
    return;
  }
  const int nsplit = (n_c + kSliceBlocks - 1) / kSliceBlocks;
  if (s >= nsplit) return;

  // ---- the bin holding the budget-th largest score
  constexpr int BPT = kNumBins / kSelThreads;  // 16 bins per thread
  int h[BPT];
  int own = 0;
#pragma unroll
  for (int k = 0; k < BPT; ++k) {
    h[k] = __ldcg(hrow + tid * BPT + k);
    own += h[k];
  }
  if (tid == 0) {
    info[0] = 0;  // threshold bin
    info[1] = 0;  // blocks in higher bins
    info[2] = 0;  // sure blocks gathered by this CTA
    info[3] = 0;  // ties gathered by this CTA
  }
  int total;
  const int excl = cta_exclusive_scan<kSelThreads>(own, scan, total);
  int running = total - excl - own;  // blocks in bins of higher threads
#pragma unroll
  for (int k = BPT - 1; k >= 0; --k) {
    if (running < a.budget && running + h[k] >= a.budget) {
      info[0] = tid * BPT + k;
      info[1] = running;
    }
    running += h[k];
  }
  __syncthreads();
  const int T = info[0], c_above = info[1];

  // ---- classify this slice: above the bin (kept) or inside it (tie)
  const float* srow = a.scores + static_cast<size_t>(b) * a.nbmax;
  const int g0 = s * kSliceBlocks, g1 = min(g0 + kSliceBlocks, n_c);
  constexpr int U = kSliceBlocks / kSelThreads;
  uint32_t keys[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int g = g0 + u * kSelThreads + tid;
    keys[u] = g < g1 ? __float_as_uint(__ldcg(srow + g)) : 0u;
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int g = g0 + u * kSelThreads + tid;
    const bool valid = g < g1;
    const int bin = static_cast<int>(keys[u] >> kBinShift);
    const bool sure = valid && bin > T, tie = valid && bin == T;
    const unsigned sm = __ballot_sync(kFull, sure), tm = __ballot_sync(kFull, tie);
    const unsigned lt = (1u << lane) - 1u;
    if (sm) {
      int p0 = 0;
      if (lane == 0) p0 = atomicAdd(&info[2], __popc(sm));
      p0 = __shfl_sync(kFull, p0, 0);
      if (sure) {
        const int at = p0 + __popc(sm & lt);
        if (at < kMaxSelect) buf_s[at] = g;
      }
    }
    if (tm) {
      int p0 = 0;
      if (lane == 0) p0 = atomicAdd(&info[3], __popc(tm));
      p0 = __shfl_sync(kFull, p0, 0);
      if (tie) {
        const int at = p0 + __popc(tm & lt);
        tkey_s[at] = keys[u];
        tid_s[at] = g;
      }
    }
  }
  __syncthreads();
  {  // one global reservation per list per CTA
    const int ns = min(info[2], kMaxSelect), nts = info[3];
    if (tid == 0) {
      info[4] = ns ? atomicAdd(ctr + 0, ns) : 0;
      info[5] = nts ? atomicAdd(ctr + 1, nts) : 0;
    }
    __syncthreads();
    const int as = info[4], at = info[5];
    for (int e = tid; e < ns; e += kSelThreads)
      if (as + e < a.budget) a.sureId[static_cast<size_t>(b) * a.budget + as + e] = buf_s[e];
    for (int e = tid; e < nts; e += kSelThreads) {
      a.tieKey[static_cast<size_t>(b) * a.nbmax + at + e] = tkey_s[e];
      a.tieId[static_cast<size_t>(b) * a.nbmax + at + e] = tid_s[e];
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) info[6] = atomicAdd(ctr + 2, 1) == nsplit - 1;
  __syncthreads();
  if (!info[6]) return;
  __threadfence();

  // ---- last CTA: kept blocks = the sure ones + the top of the tie bin by (score desc, id asc)
  const int need = a.budget - c_above;
  const int nt = __ldcg(ctr + 1);
  const uint32_t* tk = a.tieKey + static_cast<size_t>(b) * a.nbmax;
  const int32_t* ti = a.tieId + static_cast<size_t>(b) * a.nbmax;
  for (int e = tid; e < c_above; e += kSelThreads) buf_s[e] = __ldcg(a.sureId + static_cast<size_t>(b) * a.budget + e);
  if (tid == 0) info[7] = c_above;  // next free slot of buf_s
  __syncthreads();
  auto keep = [&](int id) {
    const int at = atomicAdd(&info[7], 1);
    if (at < kMaxSelect) buf_s[at] = id;
  };
  if (nt <= need) {
    for (int e = tid; e < nt; e += kSelThreads) keep(__ldcg(ti + e));
  } else {
    // bisection on the score bits inside bin T, then on the id among exact ties at the cut
    const bool regs = nt <= kTieVPT * kSelThreads;
    uint32_t key[kTieVPT];
    int id[kTieVPT];
    const int nv = regs ? max(0, min(kTieVPT, nt - tid * kTieVPT)) : 0;
#pragma unroll
    for (int v = 0; v < kTieVPT; ++v) {
      key[v] = v < nv ? __ldcg(tk + tid * kTieVPT + v) : 0u;
      id[v] = v < nv ? __ldcg(ti + tid * kTieVPT + v) : 0;
    }
    auto count_ge = [&](uint32_t x) {
      int c = 0;
      if (regs) {
#pragma unroll
        for (int v = 0; v < kTieVPT; ++v) c += (v < nv && key[v] >= x) ? 1 : 0;
      } else {
        for (int e = tid; e < nt; e += kSelThreads) c += __ldcg(tk + e) >= x ? 1 : 0;
      }
      return c;
    };
    auto count_eq_le = [&](uint32_t x, int y) {
      int c = 0;
      if (regs) {
#pragma unroll
        for (int v = 0; v < kTieVPT; ++v) c += (v < nv && key[v] == x && id[v] <= y) ? 1 : 0;
      } else {
        for (int e = tid; e < nt; e += kSelThreads) c += (__ldcg(tk + e) == x && __ldcg(ti + e) <= y) ? 1 : 0;
      }
      return c;
    };
    int phase = 0;
    uint32_t lo = static_cast<uint32_t>(T) << kBinShift, hi = static_cast<uint32_t>(T + 1) << kBinShift;
    int cnt_lo = nt, cnt_hi = 0;  // count(>= lo) >= need > count(>= hi)
    while (hi - lo > 1u) {
      const uint32_t mid = lo + ((hi - lo) >> 1);
      const int tot = cta_sum<kSelThreads>(count_ge(mid), red, phase);
      if (tot >= need) {
        lo = mid;
        cnt_lo = tot;
      } else {
        hi = mid;
        cnt_hi = tot;
      }
    }
    const uint32_t Tk = lo;
    const int n_eq = need - cnt_hi;  // keys equal to Tk to keep, lowest ids first
    int ilo = -1, ihi = a.nbmax;
    if (cnt_lo - cnt_hi != n_eq) {
      while (ihi - ilo > 1) {
        const int mid = ilo + ((ihi - ilo) >> 1);
        if (cta_sum<kSelThreads>(count_eq_le(Tk, mid), red, phase) >= n_eq)
          ihi = mid;
        else
          ilo = mid;
      }
    }
    if (regs) {
#pragma unroll
      for (int v = 0; v < kTieVPT; ++v)
        if (v < nv && (key[v] > Tk || (key[v] == Tk && id[v] <= ihi))) keep(id[v]);
    } else {
      for (int e = tid; e < nt; e += kSelThreads) {
        const uint32_t k = __ldcg(tk + e);
        const int i2 = __ldcg(ti + e);
        if (k > Tk || (k == Tk && i2 <= ihi)) keep(i2);
      }
    }
  }
  __syncthreads();
  // ---- sort the kept ids ascending (bitonic, padded to a power of two), expand with the tail
  const int nk = min(info[7], kMaxSelect);
  int np2 = 1;
  while (np2 < nk) np2 <<= 1;
  for (int e = nk + tid; e < np2; e += kSelThreads) buf_s[e] = 0x7fffffff;
  __syncthreads();
  for (int k = 2; k <= np2; k <<= 1) {
    for (int jb = k >> 1; jb > 0; jb >>= 1) {
      for (int e = tid; e < np2; e += kSelThreads) {
        const int f = e ^ jb;
        if (f > e) {
          const int x = buf_s[e], y = buf_s[f];
          const bool up = (e & k) == 0;
          if ((x > y) == up) {
            buf_s[e] = y;
            buf_s[f] = x;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int e = tid; e < nk * a.ratio && e < a.topK; e += kSelThreads) out[e] = buf_s[e / a.ratio] * a.ratio + e % a.ratio;
  const int head = nk * a.ratio;
  for (int i = head + tid; i < a.topK; i += kSelThreads) {
    const int j = n_c * a.ratio + (i - head);
    out[i] = j <= t ? j : -1;
  }
  // re-arm for the next call
  for (int i = tid; i < kNumBins; i += kSelThreads) hrow[i] = 0;
  if (tid == 0) {
    ctr[0] = 0;
    ctr[1] = 0;
    ctr[2] = 0;
  }
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace

size_t indexer_decode_workspace_bytes(int B, int maxPagesPerSeq, int ratio, int budget) {
  const int nbmax = maxPagesPerSeq * (kTokensPerPageHost / ratio);
  return ws_layout(B, nbmax, budget).total;
}

cudaError_t launch_indexer_decode(const QsaIndexerDecodeParams& p, const RopeFreqs& rf,
                                  const CUtensorMap& kbarMap) {
  const int B = p.batchSize;
  const int bpp = kTokensPerPageHost / p.compressRatio;
  const int nbmax = p.maxPagesPerSeq * bpp;
  const WsLayout l = ws_layout(B, nbmax, p.budget);
  uint8_t* ws = static_cast<uint8_t*>(p.workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  float* q = reinterpret_cast<float*>(ws + l.q);
  float* scores = reinterpret_cast<float*>(ws + l.scores);
  int32_t* hist = reinterpret_cast<int32_t*>(ws + l.hist);
  int32_t* counters = reinterpret_cast<int32_t*>(ws + l.counters);
  cudaStream_t st = static_cast<cudaStream_t>(p.stream);

  PrepArgs pa;
  pa.idxQ = static_cast<const __half*>(p.idxQ);
  pa.idxK = static_cast<const __half*>(p.idxK);
  pa.wq = p.qNormW;
  pa.wk = p.kNormW;
  pa.pool = static_cast<__half*>(p.kvPool);
  pa.pageTable = p.pageTable;
  pa.ctx = p.contextLengths;
  pa.q = q;
  pa.status = status;
  pa.Hi = p.numHeads;
  pa.Hkv = p.numKVHeads;
  pa.D = p.kvHeadDim;
  pa.poolHeadDim = p.poolHeadDim;
  pa.numFlatPages = p.numFlatPages;
  pa.maxPagesPerSeq = p.maxPagesPerSeq;
  pa.rot = p.rotDim;
  pa.ratio = p.compressRatio;
  pa.eps = p.rmsNormEps;
  pa.rf = rf;
  if (p.headDim == 64)
    decode_prep_kernel<64><<<B, 256, 0, st>>>(pa);
  else
    decode_prep_kernel<128><<<B, 256, 0, st>>>(pa);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  ScoreArgs sa;
  sa.ctx = p.contextLengths;
  sa.pageTable = p.pageTable;
  sa.q = q;
  sa.scores = scores;
  sa.hist = hist;
  sa.status = status;
  sa.B = B;
  sa.maxPagesPerSeq = p.maxPagesPerSeq;
  sa.numFlatPages = p.numFlatPages;
  sa.ratio = p.compressRatio;
  sa.nbmax = nbmax;
  const int smem = score_smem_bytes(p.headDim, p.compressRatio, B);
  if (smem > kMaxDynSmem) return cudaErrorInvalidValue;
  const long long maxPages = static_cast<long long>(B) * p.maxPagesPerSeq;
  const int grid = static_cast<int>(maxPages < sm_count() ? maxPages : sm_count());
  if (p.headDim == 64) {
    static const cudaError_t attr = cudaFuncSetAttribute(
        decode_score_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
    if (attr != cudaSuccess) return attr;
    decode_score_kernel<64><<<grid, kScoreThreads, smem, st>>>(sa, kbarMap);
  } else {
    static const cudaError_t attr = cudaFuncSetAttribute(
        decode_score_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
    if (attr != cudaSuccess) return attr;
    decode_score_kernel<128><<<grid, kScoreThreads, smem, st>>>(sa, kbarMap);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  SelectArgs se;
  se.ctx = p.contextLengths;
  se.scores = scores;
  se.hist = hist;
  se.sureId = reinterpret_cast<int32_t*>(ws + l.sureId);
  se.tieKey = reinterpret_cast<uint32_t*>(ws + l.tieKey);
  se.tieId = reinterpret_cast<int32_t*>(ws + l.tieId);
  se.counters = counters;
  se.indices = p.indices;
  se.maxPagesPerSeq = p.maxPagesPerSeq;
  se.ratio = p.compressRatio;
  se.budget = p.budget;
  se.topK = p.topK;
  se.nbmax = nbmax;
  dim3 sgrid((nbmax + kSliceBlocks - 1) / kSliceBlocks, B);
  decode_select_kernel<<<sgrid, kSelThreads, 0, st>>>(se);
  return cudaGetLastError();
}

}  // namespace qsa
