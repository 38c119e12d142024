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
//       complete blocks (one 3-D TMA copy per page: box {di, 128/r, 1} over a
//       strided view of the pool) into a 24-stage ring; 15 consumer warps
//       score one page each (8 dims x 8 heads per lane with paired fp32 FMA, a
//       transposing shuffle reduction whose head order is pre-permuted per
//       lane so that no select is needed), write the scores and add them to a
//       4096-bin histogram of the score bits per sequence.  Pages are split
//       evenly over the CTAs, so HBM streams without per-chunk stalls.
//   decode_select_kernel  (B3) per sequence: the histogram gives the bin that
//       holds the budget-th largest score; CTAs over 8192-block slices mark
//       every block above that bin in a bitmap and append the blocks inside
//       it; the last CTA to finish picks the exact top of those by (score
//       desc, id asc), expands the bitmap in ascending order with the causal
//       tail, and re-arms the histogram and counters.
// Waits on TMA barriers are bounded; on expiry the kernel records
// kErrWaitTimeout in the workspace status word and stops.
#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr size_t kStatusBytes = 256;
constexpr int kNumBins = 4096;       // histogram of (score bits >> 19): exponent + 4 mantissa bits
constexpr int kBinShift = 19;
constexpr int kSliceBlocks = 8192;   // blocks one select CTA filters
constexpr int kConsumerWarps = 15;  // + 1 producer warp = 16 warps, up to 128 registers each
constexpr int kScoreThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 24;
constexpr int kSelThreads = 256;
constexpr int kTieVPT = 16;          // tie candidates per thread held in registers
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;  // 0.2 s
constexpr int kMaxDynSmem = 227 * 1024;

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

struct WsLayout {
  size_t q, scores, hist, bitmap, tieKey, tieId, counters, total;
};
WsLayout ws_layout(int B, int nbmax) {
  WsLayout l;
  size_t off = kStatusBytes;
  l.q = off;
  off += up256(static_cast<size_t>(B) * 8 * 128 * 4);  // prepared queries fp32 [B][8][128]
  l.scores = off;
  off += up256(static_cast<size_t>(B) * nbmax * 4);     // block scores fp32 [B][nbmax]
  l.hist = off;
  off += up256(static_cast<size_t>(B) * kNumBins * 4);  // int32 [B][kNumBins], zero between calls
  l.bitmap = off;
  off += up256(static_cast<size_t>(B) * ((nbmax + 31) / 32) * 4);
  l.tieKey = off;
  off += up256(static_cast<size_t>(B) * nbmax * 4);
  l.tieId = off;
  off += up256(static_cast<size_t>(B) * nbmax * 4);
  l.counters = off;
  off += up256(static_cast<size_t>(B) * 2 * 4);         // tie count, ticket: zero between calls
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
      sincos(__dmul_rn(pos, a.rf.inv_freq[i]), &s, &c);
      r = __dsub_rn(__dmul_rn(y2_s[i], c), __dmul_rn(y2_s[i + half], s));
    } else if (i < a.rot) {
      const int k = i - half;
      double s, c;
      sincos(__dmul_rn(pos, a.rf.inv_freq[k]), &s, &c);
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

template <int DI>
__global__ void __launch_bounds__(kScoreThreads, 1) decode_score_kernel(const ScoreArgs a,
                                                                        const __grid_constant__ CUtensorMap kmap) {
  constexpr int LPB = DI / 8;          // lanes per block key (8 dims each)
  constexpr int BPW = 32 / LPB;        // block keys per warp pass
  constexpr int LOGL = LPB == 16 ? 4 : 3;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int bpp = kTokensPerPage / a.ratio;
  const int stage_bytes = bpp * DI * 2;
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * stage_bytes);
  uint64_t* empty = full + kStages;
  int* pref = reinterpret_cast<int*>(empty + kStages);  // pages of complete blocks, exclusive prefix [B+1]
  float* scr = reinterpret_cast<float*>(pref + (a.B + 1 + 3) / 4 * 4);  // [kConsumerWarps][128]
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

  if (warp == kConsumerWarps) {  // ---- producer
    if (lane == 0) {
      int b = 0;
      for (long long i = lo; i < hi; ++i) {
        while (i >= pref[b + 1]) ++b;
        const int p = static_cast<int>(i - pref[b]);
        int vp = __ldg(a.pageTable + (static_cast<size_t>(b) * 2 + 1) * a.maxPagesPerSeq + p);
        if (static_cast<unsigned>(vp) >= static_cast<unsigned>(a.numFlatPages)) {
          atomicOr(a.status, kErrBadPage);
          vp = 0;
        }
        const int j = static_cast<int>(i - lo), s = j % kStages, n = j / kStages;
        if (!mbar_wait_bounded(&empty[s], (n & 1) ^ 1, kWaitLimitNs)) {
          atomicOr(a.status, kErrWaitTimeout);
          break;
        }
        mbar_arrive_expect_tx(&full[s], stage_bytes);
        tma_load_3d(ring + s * stage_bytes, &kmap, 0, 0, vp, &full[s]);
      }
    }
    return;
  }

  // ---- consumers: warp w takes pages lo + w, lo + w + kConsumerWarps, ...
  const int sub = lane % LPB;
  const int m = (sub >> (LOGL - 3)) & 7;  // this lane's head order is h ^ m (see the reduction)
  uint64_t q2[8][4];
  int cached_b = -1, n_c = 0;
  int b = 0;
  float* myscr = scr + warp * 128;
  for (long long i = lo + warp; i < hi; i += kConsumerWarps) {
    while (i >= pref[b + 1]) ++b;
    const int p = static_cast<int>(i - pref[b]);
    const int j = static_cast<int>(i - lo), s = j % kStages, n = j / kStages;
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
    const __half* tile = reinterpret_cast<const __half*>(ring + s * stage_bytes);
    for (int pass = 0; pass < bpp / BPW; ++pass) {
      const int blk = pass * BPW + lane / LPB;
      const uint4 raw = *reinterpret_cast<const uint4*>(tile + blk * DI + sub * 8);
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
      // Transposing reduction over the LPB lanes of this key.  Lane head order
      // h ^ m makes the partner's upper half hold the same heads as this
      // lane's lower half at every step, so each step is add(shuffle).
#pragma unroll
      for (int i2 = 0; i2 < 4; ++i2) d[i2] += __shfl_xor_sync(kFull, d[i2 + 4], LPB / 2);
#pragma unroll
      for (int i2 = 0; i2 < 2; ++i2) d[i2] += __shfl_xor_sync(kFull, d[i2 + 2], LPB / 4);
      d[0] += __shfl_xor_sync(kFull, d[1], LPB / 8);
      if (LPB == 16) d[0] += __shfl_xor_sync(kFull, d[0], 1);
      float sc = d[0] > 0.f ? d[0] : 0.f;  // relu of head m's dot
      sc += __shfl_xor_sync(kFull, sc, LPB / 8);
      sc += __shfl_xor_sync(kFull, sc, LPB / 4);
      sc += __shfl_xor_sync(kFull, sc, LPB / 2);
      if (sub == 0) myscr[blk] = sc;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);  // the stage may be refilled
    float* sc_row = a.scores + static_cast<size_t>(b) * a.nbmax;
    int32_t* hrow = a.hist + static_cast<size_t>(b) * kNumBins;
    for (int r0 = 0; r0 < bpp; r0 += 32) {
      const int jb = r0 + lane;
      const int g = p * bpp + jb;
      const bool valid = jb < bpp && g < n_c;
      const float sc = valid ? myscr[jb] : 0.f;
      const int bin = static_cast<int>(__float_as_uint(sc) >> kBinShift);
      if (valid) sc_row[g] = sc;
      const unsigned act = __ballot_sync(kFull, valid);
      if (valid) {
        const unsigned peers = __match_any_sync(act, bin);
        if (lane == __ffs(peers) - 1) atomicAdd(hrow + bin, __popc(peers));
      }
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------ B3
struct SelectArgs {
  const int32_t* ctx;
  const float* scores;
  int32_t* hist;
  uint32_t* bitmap;
  uint32_t* tieKey;
  int32_t* tieId;
  int32_t* tieCnt;
  int32_t* ticket;
  int32_t* indices;
  int maxPagesPerSeq, ratio, budget, topK, nbmax, words;
};

__global__ void __launch_bounds__(kSelThreads) decode_select_kernel(const SelectArgs a) {
  __shared__ int red[2 * kSelThreads / 32];
  __shared__ int scan[kSelThreads / 32];
  __shared__ int info[4];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s = blockIdx.x, b = blockIdx.y;
  const int L = max(0, min(a.ctx[b], a.maxPagesPerSeq * kTokensPerPage));
  const int t = L - 1;
  const int n_c = L / a.ratio;
  int32_t* out = a.indices + static_cast<size_t>(b) * a.topK;
  int32_t* hrow = a.hist + static_cast<size_t>(b) * kNumBins;
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

  // ---- mark blocks above the bin, collect the blocks inside it
  const float* srow = a.scores + static_cast<size_t>(b) * a.nbmax;
  uint32_t* brow = a.bitmap + static_cast<size_t>(b) * a.words;
  const int g1 = min((s + 1) * kSliceBlocks, n_c);
  for (int base = s * kSliceBlocks + warp * 32; base < g1; base += kSelThreads) {
    const int g = base + lane;
    const bool valid = g < g1;
    const uint32_t key = valid ? __float_as_uint(__ldcg(srow + g)) : 0u;
    const int bin = static_cast<int>(key >> kBinShift);
    const unsigned sure = __ballot_sync(kFull, valid && bin > T);
    if (lane == 0) brow[base >> 5] = sure;
    const bool tie = valid && bin == T;
    const unsigned tm = __ballot_sync(kFull, tie);
    if (tm) {
      int pos0 = 0;
      if (lane == 0) pos0 = atomicAdd(a.tieCnt + b, __popc(tm));
      pos0 = __shfl_sync(kFull, pos0, 0);
      if (tie) {
        const int at = pos0 + __popc(tm & ((1u << lane) - 1u));
        a.tieKey[static_cast<size_t>(b) * a.nbmax + at] = key;
        a.tieId[static_cast<size_t>(b) * a.nbmax + at] = g;
      }
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) info[2] = atomicAdd(a.ticket + b, 1) == nsplit - 1;
  __syncthreads();
  if (!info[2]) return;
  __threadfence();

  // ---- last CTA: exact top of the tie bin by (score desc, id asc)
  const int need = a.budget - c_above;
  const int nt = __ldcg(a.tieCnt + b);
  const uint32_t* tk = a.tieKey + static_cast<size_t>(b) * a.nbmax;
  const int32_t* ti = a.tieId + static_cast<size_t>(b) * a.nbmax;
  if (nt <= need) {
    for (int e = tid; e < nt; e += kSelThreads) {
      const int id = __ldcg(ti + e);
      atomicOr(brow + (id >> 5), 1u << (id & 31));
    }
  } else if (nt <= kTieVPT * kSelThreads) {
    uint32_t key[kTieVPT];
    int id[kTieVPT];
    const int nv = max(0, min(kTieVPT, nt - tid * kTieVPT));
#pragma unroll
    for (int v = 0; v < kTieVPT; ++v) {
      key[v] = v < nv ? __ldcg(tk + tid * kTieVPT + v) : 0u;
      id[v] = v < nv ? __ldcg(ti + tid * kTieVPT + v) : 0;
    }
    int phase = 0;
    // every tie key lies in bin T: count(>= lo) >= need > count(>= hi)
    uint32_t lo = static_cast<uint32_t>(T) << kBinShift, hi = static_cast<uint32_t>(T + 1) << kBinShift;
    int cnt_lo = nt, cnt_hi = 0;
    while (hi - lo > 1u) {
      const uint32_t mid = lo + ((hi - lo) >> 1);
      int c = 0;
#pragma unroll
      for (int v = 0; v < kTieVPT; ++v) c += (v < nv && key[v] >= mid) ? 1 : 0;
      const int tot = cta_sum<kSelThreads>(c, red, phase);
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
    int ilo = -1, ihi = a.nbmax;     // count(== Tk, id <= ilo) < n_eq <= count(== Tk, id <= ihi)
    if (cnt_lo - cnt_hi == n_eq) ilo = ihi - 1;  // no exact tie at the cut: keep every key == Tk
    while (ihi - ilo > 1) {
      const int mid = ilo + ((ihi - ilo) >> 1);
      int c = 0;
#pragma unroll
      for (int v = 0; v < kTieVPT; ++v) c += (v < nv && key[v] == Tk && id[v] <= mid) ? 1 : 0;
      const int tot = cta_sum<kSelThreads>(c, red, phase);
      if (tot >= n_eq)
        ihi = mid;
      else
        ilo = mid;
    }
#pragma unroll
    for (int v = 0; v < kTieVPT; ++v)
      if (v < nv && (key[v] > Tk || (key[v] == Tk && id[v] <= ihi))) atomicOr(brow + (id[v] >> 5), 1u << (id[v] & 31));
  } else {
    // Degenerate case (very many scores in one bin, e.g. all zero): the same
    // two bisections, counting straight from global memory.
    int phase = 0;
    uint32_t lo = static_cast<uint32_t>(T) << kBinShift, hi = static_cast<uint32_t>(T + 1) << kBinShift;
    int cnt_lo = nt, cnt_hi = 0;
    while (hi - lo > 1u) {
      const uint32_t mid = lo + ((hi - lo) >> 1);
      int c = 0;
      for (int e = tid; e < nt; e += kSelThreads) c += __ldcg(tk + e) >= mid ? 1 : 0;
      const int tot = cta_sum<kSelThreads>(c, red, phase);
      if (tot >= need) {
        lo = mid;
        cnt_lo = tot;
      } else {
        hi = mid;
        cnt_hi = tot;
      }
    }
    const uint32_t Tk = lo;
    const int n_eq = need - cnt_hi;
    int ilo = -1, ihi = a.nbmax;
    if (cnt_lo - cnt_hi == n_eq) ilo = ihi - 1;
    while (ihi - ilo > 1) {
      const int mid = ilo + ((ihi - ilo) >> 1);
      int c = 0;
      for (int e = tid; e < nt; e += kSelThreads) c += (__ldcg(tk + e) == Tk && __ldcg(ti + e) <= mid) ? 1 : 0;
      const int tot = cta_sum<kSelThreads>(c, red, phase);
      if (tot >= n_eq)
        ihi = mid;
      else
        ilo = mid;
    }
    for (int e = tid; e < nt; e += kSelThreads) {
      const uint32_t k = __ldcg(tk + e);
      const int id = __ldcg(ti + e);
      if (k > Tk || (k == Tk && id <= ihi)) atomicOr(brow + (id >> 5), 1u << (id & 31));
    }
  }
  __threadfence();
  __syncthreads();

  // ---- expand the bitmap in ascending order, then the causal tail
  const int nw = (n_c + 31) / 32;
  const int wpt = (nw + kSelThreads - 1) / kSelThreads;
  const int w0 = min(tid * wpt, nw), w1 = min(w0 + wpt, nw);
  int cnt = 0;
  for (int w = w0; w < w1; ++w) cnt += __popc(__ldcg(brow + w));
  int tot;
  int pos = cta_exclusive_scan<kSelThreads>(cnt, scan, tot);
  for (int w = w0; w < w1; ++w) {
    uint32_t bits = __ldcg(brow + w);
    while (bits) {
      const int id = w * 32 + __ffs(bits) - 1;
      bits &= bits - 1;
      for (int jj = 0; jj < a.ratio; ++jj)
        if (pos * a.ratio + jj < a.topK) out[pos * a.ratio + jj] = id * a.ratio + jj;
      ++pos;
    }
  }
  const int head = tot * a.ratio;
  for (int i = head + tid; i < a.topK; i += kSelThreads) {
    const int j = n_c * a.ratio + (i - head);
    out[i] = j <= t ? j : -1;
  }
  // re-arm for the next call
  for (int i = tid; i < kNumBins; i += kSelThreads) hrow[i] = 0;
  if (tid == 0) {
    a.tieCnt[b] = 0;
    a.ticket[b] = 0;
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
  (void)budget;
  const int nbmax = maxPagesPerSeq * (kTokensPerPageHost / ratio);
  return ws_layout(B, nbmax).total;
}

cudaError_t launch_indexer_decode(const QsaIndexerDecodeParams& p, const RopeFreqs& rf,
                                  const CUtensorMap& kbarMap) {
  const int B = p.batchSize;
  const int bpp = kTokensPerPageHost / p.compressRatio;
  const int nbmax = p.maxPagesPerSeq * bpp;
  const WsLayout l = ws_layout(B, nbmax);
  uint8_t* ws = static_cast<uint8_t*>(p.workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  float* q = reinterpret_cast<float*>(ws + l.q);
  float* scores = reinterpret_cast<float*>(ws + l.scores);
  int32_t* hist = reinterpret_cast<int32_t*>(ws + l.hist);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(ws + l.bitmap);
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
  se.bitmap = bitmap;
  se.tieKey = reinterpret_cast<uint32_t*>(ws + l.tieKey);
  se.tieId = reinterpret_cast<int32_t*>(ws + l.tieId);
  se.tieCnt = counters;
  se.ticket = counters + B;
  se.indices = p.indices;
  se.maxPagesPerSeq = p.maxPagesPerSeq;
  se.ratio = p.compressRatio;
  se.budget = p.budget;
  se.topK = p.topK;
  se.nbmax = nbmax;
  se.words = (nbmax + 31) / 32;
  dim3 sgrid((nbmax + kSliceBlocks - 1) / kSliceBlocks, B);
  decode_select_kernel<<<sgrid, kSelThreads, 0, st>>>(se);
  return cudaGetLastError();
}

}  // namespace qsa
