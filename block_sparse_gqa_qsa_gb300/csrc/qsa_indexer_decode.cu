// qsa_indexer_decode.cu -- the QSA indexer for one new token per sequence over
// the paged KV pool ("Qsa Attention Plugin", step 3: B1 fused q-prep +
// predicated tail write / compress, B2 block scores from the kbar tails, B3
// deterministic top-512 + expand; "KV pool contract" for where the state lives).
//
// Three launches on the caller's stream:
//   decode_prep_kernel    (B1) one CTA per sequence: index-query prep at
//       t = L-1 (fp32, angles reduced in integer turns) into the workspace by
//       8 warps, and concurrently, by di/32 more warps, the state update: the new
//       raw key into token t's K-row tail when t leaves its block incomplete,
//       else the block t completes is pooled (from the K-row tails of its
//       first r-1 tokens and the new key; exact mean, double-float norm and
//       rotation, qsa_blockkey.cuh) and its key is stored in the V-row tail of
//       the block's first token.
//   decode_score_kernel   (B2) persistent, one CTA per SM, warp-specialised:
//       a producer warp streams the key tails of every page that holds
//       complete blocks (3-D TMA copies, box {64, 128/r, 1} with the 128-byte
//       swizzle over a strided view of the pool, page ids fetched 32 at a time)
//       into a 22-stage ring; 11 consumer warps score one page each: four
//       lanes per key (a quarter of the dims each), four keys per lane, the
//       queries read by broadcast from the CTA's shared-memory copy (written
//       by B1 in that layout), dims paired in fp32x2 FMAs; two transposing
//       shuffle exchanges join the quarters, then relu per head and the head
//       sum.  They write the scores and add them to a 4096-bin histogram of
//       the score bits per sequence.  Pages are split evenly over the CTAs.
//   decode_select_kernel  (B3) per sequence: the histogram gives the bin T that
//       holds the budget-th largest score.  A sequence of at most 8 slices of
//       2048 blocks is handled by one CTA, which loads all its scores at once
//       and compacts the candidates (blocks in bins >= T) in ascending id order
//       straight into shared memory.  Longer ones: one CTA per slice writes
//       the slice's candidates (blocks in bins >= T) in ascending id order
//       into the slice's own region (no global atomics); the last CTA to
//       finish finds the exact cut inside bin T with two radix digits of the
//       score bits in shared memory, keeps the blocks above the cut and, of
//       those equal to it, the lowest ids, and emits the list by filtering the
//       already ascending candidates; then the causal tail, and it re-arms
//       the histogram and its ticket.
// Waits on TMA barriers are bounded; on expiry the kernel records
// kErrWaitTimeout in the workspace status word and stops.
#include <atomic>

#include "qsa_blockkey.cuh"
#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr size_t kStatusBytes = 256;
constexpr int kNumBins = 4096;       // histogram of (score bits >> 19): exponent + 4 mantissa bits
constexpr int kBinShift = 19;
constexpr int kSliceBlocks = 2048;   // blocks one select CTA filters (8 per thread, one round of loads)
constexpr int kMaxSlices = 1024;     // slices per sequence (blocks <= 2M): their bases live in shared memory
constexpr int kStageCand = 4096;     // candidates the final CTA stages in shared memory (more: read from L2)
constexpr int kSingleRounds = 8;     // sequences of up to 8 slices are selected by one CTA, in rounds
constexpr int kConsumerWarps = 11;  // + 1 producer warp: 12 warps (3 per SM sub-partition), up to 168 registers
constexpr int kScoreThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 22;
constexpr int kQSlots = 8;            // sequences whose queries a scorer CTA keeps in shared memory
// Queries as the scorer reads them: per sequence 4 quarters of the dims, each
// [chunk][head slot][8 dims] plus 4 floats of padding (the quarters then start
// in different banks); in quarter t, slot p holds head p ^ (4*(t>>1) + 2*(t&1)).
constexpr int kQS128 = (128 / 32) * 64 + 4;
constexpr int kQPerSeq = 4 * kQS128;  // floats per sequence in the workspace (the 128-dim layout)
constexpr int kSelThreads = 256;
constexpr int kPrepThreads = 256 + 128;  // 8 query-prep warps + up to 4 state-update warps
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;  // 0.2 s
constexpr int kMaxDynSmem = 227 * 1024;

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

struct WsLayout {
  size_t q, scores, hist, candKey, candId, sliceCnt, ticket, total;
};
WsLayout ws_layout(int B, int nbmax) {
  const int nsplit = (nbmax + kSliceBlocks - 1) / kSliceBlocks;
  WsLayout l;
  size_t off = kStatusBytes;
  l.q = off;
  off += up256(static_cast<size_t>(B) * kQPerSeq * 4);  // prepared queries fp32, scorer layout [B][kQPerSeq]
  l.scores = off;
  off += up256(static_cast<size_t>(B) * nbmax * 4);     // block scores fp32 [B][nbmax]
  l.hist = off;
  off += up256(static_cast<size_t>(B) * kNumBins * 4);  // int32 [B][kNumBins], zero between calls
  l.candKey = off;
  off += up256(static_cast<size_t>(B) * nbmax * 4);     // selection candidates, slice-major [B][nbmax]
  l.candId = off;
  off += up256(static_cast<size_t>(B) * nbmax * 4);
  l.sliceCnt = off;
  off += up256(static_cast<size_t>(B) * nsplit * 4);    // candidates per slice [B][nsplit]
  l.ticket = off;
  off += up256(static_cast<size_t>(B) * 4);             // slices done, zero between calls
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
__global__ void __launch_bounds__(kPrepThreads) decode_prep_kernel(const PrepArgs a) {
  constexpr int PER = DI / 32;
  __shared__ float y_s[8][DI];
  __shared__ f2x key_s[DI];
  __shared__ f2x part_s[DI / 32];
  __shared__ RopeSmem rs;
  __shared__ unsigned long long turn_s[64];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x;
  const int ctx_b = a.ctx[b];  // issued first: its latency overlaps the table copy
  stage_rope(a.rf, rs);
  if (tid < 64) turn_s[tid] = a.rf.turn[tid];
  __syncthreads();
  const int L = max(0, min(ctx_b, a.maxPagesPerSeq * kTokensPerPage));
  if (L == 0) return;
  const int t = L - 1;
  const int n_c = L / a.ratio;
  const bool completes = (L % a.ratio) == 0;
  const int32_t* ptK = a.pageTable + static_cast<size_t>(b) * 2 * a.maxPagesPerSeq;
  const int32_t* ptV = ptK + a.maxPagesPerSeq;

  // warps 0..7: index-query prep, warp h -> head h (heads >= Hi are zero);
  // warps 8..: the state update, concurrently (named barrier 1 among them)
  if (warp < 8) {
    const int h = warp;
    float* qo = a.q + static_cast<size_t>(b) * kQPerSeq;
    constexpr int QS = (DI / 32) * 64 + 4;
    auto qpos = [&](int i) {  // scorer layout position of (head h, dim i)
      const int qt = i / (DI / 4), c = (i % (DI / 4)) / 8;
      return qt * QS + c * 64 + (h ^ (4 * (qt >> 1) + 2 * (qt & 1))) * 8 + (i % 8);
    };
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
          rope_cos_sin_turns(static_cast<unsigned>(t), turn_s[i], cs, sn);
          v = y[p] * cs - y_s[h][i + half] * sn;
        } else if (i < a.rot) {
          const int k = i - half;
          float cs, sn;
          rope_cos_sin_turns(static_cast<unsigned>(t), turn_s[k], cs, sn);
          v = y[p] * cs + y_s[h][k] * sn;
        }
        qo[qpos(i)] = v;
      }
    } else {
#pragma unroll
      for (int p = 0; p < PER; ++p) qo[qpos(lane + 32 * p)] = 0.f;
    }
    return;
  }
  // warps 8..: the state update
  const int u = tid - 256;  // dim of the raw key this thread copies
  if (!completes) {
    const int kp = __ldg(ptK + (t >> 7));
    if (static_cast<unsigned>(kp) < static_cast<unsigned>(a.numFlatPages)) {
      a.pool[pool_row(kp, t & 127, a.Hkv, a.poolHeadDim) + a.D + u] = a.idxK[static_cast<size_t>(b) * DI + u];
    } else if (u == 0) {
      atomicOr(a.status, kErrBadPage);
    }
    return;
  }
  const int first = (n_c - 1) * a.ratio;  // all r tokens of the block share this page
  const int kp = __ldg(ptK + (first >> 7)), vp = __ldg(ptV + (first >> 7));
  const bool okp = static_cast<unsigned>(kp) < static_cast<unsigned>(a.numFlatPages) &&
                   static_cast<unsigned>(vp) < static_cast<unsigned>(a.numFlatPages);
  if (!okp) {
    if (u == 0) atomicOr(a.status, kErrBadPage);
    return;
  }
  const __half* newk = a.idxK + static_cast<size_t>(b) * DI;
  const __half* ktail = a.pool + pool_row(kp, first & 127, a.Hkv, a.poolHeadDim) + a.D;
  const size_t tok_stride = static_cast<size_t>(a.Hkv) * a.poolHeadDim;
  block_key<DI, DI / 32>([&](int j, int i) { return first + j == t ? newk[i] : ktail[j * tok_stride + i]; }, a.ratio,
                         a.wk, a.eps, a.rot, first, rs, key_s, part_s, warp - 8, 1,
                         a.pool + pool_row(vp, first & 127, a.Hkv, a.poolHeadDim) + a.D);
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
  uint64_t waitNs;  // bound of the waits on the stream's progress (copies in flight keep kWaitLimitNs)
};

__host__ __device__ __forceinline__ int score_smem_bytes(int di, int ratio, int B) {
  const int stage = (kTokensPerPage / ratio) * di * 2;
  return kStages * stage + 2 * kStages * 8 + ((B + 1 + 3) / 4) * 16 + kConsumerWarps * 128 * 4 +
         kQSlots * 4 * ((di / 32) * 64 + 4) * 4;
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

// Scores one page (bpp <= 32 block keys in a swizzled stage) for one warp.
// Lane (kk, hh) = (lane & 7, lane >> 3) holds keys kk + 8j (j < 4) and their
// dims [hh*DI/4, (hh+1)*DI/4); its quarter of the queries (qh, scorer layout)
// is read by broadcast, dims are paired in fp32x2 FMAs, and two transposing
// exchanges (lane ^ 16, then ^ 8) leave each lane the full dot products of its
// head slots 0 and 1 -- every step one shuffle and one add.  Writes the page's
// scores to myscr[0, 32).  kSmemQ: qh points to shared memory (else global).
template <int DI, bool kSmemQ>
__device__ __forceinline__ void score_page(const uint8_t* tile, int bpp, const float* qh, float* myscr) {
  constexpr int NCH = DI / 32;
  const int lane = threadIdx.x & 31, kk = lane & 7, hh = lane >> 3;
  uint64_t acc[4][8];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int h = 0; h < 8; ++h) acc[j][h] = 0ull;
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    const int cg = hh * NCH + c;  // this lane's chunk: half cg >> 3 of the row, 16-byte slot cg & 7
    uint64_t kp[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = (kk + 8 * j) & (bpp - 1);  // rows past a short page repeat (discarded)
      const uint4 raw = *reinterpret_cast<const uint4*>(tile + (cg >> 3) * bpp * 128 + swz128(r, cg & 7));
      const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const float2 f = __half22float2(h2[jj]);
        kp[j][jj] = pack_f2(f.x, f.y);
      }
    }
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      const float4* q4 = reinterpret_cast<const float4*>(qh + c * 64 + h * 8);
      const float4 qa = kSmemQ ? q4[0] : __ldg(q4);
      const float4 qb = kSmemQ ? q4[1] : __ldg(q4 + 1);
      const uint64_t q0 = pack_f2(qa.x, qa.y), q1 = pack_f2(qa.z, qa.w);
      const uint64_t q2 = pack_f2(qb.x, qb.y), q3 = pack_f2(qb.z, qb.w);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[j][h] = ffma2(q0, kp[j][0], acc[j][h]);
        acc[j][h] = ffma2(q1, kp[j][1], acc[j][h]);
        acc[j][h] = ffma2(q2, kp[j][2], acc[j][h]);
        acc[j][h] = ffma2(q3, kp[j][3], acc[j][h]);
      }
    }
  }
  __syncwarp();  // every lane's reads of the stage are done
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float d[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) d[h] = lo_f2(acc[j][h]) + hi_f2(acc[j][h]);
#pragma unroll
    for (int h = 0; h < 4; ++h) d[h] += __shfl_xor_sync(kFull, d[h + 4], 16);
#pragma unroll
    for (int h = 0; h < 2; ++h) d[h] += __shfl_xor_sync(kFull, d[h + 2], 8);
    float t = (d[0] > 0.f ? d[0] : 0.f) + (d[1] > 0.f ? d[1] : 0.f);
    t += __shfl_xor_sync(kFull, t, 8);
    t += __shfl_xor_sync(kFull, t, 16);
    if (hh == 0) myscr[kk + 8 * j] = t;
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
  // queries of the first kQSlots sequences this CTA's pages belong to
  constexpr int QS = (DI / 32) * 64 + 4;
  float* myscr0 = reinterpret_cast<float*>(pref + (a.B + 1 + 3) / 4 * 4);
  float* qcache = myscr0 + kConsumerWarps * 128;
  auto seq_of = [&](long long page) {  // largest b with pref[b] <= page
    int l = 0, h = a.B;
    while (h - l > 1) {
      const int m = (l + h) >> 1;
      if (pref[m] <= page)
        l = m;
      else
        h = m;
    }
    return l;
  };
  const int b_first = seq_of(lo);
  const int nslot = min(kQSlots, seq_of(hi - 1) - b_first + 1);
  if (warp < kConsumerWarps) {  // the consumers fill the query cache; the producer starts streaming meanwhile
    for (int e = tid; e < nslot * QS; e += kConsumerWarps * 32) {  // float4 units: 4*QS floats per sequence
      const int bi = e / QS, w4 = e % QS;
      reinterpret_cast<float4*>(qcache)[e] =
          __ldcg(reinterpret_cast<const float4*>(a.q + static_cast<size_t>(b_first + bi) * kQPerSeq) + w4);
    }
    asm volatile("bar.sync 1, %0;\n" ::"n"(kConsumerWarps * 32) : "memory");
  }

  if (warp == kConsumerWarps) {  // ---- producer: page ids 32 at a time, one TMA per 64-dim half
    int bw = 0;  // sequence of the batch's first page
    bool alive = true;
    long long issued = 0;  // pages whose copies were issued
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
          if (!mbar_wait_bounded(&empty[s], (n & 1) ^ 1, a.waitNs)) {
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
        ++issued;
      }
    }
    // The CTA must not exit while a copy still writes into its ring (consumers
    // that gave up have left): wait, bounded, for the last page of each stage.
    if (lane == 0) {
      for (long long jx = issued - 1; jx >= 0 && jx >= issued - kStages; --jx) {
        const int s = static_cast<int>(jx % kStages), n = static_cast<int>(jx / kStages);
        if (!mbar_wait_bounded(&full[s], n & 1, kWaitLimitNs)) {
          atomicOr(a.status, kErrWaitTimeout);
          break;
        }
      }
    }
    return;
  }

  // ---- consumers: warp w scores pages lo + w, lo + w + kConsumerWarps, ...
  float* myscr = myscr0 + warp * 128;
  const int hh = lane >> 3;
  int cached_b = -1, n_c = 0;
  int b = 0;
  for (long long i = lo + warp; i < hi; i += kConsumerWarps) {
    while (i >= pref[b + 1]) ++b;
    const int p = static_cast<int>(i - pref[b]);
    const int jx = static_cast<int>(i - lo), s = jx % kStages, n = jx / kStages;
    if (b != cached_b) {
      n_c = max(0, min(a.ctx[b], MAXL)) / a.ratio;
      cached_b = b;
    }
    // Warps take pages round-robin, so this warp can reach page jx while the
    // stage's previous page (jx - kStages, another warp's) is still landing;
    // its full phase would then look complete to a parity wait.  Waiting first
    // for that page to be consumed (empty phase n-1) leaves the full barrier
    // exactly one phase short of page jx's, so the parity wait is exact.
    if ((n > 0 && !mbar_wait_bounded(&empty[s], (n - 1) & 1, a.waitNs)) ||
        !mbar_wait_bounded(&full[s], n & 1, a.waitNs)) {
      if (lane == 0) atomicOr(a.status, kErrWaitTimeout);
      break;
    }
    const uint8_t* tile = ring + s * stage_bytes;
    if (b - b_first < kQSlots)
      score_page<DI, true>(tile, bpp, qcache + (b - b_first) * 4 * QS + hh * QS, myscr);
    else
      score_page<DI, false>(tile, bpp, a.q + static_cast<size_t>(b) * kQPerSeq + hh * QS, myscr);
    if (lane == 0) mbar_arrive(&empty[s]);
    __syncwarp();
    page_epilogue(a, b, p, n_c, bpp, myscr[lane < bpp ? lane : 0]);
    __syncwarp();
  }
}

// ------------------------------------------------------------------ B3
struct SelectArgs {
  const int32_t* ctx;
  const float* scores;
  int32_t* hist;
  uint32_t* candKey;  // [B][nbmax]: slice s keeps its candidates at [s*kSliceBlocks, ...), ascending ids
  int32_t* candId;
  int32_t* sliceCnt;  // [B][nsplitmax]
  int32_t* ticket;    // [B], zero between calls
  int32_t* indices;
  int maxPagesPerSeq, ratio, budget, topK, nbmax, nsplitmax;
};

// Bin T holding the budget-th largest score and the count of blocks in higher
// bins, from the sequence's histogram (every thread gets both).
__device__ __forceinline__ void threshold_bin(const int32_t* hrow, int budget, int* scan, int* info, int& T,
                                              int& c_above) {
  constexpr int BPT = kNumBins / kSelThreads;
  const int tid = threadIdx.x;
  int h[BPT];
  int own = 0;
  if (tid == 0) {
    info[0] = 0;
    info[1] = 0;
  }
  const int4* h4 = reinterpret_cast<const int4*>(hrow + tid * BPT);
#pragma unroll
  for (int k = 0; k < BPT / 4; ++k) {
    const int4 v = __ldcg(h4 + k);
    h[4 * k] = v.x;
    h[4 * k + 1] = v.y;
    h[4 * k + 2] = v.z;
    h[4 * k + 3] = v.w;
    own += v.x + v.y + v.z + v.w;
  }
  int total;
  const int excl = cta_exclusive_scan<kSelThreads>(own, scan, total);
  int running = total - excl - own;  // blocks in the bins of higher threads
#pragma unroll
  for (int k = BPT - 1; k >= 0; --k) {
    if (running < budget && running + h[k] >= budget) {
      info[0] = tid * BPT + k;
      info[1] = running;
    }
    running += h[k];
  }
  __syncthreads();
  T = info[0];
  c_above = info[1];
  __syncthreads();
}

// Among the values of a CTA-wide histogram `rh` of `nbins` bins (counts of one
// digit), the digit U such that count(digit > U) < need <= count(digit >= U),
// and count(digit > U).
template <int NBINS>
__device__ __forceinline__ void digit_from_top(const int* rh, int need, int* scan, int* info, int& U, int& above_U) {
  constexpr int PER = NBINS / kSelThreads;
  const int tid = threadIdx.x;
  if (tid == 0) {
    info[2] = 0;
    info[3] = 0;
  }
  int own = 0;
#pragma unroll
  for (int k = 0; k < PER; ++k) own += rh[tid * PER + k];
  int total;
  const int excl = cta_exclusive_scan<kSelThreads>(own, scan, total);
  int running = total - excl - own;
#pragma unroll
  for (int k = PER - 1; k >= 0; --k) {
    const int c = rh[tid * PER + k];
    if (running < need && running + c >= need) {
      info[2] = tid * PER + k;
      info[3] = running;
    }
    running += c;
  }
  __syncthreads();
  U = info[2];
  above_U = info[3];
  __syncthreads();
}

// kRounds: the most slices one CTA filters on its own (kSingleRounds when every
// sequence of the launch has at most that many, so the grid has one CTA per
// sequence; else 1, and longer sequences go through the slice CTAs).
template <int kRounds>
__global__ void __launch_bounds__(kSelThreads) decode_select_kernel(const SelectArgs a) {
  __shared__ int scan[kSelThreads / 32];
  __shared__ int info[8];
  __shared__ int wcnt[kRounds * (kSelThreads / 32)];
  __shared__ int sbase[kMaxSlices + 1];
  __shared__ int rh[1024];
  __shared__ uint32_t ck_s[kStageCand];
  __shared__ int ci_s[kStageCand];
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
  const int nslice = (n_c + kSliceBlocks - 1) / kSliceBlocks;
  // Up to kSingleRounds slices: CTA 0 filters them all (its loads for every
  // round in flight at once) and keeps the candidates in shared memory, so
  // they make no round trip through global memory and no CTA waits on another.
  const bool single = nslice <= kRounds;
  const int nsplit = single ? 1 : nslice;
  if (s >= nsplit) return;
  const int nrounds = single ? nslice : 1;

  // ---- candidates (bin >= T), compacted in ascending id order.  Round r
  // covers blocks g0 + 2048 r + [0, 2048); in it warp w covers 256 w +
  // [0, 256), visited as lane + 32 m.  The score loads are issued before the
  // histogram is read, so the two latencies overlap.
  const float* srow = a.scores + static_cast<size_t>(b) * a.nbmax;
  const int g0 = s * kSliceBlocks;
  constexpr int M = kSliceBlocks / kSelThreads;
  uint32_t keys[kRounds][M];
#pragma unroll
  for (int r = 0; r < kRounds; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const int g = g0 + r * kSliceBlocks + warp * 32 * M + m * 32 + lane;
      keys[r][m] = r < nrounds && g < n_c ? __float_as_uint(__ldcg(srow + g)) : 0u;
    }

  int T, c_above;
  threshold_bin(hrow, a.budget, scan, info, T, c_above);

  // every round's ballots first, then one barrier for all the warp counts
  unsigned cm[kRounds][M];
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    int wc = 0;
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const int g = g0 + r * kSliceBlocks + warp * 32 * M + m * 32 + lane;
      cm[r][m] = __ballot_sync(kFull, r < nrounds && g < n_c && static_cast<int>(keys[r][m] >> kBinShift) >= T);
      wc += __popc(cm[r][m]);
    }
    if (lane == 0) wcnt[r * (kSelThreads / 32) + warp] = wc;
  }
  __syncthreads();
  uint32_t* ckey = a.candKey + static_cast<size_t>(b) * a.nbmax;
  int32_t* cid = a.candId + static_cast<size_t>(b) * a.nbmax;
  const unsigned below = (1u << lane) - 1u;
  int run = 0;  // candidates of the earlier rounds
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    int off = run, tot = 0;
#pragma unroll
    for (int w = 0; w < kSelThreads / 32; ++w) {
      const int c = wcnt[r * (kSelThreads / 32) + w];
      off += w < warp ? c : 0;
      tot += c;
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
      if ((cm[r][m] >> lane) & 1u) {
        const int e = off + __popc(cm[r][m] & below);  // position among this CTA's candidates
        const uint32_t k = keys[r][m];
        const int g = g0 + r * kSliceBlocks + warp * 32 * M + m * 32 + lane;
        ckey[g0 + e] = k;
        cid[g0 + e] = g;
        if (single && e < kStageCand) {
          ck_s[e] = k;
          ci_s[e] = g;
        }
      }
      off += __popc(cm[r][m]);
    }
    run += tot;
  }
  if (single) {
    // candidates past kStageCand are read back from global memory (.cg, at
    // L2) by other threads of this CTA: make the stores visible there first
    if (run > kStageCand) __threadfence();
    if (tid == 0) {
      sbase[0] = 0;
      sbase[kMaxSlices] = run;
    }
    __syncthreads();
  } else {
    if (tid == 0) a.sliceCnt[static_cast<size_t>(b) * a.nsplitmax + s] = run;
    __threadfence();
    __syncthreads();
    if (tid == 0) info[6] = atomicAdd(a.ticket + b, 1) == nsplit - 1;
    __syncthreads();
    if (!info[6]) return;
    __threadfence();

    // ---- last CTA of the sequence: the candidates of all slices, in id order
    constexpr int PER = kMaxSlices / kSelThreads;
    int v[PER], own = 0;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int sl = tid * PER + k;
      v[k] = sl < nsplit ? __ldcg(a.sliceCnt + static_cast<size_t>(b) * a.nsplitmax + sl) : 0;
      own += v[k];
    }
    int total;
    int rs = cta_exclusive_scan<kSelThreads>(own, scan, total);
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      sbase[tid * PER + k] = rs;
      rs += v[k];
    }
    if (tid == 0) sbase[kMaxSlices] = total;
    __syncthreads();
  }
  const int ncand = sbase[kMaxSlices];
  auto locate = [&](int e) {  // flat candidate index -> position in the slice-major arrays
    int lo = 0, hi = nsplit;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (sbase[mid] <= e)
        lo = mid;
      else
        hi = mid;
    }
    return lo * kSliceBlocks + (e - sbase[lo]);
  };
  const bool staged = ncand <= kStageCand;
  if (staged && !single) {  // four candidates per thread per pass, their loads in flight together
    for (int e0 = tid; e0 < ncand; e0 += 4 * kSelThreads) {
      uint32_t kk[4];
      int ii[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * kSelThreads;
        const int at = e < ncand ? locate(e) : 0;
        kk[u] = e < ncand ? __ldcg(ckey + at) : 0u;
        ii[u] = e < ncand ? __ldcg(cid + at) : 0;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * kSelThreads;
        if (e < ncand) {
          ck_s[e] = kk[u];
          ci_s[e] = ii[u];
        }
      }
    }
    __syncthreads();
  }
  auto key_at = [&](int e) { return staged ? ck_s[e] : __ldcg(ckey + locate(e)); };
  auto id_at = [&](int e) { return staged ? ci_s[e] : __ldcg(cid + locate(e)); };

  // ---- the cut inside bin T: two radix digits (bits 18..9, then 8..0)
  const int need = a.budget - c_above;  // >= 1 blocks of bin T to keep
  for (int i = tid; i < 1024; i += kSelThreads) rh[i] = 0;
  __syncthreads();
  for (int e = tid; e < ncand; e += kSelThreads) {
    const uint32_t k = key_at(e);
    if (static_cast<int>(k >> kBinShift) == T) atomicAdd(&rh[(k >> 9) & 1023], 1);
  }
  __syncthreads();
  int U, above_U;
  digit_from_top<1024>(rh, need, scan, info, U, above_U);
  for (int i = tid; i < 512; i += kSelThreads) rh[i] = 0;
  __syncthreads();
  const uint32_t hiU = (static_cast<uint32_t>(T) << 10) | static_cast<uint32_t>(U);
  for (int e = tid; e < ncand; e += kSelThreads) {
    const uint32_t k = key_at(e);
    if ((k >> 9) == hiU) atomicAdd(&rh[k & 511], 1);
  }
  __syncthreads();
  int V, above_V;
  digit_from_top<512>(rh, need - above_U, scan, info, V, above_V);
  const uint32_t Tk = (hiU << 9) | static_cast<uint32_t>(V);
  const int n_eq = need - above_U - above_V;  // keys equal to Tk to keep, lowest ids first

  // ---- keep: key > Tk, or key == Tk among the first n_eq such in id order;
  // each thread filters a contiguous run of the (ascending) candidates
  const int C = (ncand + kSelThreads - 1) / kSelThreads;
  const int e0 = min(tid * C, ncand), e1 = min(e0 + C, ncand);
  int ceq = 0;
  for (int e = e0; e < e1; ++e) ceq += key_at(e) == Tk ? 1 : 0;
  int tmp;
  const int eq_before = cta_exclusive_scan<kSelThreads>(ceq, scan, tmp);
  int nk = 0;
  {
    int r = eq_before;
    for (int e = e0; e < e1; ++e) {
      const uint32_t k = key_at(e);
      nk += (k > Tk || (k == Tk && r < n_eq)) ? 1 : 0;
      r += k == Tk ? 1 : 0;
    }
  }
  int kept;
  int pos = cta_exclusive_scan<kSelThreads>(nk, scan, kept);
  {
    int r = eq_before;
    for (int e = e0; e < e1; ++e) {
      const uint32_t k = key_at(e);
      if (k > Tk || (k == Tk && r < n_eq)) {
        const int g = id_at(e);
        if ((pos + 1) * a.ratio <= a.topK)
          for (int j = 0; j < a.ratio; ++j) out[pos * a.ratio + j] = g * a.ratio + j;
        ++pos;
      }
      r += k == Tk ? 1 : 0;
    }
  }
  const int head = min(kept * a.ratio, a.topK);
  for (int i = head + tid; i < a.topK; i += kSelThreads) {
    const int j = n_c * a.ratio + (i - head);
    out[i] = j <= t ? j : -1;
  }
  // re-arm for the next call
  for (int i = tid; i < kNumBins; i += kSelThreads) hrow[i] = 0;
  if (tid == 0) a.ticket[b] = 0;
}

std::atomic<uint64_t> g_wait_limit_ns{0};

}  // namespace

void set_decode_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns, std::memory_order_relaxed); }

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

size_t indexer_decode_workspace_bytes(int B, int maxPagesPerSeq, int ratio, int budget) {
  const int nbmax = maxPagesPerSeq * (kTokensPerPageHost / ratio);
  (void)budget;
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
    decode_prep_kernel<64><<<B, 256 + 64, 0, st>>>(pa);
  else
    decode_prep_kernel<128><<<B, 256 + 128, 0, st>>>(pa);
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
  const uint64_t wl = g_wait_limit_ns.load(std::memory_order_relaxed);
  sa.waitNs = wl ? wl : kWaitLimitNs;
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
  se.candKey = reinterpret_cast<uint32_t*>(ws + l.candKey);
  se.candId = reinterpret_cast<int32_t*>(ws + l.candId);
  se.sliceCnt = reinterpret_cast<int32_t*>(ws + l.sliceCnt);
  se.ticket = reinterpret_cast<int32_t*>(ws + l.ticket);
  se.indices = p.indices;
  se.maxPagesPerSeq = p.maxPagesPerSeq;
  se.ratio = p.compressRatio;
  se.budget = p.budget;
  se.topK = p.topK;
  se.nbmax = nbmax;
  se.nsplitmax = (nbmax + kSliceBlocks - 1) / kSliceBlocks;
  if (se.nsplitmax > kMaxSlices) return cudaErrorInvalidValue;
  if (se.nsplitmax <= kSingleRounds)
    decode_select_kernel<kSingleRounds><<<dim3(1, B), kSelThreads, 0, st>>>(se);
  else
    decode_select_kernel<1><<<dim3(se.nsplitmax, B), kSelThreads, 0, st>>>(se);
  return cudaGetLastError();
}

}  // namespace qsa
