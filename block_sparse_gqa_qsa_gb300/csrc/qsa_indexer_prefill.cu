// qsa_indexer_prefill.cu -- the weight-free QSA indexer over a padded prefill
// batch ("Qsa Attention Plugin", fused step 2; "spark_model/layers/ops/qsa.rs",
// qsa_block_pool / qsa_qprep_rows / qsa_score_rows).
//
// Two kernels:
//   block_pool_kernel      one warp per complete block: mean of r raw keys ->
//                          RMSNorm*(1+w) -> RoPE at the block start, stored
//                          fp16 (RNE) from an exact mean and double-float
//                          arithmetic (qsa_blockkey.cuh), so the fp16 rounding
//                          of every key is the decision an f64 evaluation
//                          takes; the pass is tiny (S/r * di values).
//   prefill_select_kernel  persistent, two CTAs per SM, work items of 8
//                          consecutive rows of one sequence taken from a
//                          counter, longest rows first.  A group whose rows
//                          need a selection (n_c > budget) is scored by the
//                          whole CTA: index-query prep (fp32, angles reduced
//                          in integer turns), block scores on the CUDA cores
//                          (fp32 FMA, a register-tiled contraction of 8 rows x
//                          8 heads against 128-block tiles staged in shared
//                          memory, heads paired in fp32x2 FMAs), the
//                          relu/head sum into the CTA's own score
//                          slot and a 256-bin histogram of the score bits per
//                          row.  Then each warp selects its row: the bin of
//                          the cut from the histogram, radix narrowing of that
//                          bin (over the slot, then over at most 1024 keys
//                          staged in shared memory), exact ties to the lower
//                          block id, and one pass that expands the kept blocks
//                          into the ascending list.  Rows with n_c <= budget
//                          list 0..t and rows t >= L are all -1.  Memory is
//                          linear in S: no row's scores outlive its selection.
#include "qsa_blockkey.cuh"
#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr size_t kStatusBytes = 256;  // head of every indexer workspace: status word

struct PoolArgs {
  const __half* idxK;
  const float* wk;
  const int32_t* ctx;
  __half* kbar;
  int32_t* queue;  // work counter of the select kernel that follows: set to zero here
  int S, nbmax, ratio, rot;
  float eps;
  RopeFreqs rf;
};

template <int DI>
__global__ void __launch_bounds__(256) block_pool_kernel(const PoolArgs a) {
  __shared__ f2x y_s[8][DI];
  __shared__ RopeSmem rs;
  const int warp = threadIdx.x >> 5;
  const int b = blockIdx.y;
  const int g = blockIdx.x * 8 + warp;
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *a.queue = 0;
  stage_rope(a.rf, rs);
  __syncthreads();
  const int L = max(0, min(a.ctx[b], a.S));  // lengths outside [0, S] are clamped, never trusted
  if (g >= L / a.ratio) return;              // complete blocks only; warp-uniform
  const __half* raw = a.idxK + (static_cast<size_t>(b) * a.S + static_cast<size_t>(g) * a.ratio) * DI;
  block_key<DI, 1>([&](int j, int i) { return raw[j * DI + i]; }, a.ratio, a.wk, a.eps, a.rot, g * a.ratio, rs, y_s[warp],
                   nullptr, 0, 0, a.kbar + (static_cast<size_t>(b) * a.nbmax + g) * DI);
}

struct SelArgs {
  const __half* idxQ;
  const float* wq;
  const int32_t* ctx;
  const __half* kbar;
  float* scores;  // [slots][kRows][nbmax]: the block scores of the rows one CTA is selecting
  int32_t* queue; // work counter, set to zero by the pool kernel of the same call
  int32_t* indices;
  int B, S, Hi, nbmax, ratio, rot, budget, topK, ngroups, nitems;
  float eps;
  RopeFreqs rf;
};

constexpr int kRows = kPrefillRowsPerCta;  // rows per work item (one warp each)
constexpr int kThreads = 256;
constexpr int kTile = 128;                  // blocks per score tile (4 per lane)
constexpr int kBPL = kTile / 32;            // blocks per lane
constexpr int kKC = 32;                     // key dims staged per step
constexpr int kKS = kKC + 2;                // padded row stride (17 x 8 bytes): float2 reads are conflict-free
constexpr int kHI = 8;                      // heads per thread tile (Hi <= 8, extra heads are zero)
constexpr int kBins = 256;                  // per-row histogram of the score bits, filled while scoring
constexpr int kBinBase = 123 * 16;          // (bits >> 19) of 2^-4: bin 0 holds smaller scores, bin 255 2^12 and up
constexpr int kCandCap = 1024;              // keys of the cut's range one warp stages in shared memory

// Two fp16 values packed in 32 bits, widened to fp32.
__device__ __forceinline__ float2 bits_to_float2(uint32_t u) {
  __half2_raw r;
  r.x = static_cast<unsigned short>(u & 0xffffu);
  r.y = static_cast<unsigned short>(u >> 16);
  return __half22float2(__half2(r));
}

// Scores are sums of relu terms, so they are +0 or positive and their bits
// order like the values.  Bin b covers one sixteenth of an octave: the
// exponent and top four mantissa bits, over 16 octaves from 2^-4.
__device__ __forceinline__ int score_bin(uint32_t key) {
  return min(max(static_cast<int>(key >> 19) - kBinBase, 0), kBins - 1);
}

template <int DI>
constexpr size_t select_smem_bytes() {
  return sizeof(float) * (static_cast<size_t>(DI) * kRows * kHI + 2 * kTile * kKS + kRows * DI + kRows * 128 +
                          kRows * kBins);
}
static_assert(kRows * kCandCap <= 64 * kRows * kHI + 2 * kTile * kKS, "candidate keys reuse the query and key tiles");

// Index-query prep and block scores of the live rows [t0, t0 + nlive) of
// sequence b against blocks [0, n_hi): each warp owns one row; the rows that
// select (srow != nullptr) write their n_c scores to srow and count them in
// their warp's histogram.  Every thread of the CTA takes part.
template <int DI>
__device__ __noinline__ void score_rows(const SelArgs& a, float* smem, int b, int t0, int nlive, int n_hi,
                                           float* srow, int n_c, uint32_t* hist) {
  float* q_s = smem;                          // [DI][kRows][kHI] prepared queries
  float* kb_s = q_s + DI * kRows * kHI;       // [2][kTile][kKS]  block-key tile (fp32)
  float* ys_s = kb_s + 2 * kTile * kKS;       // [kRows][DI]      per-warp RoPE scratch
  float* cs_s = ys_s + kRows * DI;            // [kRows][64][2]   cos/sin per row
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ------------------------------------------------------------ query prep
  const int half = a.rot >> 1;
  for (int e = tid; e < kRows * half; e += kThreads) {
    const int r = e / half, i = e - r * half;
    float c = 1.f, s = 0.f;
    if (r < nlive) rope_cos_sin_turns(static_cast<unsigned>(t0 + r), a.rf.turn[i], c, s);
    cs_s[r * 128 + 2 * i] = c;
    cs_s[r * 128 + 2 * i + 1] = s;
  }
  __syncthreads();
  {
    constexpr int PER = DI / 32;
    const int r = warp;
    // every head's raw query and the norm weights, loaded before any is used: one round trip, not kHI
    float xv[kHI][PER], wv[PER];
    const __half* xr = a.idxQ + (static_cast<size_t>(b) * a.S + t0 + r) * a.Hi * DI;
#pragma unroll
    for (int p = 0; p < PER; ++p) wv[p] = a.wq[lane + 32 * p];
#pragma unroll
    for (int h = 0; h < kHI; ++h)
#pragma unroll
      for (int p = 0; p < PER; ++p)
        xv[h][p] = r < nlive && h < a.Hi ? __half2float(xr[h * DI + lane + 32 * p]) : 0.f;
#pragma unroll
    for (int h = 0; h < kHI; ++h) {
      if (r < nlive && h < a.Hi) {
        float y[PER];
        float ss = 0.f;
#pragma unroll
        for (int p = 0; p < PER; ++p) {
          y[p] = xv[h][p];
          ss = fmaf(y[p], y[p], ss);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
        const float inv = 1.0f / sqrtf(ss / DI + a.eps);
#pragma unroll
        for (int p = 0; p < PER; ++p) {
          const int i = lane + 32 * p;
          y[p] = y[p] * inv * (1.0f + wv[p]);
          ys_s[r * DI + i] = y[p];
        }
        __syncwarp();
#pragma unroll
        for (int p = 0; p < PER; ++p) {
          const int i = lane + 32 * p;
          float v = y[p];
          if (i < half) {
            v = y[p] * cs_s[r * 128 + 2 * i] - ys_s[r * DI + i + half] * cs_s[r * 128 + 2 * i + 1];
          } else if (i < a.rot) {
            const int k = i - half;
            v = y[p] * cs_s[r * 128 + 2 * k] + ys_s[r * DI + k] * cs_s[r * 128 + 2 * k + 1];
          }
          q_s[(i * kRows + r) * kHI + h] = v;
        }
        __syncwarp();
      } else {
#pragma unroll
        for (int p = 0; p < PER; ++p) q_s[((lane + 32 * p) * kRows + r) * kHI + h] = 0.f;
      }
    }
  }
  __syncthreads();

  // ---------------------------------------------------------- block scores
  // Lane owns blocks lane + 32 m (m < kBPL) of the tile, for its warp's row
  // and all kHI heads: 32 accumulators, each a plain ascending-k FMA chain,
  // so a block's score does not depend on where the block sits in a tile.
  const __half* kb_g = a.kbar + static_cast<size_t>(b) * a.nbmax * DI;
  const int ntiles = (n_hi + kTile - 1) / kTile;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  // the first chunk of each tile is fetched during the previous tile's last chunk
  const uint4* src0 = reinterpret_cast<const uint4*>(kb_g + static_cast<size_t>(tid >> 1) * DI) + 2 * (tid & 1);
  uint4 pre0 = (tid >> 1) < n_hi ? __ldg(src0) : zero;
  uint4 pre1 = (tid >> 1) < n_hi ? __ldg(src0 + 1) : zero;
  for (int tile = 0; tile < ntiles; ++tile) {
    const int gbase = tile * kTile;
    const int gl = gbase + (tid >> 1);  // block this thread stages 8 dims (half a chunk) of
    const bool gok = gl < n_hi;
    const uint4* src = reinterpret_cast<const uint4*>(kb_g + static_cast<size_t>(gok ? gl : 0) * DI) + 2 * (tid & 1);
    const int gn = gl + kTile;  // this thread's block of the next tile
    const bool nok = tile + 1 < ntiles && gn < n_hi;
    const uint4* nsrc = reinterpret_cast<const uint4*>(kb_g + static_cast<size_t>(nok ? gn : 0) * DI) + 2 * (tid & 1);
    uint64_t acc[kBPL][kHI / 2];  // heads (2j, 2j+1) of block lane + 32 m as one fp32 pair
#pragma unroll
    for (int m = 0; m < kBPL; ++m)
#pragma unroll
      for (int j = 0; j < kHI / 2; ++j) acc[m][j] = 0ull;

#pragma unroll 1
    for (int kc = 0; kc < DI / kKC; ++kc) {
      float2* dst = reinterpret_cast<float2*>(kb_s + (kc & 1) * kTile * kKS + (tid >> 1) * kKS + (tid & 1) * 16);
      dst[0] = bits_to_float2(pre0.x);
      dst[1] = bits_to_float2(pre0.y);
      dst[2] = bits_to_float2(pre0.z);
      dst[3] = bits_to_float2(pre0.w);
      dst[4] = bits_to_float2(pre1.x);
      dst[5] = bits_to_float2(pre1.y);
      dst[6] = bits_to_float2(pre1.z);
      dst[7] = bits_to_float2(pre1.w);
      __syncthreads();
      if (kc + 1 < DI / kKC) {
        pre0 = gok ? __ldg(src + 4 * (kc + 1)) : zero;
        pre1 = gok ? __ldg(src + 4 * (kc + 1) + 1) : zero;
      } else {
        pre0 = nok ? __ldg(nsrc) : zero;
        pre1 = nok ? __ldg(nsrc + 1) : zero;
      }
      const float* kt = kb_s + (kc & 1) * kTile * kKS;
      const float* qk = q_s + static_cast<size_t>(kc * kKC) * kRows * kHI + warp * kHI;
#pragma unroll  // the whole chunk: loads of later dims in flight while earlier ones multiply
      for (int kp = 0; kp < kKC / 2; ++kp) {  // two dims per step: 16 key values, 16 query values, 128 FMAs in 64 pair FMAs
        float2 kv[kBPL];
#pragma unroll
        for (int m = 0; m < kBPL; ++m) kv[m] = *reinterpret_cast<const float2*>(kt + (lane + 32 * m) * kKS + kp * 2);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          // the 8 heads' query values as 4 fp32 pairs; each pair FMA is two independent fp32 FMAs,
          // so every accumulator stays the plain ascending-k chain
          const ulonglong2* qp = reinterpret_cast<const ulonglong2*>(qk + (kp * 2 + kk) * kRows * kHI);
          const ulonglong2 qa = qp[0], qb = qp[1];
#pragma unroll
          for (int m = 0; m < kBPL; ++m) {
            const float kval = kk == 0 ? kv[m].x : kv[m].y;
            const uint64_t k2 = pack_f2(kval, kval);
            acc[m][0] = ffma2(qa.x, k2, acc[m][0]);
            acc[m][1] = ffma2(qa.y, k2, acc[m][1]);
            acc[m][2] = ffma2(qb.x, k2, acc[m][2]);
            acc[m][3] = ffma2(qb.y, k2, acc[m][3]);
          }
        }
      }
    }
    if (srow) {
#pragma unroll
      for (int m = 0; m < kBPL; ++m) {
        const int g = gbase + lane + 32 * m;
        if (g < n_c) {
          float sc = 0.f;
#pragma unroll
          for (int j = 0; j < kHI / 2; ++j) {
            const float h0 = lo_f2(acc[m][j]), h1 = hi_f2(acc[m][j]);
            sc += h0 > 0.f ? h0 : 0.f;
            sc += h1 > 0.f ? h1 : 0.f;
          }
          srow[g] = sc;  // read back later by this same lane only
          atomicAdd(hist + score_bin(__float_as_uint(sc)), 1u);
        }
      }
    }
  }
}

// The bin holding the need-th largest key of a warp's 256-bin histogram
// (lane l owns bins 8l .. 8l+7): T, the count of keys in higher bins, and the
// count in bin T.  Every lane gets all three; need must not exceed the total.
__device__ __forceinline__ void find_bin(const uint32_t* hist, int need, int& T, int& above, int& nT) {
  const int lane = threadIdx.x & 31;
  const uint4 h0 = *reinterpret_cast<const uint4*>(hist + lane * 8);
  const uint4 h1 = *reinterpret_cast<const uint4*>(hist + lane * 8 + 4);
  const int hb[8] = {static_cast<int>(h0.x), static_cast<int>(h0.y), static_cast<int>(h0.z), static_cast<int>(h0.w),
                     static_cast<int>(h1.x), static_cast<int>(h1.y), static_cast<int>(h1.z), static_cast<int>(h1.w)};
  int own = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) own += hb[j];
  int suffix = own;  // keys in the bins of lanes >= this one
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_down_sync(kFull, suffix, o);
    if (lane + o < 32) suffix += y;
  }
  int run = suffix - own, t = -1, ab = 0, n = 0;
#pragma unroll
  for (int j = 7; j >= 0; --j) {
    if (run < need && run + hb[j] >= need) {
      t = lane * 8 + j;
      ab = run;
      n = hb[j];
    }
    run += hb[j];
  }
  const int src = __ffs(__ballot_sync(kFull, t >= 0)) - 1;  // exactly one lane holds the bin
  T = __shfl_sync(kFull, t, src);
  above = __shfl_sync(kFull, ab, src);
  nT = __shfl_sync(kFull, n, src);
}

// Keys of one row for the radix narrowing: the row's n_c scores in global
// memory (each lane reads back only the blocks it wrote, g = lane mod 32), or
// the warp's staged candidates in shared memory.
struct GlobalKeys {
  const float* srow;
  int n;
  template <class F>
  __device__ __forceinline__ void each(F&& f) const {
    const int lane = threadIdx.x & 31;
    constexpr int U = 16;
    for (int g0 = 0; g0 < n; g0 += 32 * U) {
      uint32_t k[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int g = g0 + 32 * u + lane;
        k[u] = g < n ? __float_as_uint(srow[g]) : 0u;
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (g0 + 32 * u + lane < n) f(k[u]);
    }
  }
};
struct SharedKeys {
  const uint32_t* keys;
  int n;
  template <class F>
  __device__ __forceinline__ void each(F&& f) const {
    for (int i = threadIdx.x & 31; i < n; i += 32) f(keys[i]);
  }
};

// Narrows the key range [blo, blo + span], which holds nT keys of which the
// `need` largest are kept, through 256-bin histograms of (key - blo) >> sh in
// the warp's shared memory, until it holds at most `limit` keys or one value.
template <class Keys>
__device__ __forceinline__ void narrow(const Keys& keys, uint32_t* hist, uint32_t& blo, uint32_t& span, int& need,
                                       int& nT, int limit) {
  const int lane = threadIdx.x & 31;
  while (nT > limit && span != 0u) {
    const int sh = max(0, 24 - static_cast<int>(__clz(span)));  // span >> sh < 256
#pragma unroll
    for (int j = 0; j < 8; ++j) hist[lane * 8 + j] = 0u;
    __syncwarp();
    const uint32_t lo = blo, sp = span;
    keys.each([&](uint32_t k) {
      const uint32_t d = k - lo;  // keys below lo wrap past span
      if (d <= sp) atomicAdd(hist + (d >> sh), 1u);
    });
    __syncwarp();
    int T, above, n;
    find_bin(hist, need, T, above, n);
    need -= above;
    nT = n;
    blo += static_cast<uint32_t>(T) << sh;
    span = sh == 0 ? 0u : min(span - (static_cast<uint32_t>(T) << sh), (1u << sh) - 1u);
    __syncwarp();  // every lane has read the histogram
  }
}

// Row t of sequence b, whose n_c > budget scores sit in srow and are counted
// in hist: the cut key and how many keys equal to it are kept (lowest ids
// first), so that the kept set is the top `budget` by (score desc, id asc).
__device__ __forceinline__ void row_cut(const float* srow, int n_c, int budget, uint32_t* hist, uint32_t* cand,
                                        uint32_t& cut, int& quota) {
  const int lane = threadIdx.x & 31;
  const unsigned below = (1u << lane) - 1u;
  int T, above, nT;
  find_bin(hist, budget, T, above, nT);
  int need = budget - above;
  // bin T as a key range; the end bins are open
  uint32_t blo = T == 0 ? 0u : static_cast<uint32_t>(T + kBinBase) << 19;
  uint32_t span = T == kBins - 1 ? 0xffffffffu - blo : (static_cast<uint32_t>(T + kBinBase + 1) << 19) - 1u - blo;
  __syncwarp();  // the histogram is read; narrowing reuses it
  const GlobalKeys gk{srow, n_c};
  narrow(gk, hist, blo, span, need, nT, kCandCap);
  if (span == 0u) {
    cut = blo;
    quota = need;
    return;
  }
  // stage the range's nT <= kCandCap keys, then narrow in shared memory
  {
    int at = 0;
    constexpr int U = 16;
    for (int g0 = 0; g0 < n_c; g0 += 32 * U) {
      uint32_t k[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int g = g0 + 32 * u + lane;
        k[u] = g < n_c ? __float_as_uint(srow[g]) : 0u;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const bool in = g0 + 32 * u + lane < n_c && k[u] - blo <= span;
        const unsigned m = __ballot_sync(kFull, in);
        const int e = at + __popc(m & below);
        if (in && e < kCandCap) cand[e] = k[u];
        at += __popc(m);
      }
    }
    __syncwarp();
  }
  const SharedKeys sk{cand, min(nT, kCandCap)};
  narrow(sk, hist, blo, span, need, nT, 32);
  if (span == 0u) {
    cut = blo;
    quota = need;
    return;
  }
  // at most 32 keys left in range: one per lane, then each one's count of larger and equal keys
  uint32_t* last = hist;
  {
    int at = 0;
    for (int i0 = 0; i0 < sk.n; i0 += 32) {
      const int i = i0 + lane;
      const uint32_t k = i < sk.n ? cand[i] : 0u;
      const bool in = i < sk.n && k - blo <= span;
      const unsigned m = __ballot_sync(kFull, in);
      const int e = at + __popc(m & below);
      if (in && e < 32) last[e] = k;
      at += __popc(m);
    }
  }
  __syncwarp();
  nT = min(nT, 32);
  const uint32_t mine = lane < nT ? last[lane] : 0u;
  int gt = 0, eq = 0;
  for (int j = 0; j < nT; ++j) {
    const uint32_t v = __shfl_sync(kFull, mine, j);
    gt += v > mine ? 1 : 0;
    eq += v == mine ? 1 : 0;
  }
  const int hit = __ffs(__ballot_sync(kFull, lane < nT && gt < need && need <= gt + eq)) - 1;
  cut = __shfl_sync(kFull, mine, hit);
  quota = need - __shfl_sync(kFull, gt, hit);
  __syncwarp();
}

// Writes row t's list: all -1 for t >= L; 0..t when every complete block is
// kept; else the kept blocks in ascending order (from srow, cut, quota), each
// expanded to its r token ids, then the causal tail r*n_c .. t, then -1.
template <int R>
__device__ __forceinline__ void write_row(const SelArgs& a, int32_t* out, int t, int L, const float* srow, uint32_t cut,
                                          int quota) {
  const int ratio = R > 0 ? R : a.ratio;
  const int lane = threadIdx.x & 31;
  if (t >= L) {
    for (int i = lane; i < a.topK; i += 32) out[i] = -1;
    return;
  }
  const int n_c = (t + 1) / ratio;
  if (n_c <= a.budget) {  // every block kept: the row lists 0..t
    for (int i = lane; i < a.topK; i += 32) out[i] = i <= t ? i : -1;
    return;
  }
  const unsigned below = (1u << lane) - 1u;
  int pos = 0;
  constexpr int U = 16;
  for (int g0 = 0; g0 < n_c; g0 += 32 * U) {
    uint32_t k[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int g = g0 + 32 * u + lane;
      k[u] = g < n_c ? __float_as_uint(srow[g]) : 0u;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int g = g0 + 32 * u + lane;
      const bool valid = g < n_c;
      const bool eq = valid && k[u] == cut;
      const unsigned eqm = __ballot_sync(kFull, eq);
      const bool take = valid && (k[u] > cut || (eq && __popc(eqm & below) < quota));
      quota = max(0, quota - __popc(eqm));
      const unsigned tm = __ballot_sync(kFull, take);
      if (take && (pos + __popc(tm & below) + 1) * ratio <= a.topK) {  // the row holds budget * r <= topK
        const int at = (pos + __popc(tm & below)) * ratio;
        if (R > 0) {
#pragma unroll
          for (int j = 0; j < (R > 0 ? R : 1); ++j) out[at + j] = g * ratio + j;
        } else {
          for (int j = 0; j < ratio; ++j) out[at + j] = g * ratio + j;
        }
      }
      pos += __popc(tm);
    }
  }
  const int head = min(pos * ratio, a.topK);
  for (int i = head + lane; i < a.topK; i += 32) {
    const int j = n_c * ratio + (i - head);
    out[i] = j <= t ? j : -1;
  }
}

// Persistent: CTAs take work items from a counter.  Item i is the group of 8
// rows t0 .. t0+7 of sequence i mod B, t0 = 8 * (ngroups - 1 - i / B): the
// groups of every sequence from the last rows down, so the longest rows start
// first and the run ends on rows that only write lists.  Each warp owns one
// row of the group.  A group whose last live row sees more than `budget`
// complete blocks is scored by the whole CTA (query prep, then the register
// tiled contraction against 128-block tiles of fp32 keys staged in shared
// memory); each selecting row's scores go to the CTA's own slot of the
// workspace and into its warp's 256-bin histogram.  Each warp then finds its
// row's cut (the bin from the histogram, then narrowing passes over the
// scores, the last ones on at most kCandCap keys staged in shared memory)
// and writes its list in one more pass.  Two CTAs share an SM, so one's
// selection and list writes overlap the other's scoring.
template <int DI, int R>
__global__ void __launch_bounds__(kThreads, 2) prefill_select_kernel(const SelArgs a) {
  extern __shared__ __align__(16) float smem[];
  __shared__ int item_s[2];
  float* kb_s = smem + DI * kRows * kHI;
  uint32_t* hist_s = reinterpret_cast<uint32_t*>(kb_s + 2 * kTile * kKS + kRows * DI + kRows * 128);
  const int ratio = R > 0 ? R : a.ratio;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t* hist = hist_s + warp * kBins;
  uint32_t* cand = reinterpret_cast<uint32_t*>(smem) + warp * kCandCap;  // query and key tiles, free once scored
  float* srow = a.scores + (static_cast<size_t>(blockIdx.x) * kRows + warp) * a.nbmax;
  if (tid == 0) item_s[0] = atomicAdd(a.queue, 1);
  __syncthreads();
  for (int it = 0;; ++it) {
    const int item = item_s[it & 1];
    if (item >= a.nitems) break;
    int nxt = 0;
    if (tid == 0) nxt = atomicAdd(a.queue, 1);  // the next item, waited for only at the end
    const int pos = item / a.B, b = item - pos * a.B;
    const int t0 = (a.ngroups - 1 - pos) * kRows;
    const int L = max(0, min(__ldg(a.ctx + b), a.S));
    const int nlive = max(0, min(t0 + kRows, L) - t0);
    const int n_hi = (t0 + nlive) / ratio;  // complete blocks seen by the group's last live row
    const int t = t0 + warp;
    const int n_c = (t + 1) / ratio;
    const bool selects = warp < nlive && n_c > a.budget;
    uint32_t cut = 0u;
    int quota = 0;
    if (nlive > 0 && n_hi > a.budget) {  // uniform over the CTA
#pragma unroll
      for (int j = 0; j < kBins / 32; ++j) hist[lane * (kBins / 32) + j] = 0u;
      score_rows<DI>(a, smem, b, t0, nlive, n_hi, selects ? srow : nullptr, n_c, hist);
      __syncthreads();  // the query and key tiles are free: they hold the candidate keys from here on
      if (selects) row_cut(srow, n_c, a.budget, hist, cand, cut, quota);
    }
    if (t < a.S) write_row<R>(a, a.indices + (static_cast<size_t>(b) * a.S + t) * a.topK, t, L, srow, cut, quota);
    if (tid == 0) item_s[(it + 1) & 1] = nxt;
    __syncthreads();
  }
}

template <int DI>
cudaError_t launch_select(const SelArgs& a, cudaStream_t st) {
  constexpr size_t smem = select_smem_bytes<DI>();
  cudaError_t e = cudaSuccess;
  if (a.ratio == 4) {
    static const cudaError_t attr = cudaFuncSetAttribute(
        prefill_select_kernel<DI, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    e = attr;
  } else {
    static const cudaError_t attr = cudaFuncSetAttribute(
        prefill_select_kernel<DI, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    e = attr;
  }
  if (e != cudaSuccess) return e;
  const int grid = min(min(kPrefillScoreSlots, 2 * sm_count()), a.nitems);
  if (a.ratio == 4)
    prefill_select_kernel<DI, 4><<<grid, kThreads, smem, st>>>(a);
  else
    prefill_select_kernel<DI, 0><<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

// ------------------------------------------------ prefill -> decode hand-off
struct HandoffArgs {
  const __half* idxK;
  const int32_t* ctx;
  const __half* kbar;
  int32_t* status;
  __half* pool;
  const int32_t* pageTable;
  int S, nbmax, ratio, Hkv, D, poolHeadDim, numFlatPages, maxPagesPerSeq;
};

// One warp per item of a sequence: items g < n_c copy block g's key into the
// V-row tail of token r*g; item n_c copies the raw keys of the trailing
// incomplete block into their K-row tails.  16-byte copies.
template <int DI>
__global__ void __launch_bounds__(256) handoff_kernel(const HandoffArgs a) {
  constexpr int CH = DI / 8;  // 16-byte chunks of a key
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.y;
  const int g = blockIdx.x * 8 + warp;
  const int L = max(0, min(a.ctx[b], min(a.S, a.maxPagesPerSeq * kTokensPerPageHost)));
  const int n_c = L / a.ratio;
  if (g > n_c) return;
  const int32_t* ptK = a.pageTable + static_cast<size_t>(b) * 2 * a.maxPagesPerSeq;
  const int32_t* ptV = ptK + a.maxPagesPerSeq;
  auto tail_row = [&](int page, int tok) {
    return a.pool + ((static_cast<size_t>(page) * kTokensPerPageHost + (tok & 127)) * a.Hkv) * a.poolHeadDim + a.D;
  };
  if (g < n_c) {
    const int tok = g * a.ratio;
    const int vp = __ldg(ptV + (tok >> 7));
    if (static_cast<unsigned>(vp) >= static_cast<unsigned>(a.numFlatPages)) {
      if (lane == 0) atomicOr(a.status, kErrBadPage);
      return;
    }
    const uint4* src = reinterpret_cast<const uint4*>(a.kbar + (static_cast<size_t>(b) * a.nbmax + g) * DI);
    uint4* dst = reinterpret_cast<uint4*>(tail_row(vp, tok));
    if (lane < CH) dst[lane] = __ldg(src + lane);
    return;
  }
  // g == n_c: raw keys of tokens r*n_c .. L-1
  for (int e = lane; e < (L - n_c * a.ratio) * CH; e += 32) {
    const int tok = n_c * a.ratio + e / CH, c = e % CH;
    const int kp = __ldg(ptK + (tok >> 7));
    if (static_cast<unsigned>(kp) >= static_cast<unsigned>(a.numFlatPages)) {
      atomicOr(a.status, kErrBadPage);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(a.idxK + (static_cast<size_t>(b) * a.S + tok) * DI);
    reinterpret_cast<uint4*>(tail_row(kp, tok))[c] = __ldg(src + c);
  }
}

// Workspace: status word, block keys fp16 [B][S/r][di], the select kernel's
// work counter, then one score slot per select CTA: fp32 [kRows][S/r], the
// scores of the rows that CTA is selecting.  Linear in S, independent of B.
size_t kbar_region_bytes(int B, int S, int di, int ratio) {
  return (static_cast<size_t>(B) * (S / ratio) * di * sizeof(__half) + 255) / 256 * 256;
}
constexpr size_t kQueueBytes = 256;
size_t indexer_prefill_workspace_bytes(int B, int S, int di, int ratio) {
  return kStatusBytes + kbar_region_bytes(B, S, di, ratio) + kQueueBytes +
         static_cast<size_t>(kPrefillScoreSlots) * kRows * static_cast<size_t>(S / ratio) * sizeof(float);
}

cudaError_t launch_indexer_prefill(const QsaIndexerPrefillParams& p, const RopeFreqs& rf) {
  cudaStream_t st = static_cast<cudaStream_t>(p.stream);
  const int nbmax = p.seqLen / p.compressRatio;
  char* ws = static_cast<char*>(p.workspace);
  __half* kbar = reinterpret_cast<__half*>(ws + kStatusBytes);
  const size_t kb_bytes = kbar_region_bytes(p.batchSize, p.seqLen, p.headDim, p.compressRatio);
  int32_t* queue = reinterpret_cast<int32_t*>(ws + kStatusBytes + kb_bytes);
  {  // always launched: it also zeroes the select kernel's work counter
    PoolArgs pa;
    pa.idxK = static_cast<const __half*>(p.idxK);
    pa.wk = p.kNormW;
    pa.ctx = p.contextLengths;
    pa.kbar = kbar;
    pa.queue = queue;
    pa.S = p.seqLen;
    pa.nbmax = nbmax;
    pa.ratio = p.compressRatio;
    pa.rot = p.rotDim;
    pa.eps = p.rmsNormEps;
    pa.rf = rf;
    dim3 grid(max(1, (nbmax + 7) / 8), p.batchSize);
    if (p.headDim == 64)
      block_pool_kernel<64><<<grid, 256, 0, st>>>(pa);
    else
      block_pool_kernel<128><<<grid, 256, 0, st>>>(pa);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  SelArgs sa;
  sa.idxQ = static_cast<const __half*>(p.idxQ);
  sa.wq = p.qNormW;
  sa.ctx = p.contextLengths;
  sa.kbar = kbar;
  sa.scores = reinterpret_cast<float*>(ws + kStatusBytes + kb_bytes + kQueueBytes);
  sa.queue = queue;
  sa.indices = p.indices;
  sa.B = p.batchSize;
  sa.S = p.seqLen;
  sa.Hi = p.numHeads;
  sa.nbmax = nbmax;
  sa.ratio = p.compressRatio;
  sa.rot = p.rotDim;
  sa.budget = p.budget;
  sa.topK = p.topK;
  sa.ngroups = (p.seqLen + kRows - 1) / kRows;
  sa.nitems = sa.ngroups * p.batchSize;
  sa.eps = p.rmsNormEps;
  sa.rf = rf;
  return p.headDim == 64 ? launch_select<64>(sa, st) : launch_select<128>(sa, st);
}

cudaError_t launch_indexer_handoff(const QsaIndexerHandoffParams& p) {
  HandoffArgs a;
  a.idxK = static_cast<const __half*>(p.idxK);
  a.ctx = p.contextLengths;
  a.kbar = reinterpret_cast<const __half*>(static_cast<const char*>(p.workspace) + kStatusBytes);
  a.status = static_cast<int32_t*>(p.workspace);
  a.pool = static_cast<__half*>(p.kvPool);
  a.pageTable = p.pageTable;
  a.S = p.seqLen;
  a.nbmax = p.seqLen / p.compressRatio;
  a.ratio = p.compressRatio;
  a.Hkv = p.numKVHeads;
  a.D = p.kvHeadDim;
  a.poolHeadDim = p.poolHeadDim;
  a.numFlatPages = p.numFlatPages;
  a.maxPagesPerSeq = p.maxPagesPerSeq;
  dim3 grid((a.nbmax + 1 + 7) / 8, p.batchSize);  // items 0..nbmax (the last one: the raw tail)
  cudaStream_t st = static_cast<cudaStream_t>(p.stream);
  if (p.headDim == 64)
    handoff_kernel<64><<<grid, 256, 0, st>>>(a);
  else
    handoff_kernel<128><<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace qsa
