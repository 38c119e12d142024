// qsa_indexer_prefill.cu -- the weight-free QSA indexer over a padded prefill
// batch ("Qsa Attention Plugin", fused step 2; "spark_model/layers/ops/qsa.rs",
// qsa_block_pool / qsa_qprep_rows / qsa_score_rows).
//
// Three kernels:
//   block_pool_kernel      one warp per complete block: mean of r raw keys ->
//                          RMSNorm*(1+w) -> RoPE at the block start, stored
//                          fp16 (RNE) from an exact mean and double-float
//                          arithmetic (qsa_blockkey.cuh), so the fp16 rounding
//                          of every key is the decision an f64 evaluation
//                          takes; the pass is tiny (S/r * di values).
//   prefill_score_kernel   one CTA per 8 consecutive query rows of one
//                          sequence whose rows need a selection (n_c > budget):
//                          index-query prep (fp32, angles reduced in integer
//                          turns), block scores on the CUDA cores (fp32 FMA, a
//                          register-tiled contraction of 8 rows x 8 heads
//                          against 256-block tiles staged in shared memory),
//                          the relu/head sum, written to the workspace (each
//                          row's n_c scores, rows packed back to back).  Two
//                          CTAs share an SM.
//   prefill_topk_kernel    one warp per row: a deterministic top-`budget`
//                          select over the row's scores (a radix select on
//                          the score bits in per-warp histograms, exact ties
//                          to the lower block id) and the expansion into the row's
//                          ascending index list; rows with n_c <= budget list
//                          0..t and rows t >= L are all -1.
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
  float* scores;  // [B][tri_offset(S)]: row t's n_c(t) scores at tri_offset(t)
  int32_t* indices;
  int S, Hi, nbmax, ratio, rot, budget, topK;
  long long triPerSeq;
  float eps;
  RopeFreqs rf;
};

constexpr int kRows = kPrefillRowsPerCta;  // rows per CTA (one warp each)
constexpr int kThreads = 256;
constexpr int kTile = 256;                  // blocks per score tile (8 per lane)
constexpr int kKC = 16;                     // key dims staged per step
constexpr int kKS = kKC + 2;                // padded row stride: float2 reads and writes are conflict-free
constexpr int kHI = 8;                      // heads per thread tile (Hi <= 8, extra heads are zero)

// Two fp16 values packed in 32 bits, widened to fp32.
__device__ __forceinline__ float2 bits_to_float2(uint32_t u) {
  __half2_raw r;
  r.x = static_cast<unsigned short>(u & 0xffffu);
  r.y = static_cast<unsigned short>(u >> 16);
  return __half22float2(__half2(r));
}

// Start of row t's scores within its sequence: sum over u = 1..t of floor(u / r),
// i.e. the complete-block counts n_c of rows 0..t-1.
__host__ __device__ __forceinline__ long long tri_offset(long long t, int r) {
  const long long k = t / r;
  return r * k * (k - 1) / 2 + k * (t - k * r + 1);
}

template <int DI>
constexpr size_t score_smem_bytes() {
  return sizeof(float) * (static_cast<size_t>(DI) * kRows * kHI + 2 * kTile * kKS + kRows * DI + kRows * 128);
}

// Block scores of 8 consecutive query rows of one sequence (rows whose n_c
// exceeds the budget; the others need no scores), written to the workspace.
// Two CTAs share an SM (80 KB of shared memory each at di = 128), so the
// staging barriers and shared-memory latencies of one are covered by the other.
template <int DI>
__global__ void __launch_bounds__(kThreads, 2) prefill_score_kernel(const SelArgs a) {
  extern __shared__ __align__(16) float smem[];
  float* q_s = smem;                          // [DI][kRows][kHI] prepared queries
  float* kb_s = q_s + DI * kRows * kHI;       // [2][kTile][kKS]  block-key tile (fp32)
  float* ys_s = kb_s + 2 * kTile * kKS;       // [kRows][DI]      per-warp RoPE scratch
  float* cs_s = ys_s + kRows * DI;            // [kRows][64][2]   cos/sin per row

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.y;
  const int ngroups = (a.S + kRows - 1) / kRows;
  const int t0 = (ngroups - 1 - static_cast<int>(blockIdx.x)) * kRows;  // longest rows first
  const int L = max(0, min(a.ctx[b], a.S));
  const int t_end = min(t0 + kRows, L);  // live rows [t0, t_end)
  if (t0 >= L) return;
  const int nlive = t_end - t0;
  const int n_hi = t_end / a.ratio;  // complete blocks seen by the group's last live row
  if (n_hi <= a.budget) return;

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
    for (int h = 0; h < kHI; ++h) {
      if (r < nlive && h < a.Hi) {
        const __half* x = a.idxQ + ((static_cast<size_t>(b) * a.S + t0 + r) * a.Hi + h) * DI;
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
  // Lane owns blocks lane + 32 m (m < 8) of the tile, for its warp's row
  // and all kHI heads: 64 accumulators, each a plain ascending-k FMA chain,
  // so a block's score does not depend on where the block sits in a tile.
  const int t = t0 + warp;
  const int n_c = (t + 1) / a.ratio;
  const bool store = warp < nlive && n_c > a.budget;  // this row needs its scores
  float* srow = a.scores + static_cast<size_t>(b) * a.triPerSeq + tri_offset(t, a.ratio);
  const __half* kb_g = a.kbar + static_cast<size_t>(b) * a.nbmax * DI;
  const int ntiles = (n_hi + kTile - 1) / kTile;
  for (int tile = 0; tile < ntiles; ++tile) {
    const int gbase = tile * kTile;
    const int gl = gbase + tid;  // block staged by this thread
    const bool gok = gl < n_hi;
    const uint4* src = reinterpret_cast<const uint4*>(kb_g + static_cast<size_t>(gok ? gl : 0) * DI);
    const uint4 zero = make_uint4(0, 0, 0, 0);
    uint4 pre0 = gok ? __ldg(src) : zero;
    uint4 pre1 = gok ? __ldg(src + 1) : zero;
    float acc[8][kHI];
#pragma unroll
    for (int m = 0; m < 8; ++m)
#pragma unroll
      for (int h = 0; h < kHI; ++h) acc[m][h] = 0.f;

#pragma unroll 1
    for (int kc = 0; kc < DI / kKC; ++kc) {
      float2* dst = reinterpret_cast<float2*>(kb_s + (kc & 1) * kTile * kKS + tid * kKS);
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
        pre0 = gok ? __ldg(src + 2 * (kc + 1)) : zero;
        pre1 = gok ? __ldg(src + 2 * (kc + 1) + 1) : zero;
      }
      const float* kt = kb_s + (kc & 1) * kTile * kKS;
      const float* qk = q_s + static_cast<size_t>(kc * kKC) * kRows * kHI + warp * kHI;
#pragma unroll 4
      for (int kp = 0; kp < kKC / 2; ++kp) {  // two dims per step: 16 key values, 16 query values, 128 FMAs
        float2 kv[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) kv[m] = *reinterpret_cast<const float2*>(kt + (lane + 32 * m) * kKS + kp * 2);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const float* qp = qk + (kp * 2 + kk) * kRows * kHI;
          const float4 qa = *reinterpret_cast<const float4*>(qp);
          const float4 qb = *reinterpret_cast<const float4*>(qp + 4);
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            const float kval = kk == 0 ? kv[m].x : kv[m].y;
            acc[m][0] = fmaf(qa.x, kval, acc[m][0]);
            acc[m][1] = fmaf(qa.y, kval, acc[m][1]);
            acc[m][2] = fmaf(qa.z, kval, acc[m][2]);
            acc[m][3] = fmaf(qa.w, kval, acc[m][3]);
            acc[m][4] = fmaf(qb.x, kval, acc[m][4]);
            acc[m][5] = fmaf(qb.y, kval, acc[m][5]);
            acc[m][6] = fmaf(qb.z, kval, acc[m][6]);
            acc[m][7] = fmaf(qb.w, kval, acc[m][7]);
          }
        }
      }
    }
    if (store) {
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int g = gbase + lane + 32 * m;
        if (g < n_c) {
          float sc = 0.f;
#pragma unroll
          for (int h = 0; h < kHI; ++h) sc += acc[m][h] > 0.f ? acc[m][h] : 0.f;
          srow[g] = sc;
        }
      }
    }
  }
}

// ------------------------------------ select + expand, one warp per row
// Lane l holds the scores of blocks l + 32 m.  Keys are the score bits + 1
// (order-preserving for scores >= 0; 0 marks blocks past the row's n_c).
// A radix select finds the cut T with count(key > T) < budget <=
// count(key >= T): 8-bit digits of (key - lo) over the range still in play,
// counted in a per-warp shared-memory histogram, narrow the range to the bin
// holding the cut (at most four passes), and once that bin holds at most 32
// keys their exact order is taken by pairwise counts.  The blocks above T are
// kept, and of those equal to T the lowest ids, so the kept set is the top
// `budget` by (score desc, id asc).  Walking m upwards visits ids in ascending
// order, so ballots compact the kept blocks straight into the ascending list.
// Rows t >= L are all -1 and rows with n_c <= budget list 0..t.  R: the
// compress ratio fixed at compile time (the r token ids of a kept block are
// then straight-line stores), or 0 to read it from the arguments.
template <int VPT, int R>
__global__ void __launch_bounds__(kThreads) prefill_topk_kernel(const SelArgs a) {
  constexpr int KPL = kThreads * VPT / 32;
  const int ratio = R > 0 ? R : a.ratio;
  __shared__ __align__(16) uint32_t hist_s[kThreads / 32][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.y;
  const int t = blockIdx.x * kRows + warp;
  if (t >= a.S) return;
  const int L = max(0, min(a.ctx[b], a.S));
  int32_t* out = a.indices + (static_cast<size_t>(b) * a.S + t) * a.topK;
  if (t >= L) {
    for (int i = lane; i < a.topK; i += 32) out[i] = -1;
    return;
  }
  const int n_c = (t + 1) / ratio;
  if (n_c <= a.budget) {  // every block kept: the row lists 0..t
    for (int i = lane; i < a.topK; i += 32) out[i] = i <= t ? i : -1;
    return;
  }
  const float* srow = a.scores + static_cast<size_t>(b) * a.triPerSeq + tri_offset(t, ratio);
  // Keys live in registers, KPL per lane; only the first ceil(n_c / 32) of them
  // can be non-zero, so every pass skips the groups of 8 past that (a
  // warp-uniform branch, no instructions issued for them).
  constexpr int KG = 8;
  const int mlim = (n_c + 31) / 32;
  uint32_t key[KPL];
#pragma unroll
  for (int c = 0; c < KPL / KG; ++c) {
#pragma unroll
    for (int k = 0; k < KG; ++k) {
      const int g = lane + 32 * (c * KG + k);
      key[c * KG + k] = c * KG < mlim && g < n_c ? __float_as_uint(__ldcg(srow + g)) + 1u : 0u;
    }
  }
  // The cut key `lo` (the budget-th largest key) and `quota`, the number of
  // keys equal to it that are kept (lowest ids first).  Score-0 blocks (key 1) sit below
  // every positive one; among the positive keys a radix select refines a
  // 256-bin histogram of (key - lo) >> sh in this warp's shared memory until
  // the bin holding the cut has at most 32 keys (or is one key value), whose
  // exact order is then taken by counting.
  uint32_t* hist = hist_s[warp];
  uint32_t kmx = 0u, kmn = 0xffffffffu;
  int npos = 0;
#pragma unroll
  for (int c = 0; c < KPL / KG; ++c) {
    if (c * KG < mlim) {
#pragma unroll
      for (int k = 0; k < KG; ++k) {
        const uint32_t kk = key[c * KG + k];
        if (kk >= 2u) {
          kmx = max(kmx, kk);
          kmn = min(kmn, kk);
          ++npos;
        }
      }
    }
  }
  kmx = __reduce_max_sync(kFull, kmx);
  kmn = __reduce_min_sync(kFull, kmn);
  npos = static_cast<int>(__reduce_add_sync(kFull, static_cast<unsigned>(npos)));
  uint32_t lo;
  int quota;
  if (npos < a.budget) {  // every positive block is kept, then score-0 blocks by lowest id
    lo = 1u;
    quota = a.budget - npos;
  } else {
    uint32_t blo = kmn, span = kmx - kmn;  // keys of the current bin: [blo, blo + span]
    int need = a.budget;                   // keys of the current bin to keep
    for (;;) {
      const int sh = max(0, 24 - static_cast<int>(__clz(span)));  // span >> sh < 256
#pragma unroll
      for (int j = 0; j < 8; ++j) hist[lane * 8 + j] = 0u;
      __syncwarp();
#pragma unroll
      for (int c = 0; c < KPL / KG; ++c) {
        if (c * KG < mlim) {
#pragma unroll
          for (int k = 0; k < KG; ++k) {
            const uint32_t d = key[c * KG + k] - blo;  // keys below blo wrap past span
            if (d <= span) atomicAdd(hist + (d >> sh), 1u);
          }
        }
      }
      __syncwarp();
      // lane l owns bins 8l .. 8l+7; `run` counts the keys in higher bins
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
      int run = suffix - own, T = -1, above = 0, nT = 0;
#pragma unroll
      for (int j = 7; j >= 0; --j) {
        if (run < need && run + hb[j] >= need) {
          T = lane * 8 + j;
          above = run;
          nT = hb[j];
        }
        run += hb[j];
      }
      const int src = __ffs(__ballot_sync(kFull, T >= 0)) - 1;  // exactly one lane holds the bin
      T = __shfl_sync(kFull, T, src);
      need -= __shfl_sync(kFull, above, src);
      nT = __shfl_sync(kFull, nT, src);
      blo += static_cast<uint32_t>(T) << sh;
      span = sh == 0 ? 0u : min(span - (static_cast<uint32_t>(T) << sh), (1u << sh) - 1u);
      __syncwarp();  // every lane has read the histogram
      if (span == 0u) {  // one key value: its `need` lowest ids
        lo = blo;
        quota = need;
        break;
      }
      if (nT <= 32) {
        // the bin's keys, one per lane, then each one's count of larger and equal keys
        uint32_t* cand = hist;
        int at = 0;
#pragma unroll
        for (int c = 0; c < KPL / KG; ++c) {
          if (c * KG < mlim) {
#pragma unroll
            for (int k = 0; k < KG; ++k) {
              const bool in = key[c * KG + k] - blo <= span;
              const unsigned m = __ballot_sync(kFull, in);
              if (in) cand[at + __popc(m & ((1u << lane) - 1u))] = key[c * KG + k];
              at += __popc(m);
            }
          }
        }
        __syncwarp();
        const uint32_t mine = lane < nT ? cand[lane] : 0u;
        int gt = 0, eq = 0;
        for (int j = 0; j < nT; ++j) {
          const uint32_t v = __shfl_sync(kFull, mine, j);
          gt += v > mine ? 1 : 0;
          eq += v == mine ? 1 : 0;
        }
        const int hit = __ffs(__ballot_sync(kFull, lane < nT && gt < need && need <= gt + eq)) - 1;
        lo = __shfl_sync(kFull, mine, hit);
        quota = need - __shfl_sync(kFull, gt, hit);
        break;
      }
    }
  }
  int pos = 0;
  const unsigned below = (1u << lane) - 1u;
#pragma unroll
  for (int c = 0; c < KPL / KG; ++c) {
    if (c * KG < mlim) {
#pragma unroll
      for (int k = 0; k < KG; ++k) {
        const int m = c * KG + k;
        const bool eq = key[m] == lo;
        const unsigned eqm = __ballot_sync(kFull, eq);
        const bool take = key[m] > lo || (eq && __popc(eqm & below) < quota);
        quota = max(0, quota - __popc(eqm));
        const unsigned tm = __ballot_sync(kFull, take);
        if (take) {
          const int at = (pos + __popc(tm & below)) * ratio, g = lane + 32 * m;
          for (int j = 0; j < ratio; ++j) out[at + j] = g * ratio + j;
        }
        pos += __popc(tm);
      }
    }
  }
  const int head = pos * ratio;
  for (int i = head + lane; i < a.topK; i += 32) {
    const int j = n_c * ratio + (i - head);
    out[i] = j <= t ? j : -1;
  }
}

template <int DI>
cudaError_t launch_score(const SelArgs& a, int B, cudaStream_t st) {
  constexpr size_t smem = score_smem_bytes<DI>();
  static const cudaError_t attr = cudaFuncSetAttribute(
      prefill_score_kernel<DI>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (attr != cudaSuccess) return attr;
  dim3 grid((a.S + kRows - 1) / kRows, B);
  prefill_score_kernel<DI><<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

template <int VPT>
cudaError_t launch_topk(const SelArgs& a, int B, cudaStream_t st) {
  dim3 grid((a.S + kRows - 1) / kRows, B);
  if (a.ratio == 4)
    prefill_topk_kernel<VPT, 4><<<grid, kThreads, 0, st>>>(a);
  else
    prefill_topk_kernel<VPT, 0><<<grid, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_topk_any(const SelArgs& a, int B, cudaStream_t st) {
  const int nb = a.nbmax;
  if (nb <= 2 * kThreads) return launch_topk<2>(a, B, st);
  if (nb <= 4 * kThreads) return launch_topk<4>(a, B, st);
  if (nb <= 8 * kThreads) return launch_topk<8>(a, B, st);
  return launch_topk<16>(a, B, st);
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

// Workspace: status word, block keys fp16 [B][S/r][di], then the block scores
// fp32 of every row, per sequence in row order (tri_offset(S) floats each).
size_t kbar_region_bytes(int B, int S, int di, int ratio) {
  return (static_cast<size_t>(B) * (S / ratio) * di * sizeof(__half) + 255) / 256 * 256;
}
size_t indexer_prefill_workspace_bytes(int B, int S, int di, int ratio) {
  return kStatusBytes + kbar_region_bytes(B, S, di, ratio) +
         static_cast<size_t>(B) * static_cast<size_t>(tri_offset(S, ratio)) * sizeof(float);
}

cudaError_t launch_indexer_prefill(const QsaIndexerPrefillParams& p, const RopeFreqs& rf) {
  cudaStream_t st = static_cast<cudaStream_t>(p.stream);
  const int nbmax = p.seqLen / p.compressRatio;
  __half* kbar = reinterpret_cast<__half*>(static_cast<char*>(p.workspace) + kStatusBytes);
  if (nbmax > 0) {
    PoolArgs pa;
    pa.idxK = static_cast<const __half*>(p.idxK);
    pa.wk = p.kNormW;
    pa.ctx = p.contextLengths;
    pa.kbar = kbar;
    pa.S = p.seqLen;
    pa.nbmax = nbmax;
    pa.ratio = p.compressRatio;
    pa.rot = p.rotDim;
    pa.eps = p.rmsNormEps;
    pa.rf = rf;
    dim3 grid((nbmax + 7) / 8, p.batchSize);
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
  sa.scores = reinterpret_cast<float*>(static_cast<char*>(p.workspace) + kStatusBytes +
                                       kbar_region_bytes(p.batchSize, p.seqLen, p.headDim, p.compressRatio));
  sa.triPerSeq = tri_offset(p.seqLen, p.compressRatio);
  sa.indices = p.indices;
  sa.S = p.seqLen;
  sa.Hi = p.numHeads;
  sa.nbmax = nbmax;
  sa.ratio = p.compressRatio;
  sa.rot = p.rotDim;
  sa.budget = p.budget;
  sa.topK = p.topK;
  sa.eps = p.rmsNormEps;
  sa.rf = rf;
  const cudaError_t e = p.headDim == 64 ? launch_score<64>(sa, p.batchSize, st) : launch_score<128>(sa, p.batchSize, st);
  if (e != cudaSuccess) return e;
  return launch_topk_any(sa, p.batchSize, st);
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
