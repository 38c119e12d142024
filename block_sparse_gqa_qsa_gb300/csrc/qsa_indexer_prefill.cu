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
//   prefill_select_kernel  one CTA per 8 consecutive query rows of one
//                          sequence: index-query prep (fp32, angles reduced
//                          in integer turns), block
//                          scores on the CUDA cores (fp32 FMA, a register-tiled
//                          contraction of 8 rows x 8 heads against 256-block
//                          tiles staged in shared memory), the relu/head sum,
//                          then one warp per row: a deterministic top-`budget`
//                          select (bisection on the score bits with warp
//                          reductions, exact ties to the lower block id) and
//                          the expansion into the row's ascending index list.
//                          A row group's scores never leave shared memory.
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
  int32_t* indices;
  int S, Hi, nbmax, ratio, rot, budget, topK;
  float eps;
  RopeFreqs rf;
};

constexpr int kRows = kPrefillRowsPerCta;  // rows per CTA (one warp each)
constexpr int kThreads = 256;
constexpr int kTile = 256;                  // blocks per score tile (8 per lane)
constexpr int kKC = 16;                     // key dims staged per step
constexpr int kKS = kKC + 4;                // padded row stride (conflict-free float4 reads)
constexpr int kHI = 8;                      // heads per thread tile (Hi <= 8, extra heads are zero)

template <int DI, int VPT>
constexpr size_t select_smem_bytes() {
  return sizeof(float) * (static_cast<size_t>(DI) * kRows * kHI + 2 * kTile * kKS + kRows * kThreads * VPT +
                          kRows * DI + kRows * 128);
}

template <int DI, int VPT>
__global__ void __launch_bounds__(kThreads, 1) prefill_select_kernel(const SelArgs a) {
  constexpr int NBMAX = kThreads * VPT;
  extern __shared__ __align__(16) float smem[];
  float* q_s = smem;                          // [DI][kRows][kHI] prepared queries
  float* kb_s = q_s + DI * kRows * kHI;       // [2][kTile][kKS]  block-key tile (fp32)
  float* sc_s = kb_s + 2 * kTile * kKS;       // [kRows][NBMAX]   block scores
  float* ys_s = sc_s + kRows * NBMAX;         // [kRows][DI]      per-warp RoPE scratch
  float* cs_s = ys_s + kRows * DI;            // [kRows][64][2]   cos/sin per row

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.y;
  const int ngroups = (a.S + kRows - 1) / kRows;
  const int t0 = (ngroups - 1 - static_cast<int>(blockIdx.x)) * kRows;  // longest rows first
  const int L = max(0, min(a.ctx[b], a.S));
  int32_t* ind_b = a.indices + static_cast<size_t>(b) * a.S * a.topK;
  const int t_end = min(t0 + kRows, L);  // live rows [t0, t_end)
  {
    const int first_pad = max(t0, t_end);
    const int npad = min(t0 + kRows, a.S) - first_pad;
    for (int i = tid; i < npad * a.topK; i += kThreads) ind_b[static_cast<size_t>(first_pad) * a.topK + i] = -1;
  }
  if (t0 >= L) return;
  const int nlive = t_end - t0;
  const int n_hi = t_end / a.ratio;  // complete blocks seen by the group's last live row

  if (n_hi > a.budget) {
    // ---------------------------------------------------------- query prep
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

    // ------------------------------------------------------- block scores
    // Lane owns blocks lane + 32 m (m < 8) of the tile, for its warp's row
    // and all kHI heads: 64 accumulators, each a plain ascending-k FMA chain,
    // so a block's score does not depend on where the block sits in a tile.
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
        float* dst = kb_s + (kc & 1) * kTile * kKS + tid * kKS;
        {
          const __half2* h0 = reinterpret_cast<const __half2*>(&pre0);
          const __half2* h1 = reinterpret_cast<const __half2*>(&pre1);
          float4 f[4];
          float2 t;
          t = __half22float2(h0[0]); f[0].x = t.x; f[0].y = t.y;
          t = __half22float2(h0[1]); f[0].z = t.x; f[0].w = t.y;
          t = __half22float2(h0[2]); f[1].x = t.x; f[1].y = t.y;
          t = __half22float2(h0[3]); f[1].z = t.x; f[1].w = t.y;
          t = __half22float2(h1[0]); f[2].x = t.x; f[2].y = t.y;
          t = __half22float2(h1[1]); f[2].z = t.x; f[2].w = t.y;
          t = __half22float2(h1[2]); f[3].x = t.x; f[3].y = t.y;
          t = __half22float2(h1[3]); f[3].z = t.x; f[3].w = t.y;
#pragma unroll
          for (int i = 0; i < 4; ++i) reinterpret_cast<float4*>(dst)[i] = f[i];
        }
        __syncthreads();
        if (kc + 1 < DI / kKC) {
          pre0 = gok ? __ldg(src + 2 * (kc + 1)) : zero;
          pre1 = gok ? __ldg(src + 2 * (kc + 1) + 1) : zero;
        }
        const float* kt = kb_s + (kc & 1) * kTile * kKS;
        const float* qk = q_s + static_cast<size_t>(kc * kKC) * kRows * kHI + warp * kHI;
#pragma unroll
        for (int kq = 0; kq < kKC / 4; ++kq) {
          float4 kv[8];
#pragma unroll
          for (int m = 0; m < 8; ++m) kv[m] = *reinterpret_cast<const float4*>(kt + (lane + 32 * m) * kKS + kq * 4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const float* qp = qk + (kq * 4 + kk) * kRows * kHI;
            const float4 qa = *reinterpret_cast<const float4*>(qp);
            const float4 qb = *reinterpret_cast<const float4*>(qp + 4);
            const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              const float kval = kk == 0 ? kv[m].x : kk == 1 ? kv[m].y : kk == 2 ? kv[m].z : kv[m].w;
#pragma unroll
              for (int h = 0; h < kHI; ++h) acc[m][h] = fmaf(qv[h], kval, acc[m][h]);
            }
          }
        }
      }
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int g = gbase + lane + 32 * m;
        if (g < n_hi) {
          float s = 0.f;
#pragma unroll
          for (int h = 0; h < kHI; ++h) s += acc[m][h] > 0.f ? acc[m][h] : 0.f;
          sc_s[warp * NBMAX + g] = s;
        }
      }
    }
    __syncthreads();
  }

  // ------------------------------------ select + expand, one warp per row
  // Lane l holds the scores of blocks l + 32 m.  Keys are the score bits + 1
  // (order-preserving for scores >= 0; 0 marks blocks past the row's n_c).
  // Bisection on the key finds T with count(key >= T) >= budget >
  // count(key > T); the blocks above T are kept, and of those equal to T the
  // lowest ids, so the kept set is the top `budget` by (score desc, id asc).
  // Walking m upwards visits ids in ascending order, so ballots compact the
  // kept blocks straight into the ascending list.
  if (warp < nlive) {
    constexpr int KPL = NBMAX / 32;
    const int t = t0 + warp;
    const int n_c = (t + 1) / a.ratio;
    int32_t* out = ind_b + static_cast<size_t>(t) * a.topK;
    if (n_c <= a.budget) {  // every block kept: the row lists 0..t
      for (int i = lane; i < a.topK; i += 32) out[i] = i <= t ? i : -1;
    } else {
      uint32_t key[KPL];
#pragma unroll
      for (int m = 0; m < KPL; ++m) {
        const int g = lane + 32 * m;
        key[m] = g < n_c ? __float_as_uint(sc_s[warp * NBMAX + g]) + 1u : 0u;
      }
      uint32_t lo = 1u, hi = 0x80000001u;  // count(>= lo) >= budget > count(>= hi)
      int c_hi = 0;
      while (hi - lo > 1u) {
        const uint32_t mid = lo + ((hi - lo) >> 1);
        int c = 0;
#pragma unroll
        for (int m = 0; m < KPL; ++m) c += key[m] >= mid ? 1 : 0;
        c = static_cast<int>(__reduce_add_sync(kFull, static_cast<unsigned>(c)));
        if (c >= a.budget) {
          lo = mid;
        } else {
          hi = mid;
          c_hi = c;
        }
      }
      int quota = a.budget - c_hi;  // blocks with key == lo to keep, lowest ids first
      int pos = 0;
      const unsigned below = (1u << lane) - 1u;
#pragma unroll
      for (int m = 0; m < KPL; ++m) {
        const bool eq = key[m] == lo;
        const unsigned eqm = __ballot_sync(kFull, eq);
        const bool take = key[m] > lo || (eq && __popc(eqm & below) < quota);
        quota = max(0, quota - __popc(eqm));
        const unsigned tm = __ballot_sync(kFull, take);
        if (take) {
          const int at = (pos + __popc(tm & below)) * a.ratio, g = lane + 32 * m;
          for (int j = 0; j < a.ratio; ++j) out[at + j] = g * a.ratio + j;
        }
        pos += __popc(tm);
      }
      const int head = pos * a.ratio;
      for (int i = head + lane; i < a.topK; i += 32) {
        const int j = n_c * a.ratio + (i - head);
        out[i] = j <= t ? j : -1;
      }
    }
  }
}

template <int DI, int VPT>
cudaError_t launch_select(const SelArgs& a, int B, cudaStream_t st) {
  constexpr size_t smem = select_smem_bytes<DI, VPT>();
  static const cudaError_t attr = cudaFuncSetAttribute(
      prefill_select_kernel<DI, VPT>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (attr != cudaSuccess) return attr;
  dim3 grid((a.S + kRows - 1) / kRows, B);
  prefill_select_kernel<DI, VPT><<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

template <int DI>
cudaError_t launch_select_di(const SelArgs& a, int B, cudaStream_t st) {
  const int nb = a.nbmax;
  if (nb <= 2 * kThreads) return launch_select<DI, 2>(a, B, st);
  if (nb <= 4 * kThreads) return launch_select<DI, 4>(a, B, st);
  if (nb <= 8 * kThreads) return launch_select<DI, 8>(a, B, st);
  return launch_select<DI, 16>(a, B, st);
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

size_t indexer_prefill_workspace_bytes(int B, int S, int di, int ratio) {
  return kStatusBytes + static_cast<size_t>(B) * (S / ratio) * di * sizeof(__half);
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
  return p.headDim == 64 ? launch_select_di<64>(sa, p.batchSize, st) : launch_select_di<128>(sa, p.batchSize, st);
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
