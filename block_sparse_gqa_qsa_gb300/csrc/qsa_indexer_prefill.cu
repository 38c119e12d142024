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
//                          select over the row's scores (bisection on the
//                          score bits with warp reductions, exact ties to the
//                          lower block id) and the expansion into the row's
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

constexpr int kRows = kPrefillRowsPerCta;  // rows per top-k CTA (one warp each)
constexpr int kThreads = 256;
constexpr int kSRows = 16;                 // rows per score CTA (two per warp)
constexpr int kKT = 64;                    // block keys per staged tile
constexpr int kKStages = 3;                // tiles in flight

// Start of row t's scores within its sequence: sum over u = 1..t of floor(u / r),
// i.e. the complete-block counts n_c of rows 0..t-1.
__host__ __device__ __forceinline__ long long tri_offset(long long t, int r) {
  const long long k = t / r;
  return r * k * (k - 1) / 2 + k * (t - k * r + 1);
}

template <int DI>
__host__ __device__ constexpr int qw_stride() {
  return DI + 8;
}
template <int DI>
constexpr size_t score_smem_bytes() {
  return static_cast<size_t>(kKStages) * kKT * DI * 2 + sizeof(float) * 8 * 8 * qw_stride<DI>();
}

// Block scores of 16 consecutive query rows of one sequence (rows whose n_c
// exceeds the budget; the others need no scores), written to the workspace.
// Warp w owns rows 2w and 2w+1: it prepares their index queries (RMSNorm*(1+w),
// RoPE in fp32 with angles reduced in integer turns), scales and splits them
// into hi/lo fp16 mma fragments held in registers (B operands: n = head,
// k = dim), and contracts them on the tensor cores (mma.sync m16n8k16, fp32
// accumulators) against 64-block tiles of fp16 block keys (A operands: m =
// block, k = dim) that the CTA streams through a 3-stage cp.async ring with a
// 16-byte XOR swizzle, read by ldmatrix without bank conflicts.  Relu and the
// head sum run on the accumulators.  Two CTAs share an SM.
template <int DI>
__global__ void __launch_bounds__(kThreads, 2) prefill_score_kernel(const SelArgs a) {
  constexpr int PER = DI / 32;
  constexpr int KS = DI / 16;          // k-steps of 16 dims
  constexpr int ROWB = DI * 2;         // bytes of one block key
  constexpr int TILEB = kKT * ROWB;    // bytes of one tile
  constexpr int CPR = DI / 8;          // 16-byte chunks of one block key
  constexpr int QWS = qw_stride<DI>();
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* tiles = smem;                                               // [kKStages][kKT][DI] fp16, swizzled
  float* qw = reinterpret_cast<float*>(smem + kKStages * TILEB);       // [8 warps][8 heads][QWS]
  __shared__ unsigned long long turn_s[64];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.y;
  const int ngroups = (a.S + kSRows - 1) / kSRows;
  const int t0 = (ngroups - 1 - static_cast<int>(blockIdx.x)) * kSRows;  // longest rows first
  const int L = max(0, min(a.ctx[b], a.S));
  const int t_end = min(t0 + kSRows, L);  // live rows [t0, t_end)
  if (t0 >= L) return;
  const int n_hi = t_end / a.ratio;  // complete blocks seen by the group's last live row
  if (n_hi <= a.budget) return;

  // the first tiles start landing while the queries are prepared
  const __half* kb_g = a.kbar + static_cast<size_t>(b) * a.nbmax * DI;
  const int ntiles = (n_hi + kKT - 1) / kKT;
  auto issue = [&](int tile) {
    uint8_t* dst = tiles + (tile % kKStages) * TILEB;
    const int gbase = tile * kKT;
#pragma unroll
    for (int k = 0; k < kKT * CPR / kThreads; ++k) {
      const int e = tid + k * kThreads;
      const int row = e / CPR, c = e % CPR;
      const bool ok = gbase + row < n_hi;
      cp_async16(smem_addr(dst + row * ROWB + ((c ^ (row & 7)) << 4)),
                 kb_g + static_cast<size_t>(ok ? gbase + row : 0) * DI + c * 8, ok);
    }
  };
  issue(0);
  cp_async_commit();
  if (ntiles > 1) issue(1);
  cp_async_commit();
  if (tid < 64) turn_s[tid] = a.rf.turn[tid];
  __syncthreads();

  // ------------------------------------------------------------ query prep
  uint32_t qf[2][KS][4];  // per row and k-step: hi b0, hi b1, lo b0, lo b1
  float* qwarp = qw + warp * 8 * QWS;
  const int half = a.rot >> 1;
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int t = t0 + 2 * warp + rr;
    const bool live = t < t_end;
    float cs[PER], sn[PER];
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      const int i = lane + 32 * p;
      cs[p] = 1.f;
      sn[p] = 0.f;
      if (live && i < a.rot) rope_cos_sin_turns(static_cast<unsigned>(t), turn_s[i < half ? i : i - half], cs[p], sn[p]);
    }
    float mx = 0.f;
    for (int h = 0; h < 8; ++h) {
      float* qh = qwarp + h * QWS;
      if (live && h < a.Hi) {
        const __half* x = a.idxQ + ((static_cast<size_t>(b) * a.S + t) * a.Hi + h) * DI;
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
          qh[i] = y[p];
        }
        __syncwarp();
        float v[PER];
#pragma unroll
        for (int p = 0; p < PER; ++p) {
          const int i = lane + 32 * p;
          v[p] = y[p];
          if (i < half)
            v[p] = y[p] * cs[p] - qh[i + half] * sn[p];
          else if (i < a.rot)
            v[p] = y[p] * cs[p] + qh[i - half] * sn[p];
          mx = fmaxf(mx, fabsf(v[p]));
        }
        __syncwarp();
#pragma unroll
        for (int p = 0; p < PER; ++p) qh[lane + 32 * p] = v[p];
      } else {
#pragma unroll
        for (int p = 0; p < PER; ++p) qh[lane + 32 * p] = 0.f;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    __syncwarp();
    const float scale = index_q_scale(mx);
    const float* qn = qwarp + (lane >> 2) * QWS + (lane & 3) * 2;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const float2 x0 = *reinterpret_cast<const float2*>(qn + ks * 16);
      const float2 x1 = *reinterpret_cast<const float2*>(qn + ks * 16 + 8);
      split_half2(x0.x * scale, x0.y * scale, qf[rr][ks][0], qf[rr][ks][2]);
      split_half2(x1.x * scale, x1.y * scale, qf[rr][ks][1], qf[rr][ks][3]);
    }
    __syncwarp();
  }

  // ---------------------------------------------------------- block scores
  int n_c[2];
  bool store[2];
  float* srow[2];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int t = t0 + 2 * warp + rr;
    n_c[rr] = (t + 1) / a.ratio;
    store[rr] = t < t_end && n_c[rr] > a.budget;  // this row needs its scores
    srow[rr] = a.scores + static_cast<size_t>(b) * a.triPerSeq + tri_offset(t, a.ratio);
  }
  const int arow = lane & 15, achunk = lane >> 4;  // this lane's ldmatrix row and chunk within a 16x16 A tile
  for (int tile = 0; tile < ntiles; ++tile) {
    cp_async_wait<1>();
    __syncthreads();  // tile `tile` visible to all; every warp is done with tile - 1
    if (tile + 2 < ntiles) issue(tile + 2);
    cp_async_commit();
    const uint32_t tb = smem_addr(tiles + (tile % kKStages) * TILEB);
    const int gbase = tile * kKT;
#pragma unroll 1
    for (int mt = 0; mt < kKT / 16; mt += 2) {
      float acc[2][2][2][4];  // [m-tile][row][hi, lo][fragment]
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr)
#pragma unroll
          for (int hl = 0; hl < 2; ++hl)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[u][rr][hl][j] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int row = (mt + u) * 16 + arow;
          uint32_t af[4];
          ldsm_x4(tb + row * ROWB + (((ks * 2 + achunk) ^ (row & 7)) << 4), af[0], af[1], af[2], af[3]);
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            mma16816(acc[u][rr][0], af, qf[rr][ks][0], qf[rr][ks][1]);
            mma16816(acc[u][rr][1], af, qf[rr][ks][2], qf[rr][ks][3]);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int g = gbase + (mt + u) * 16 + (lane >> 2) + (lane & 1) * 8;
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const float sc = relu_head_sum(acc[u][rr][0], acc[u][rr][1]);
          if (store[rr] && (lane & 2) == 0 && g < n_c[rr]) srow[rr][g] = sc;
        }
      }
    }
  }
  cp_async_wait<0>();
}

// ------------------------------------ select + expand, one warp per row
// Lane l holds the scores of blocks l + 32 m.  Keys are the score bits + 1
// (order-preserving for scores >= 0; 0 marks blocks past the row's n_c).
// Bisection on the key finds T with count(key >= T) >= budget >
// count(key > T); the blocks above T are kept, and of those equal to T the
// lowest ids, so the kept set is the top `budget` by (score desc, id asc).
// A probe with exactly `budget` keys at or above it ends the search early:
// those keys are the set (T = probe - 1 and no key equal to T is kept).
// Walking m upwards visits ids in ascending order, so ballots compact the
// kept blocks straight into the ascending list.  Rows t >= L are all -1 and
// rows with n_c <= budget list 0..t.
template <int VPT>
__global__ void __launch_bounds__(kThreads) prefill_topk_kernel(const SelArgs a) {
  constexpr int KPL = kThreads * VPT / 32;
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
  const int n_c = (t + 1) / a.ratio;
  if (n_c <= a.budget) {  // every block kept: the row lists 0..t
    for (int i = lane; i < a.topK; i += 32) out[i] = i <= t ? i : -1;
    return;
  }
  const float* srow = a.scores + static_cast<size_t>(b) * a.triPerSeq + tri_offset(t, a.ratio);
  // Keys live in registers, KPL per lane; only the first ceil(n_c / 32) of them
  // can be non-zero, so every pass skips the groups of 8 past that (a
  // warp-uniform branch, no instructions issued for them).
  constexpr int KG = 8;
  const int mlim = (n_c + 31) / 32;
  const int nslot = KG * ((mlim + KG - 1) / KG);  // keys per lane that the passes visit
  uint32_t key[KPL];
#pragma unroll
  for (int c = 0; c < KPL / KG; ++c) {
#pragma unroll
    for (int k = 0; k < KG; ++k) {
      const int g = lane + 32 * (c * KG + k);
      key[c * KG + k] = c * KG < mlim && g < n_c ? __float_as_uint(__ldcg(srow + g)) + 1u : 0u;
    }
  }
  uint32_t lo = 1u, hi = 0x80000001u;  // count(>= lo) >= budget > count(>= hi)
  int c_hi = 0;
  while (hi - lo > 1u) {
    const uint32_t mid = lo + ((hi - lo) >> 1);
    // keys lie in [0, 2^31) and mid in [1, 2^31], so key - mid as a signed
    // 32-bit value is negative exactly when key < mid
    int below_mid = 0;
#pragma unroll
    for (int c = 0; c < KPL / KG; ++c) {
      if (c * KG < mlim) {
#pragma unroll
        for (int k = 0; k < KG; ++k) below_mid += static_cast<int>(key[c * KG + k] - mid) >> 31;
      }
    }
    const int c = static_cast<int>(__reduce_add_sync(kFull, static_cast<unsigned>(nslot + below_mid)));
    if (c == a.budget) {  // exactly the budget at or above mid: keep those, no tie to break
      lo = mid - 1u;
      c_hi = a.budget;
      break;
    }
    if (c > a.budget) {
      lo = mid;
    } else {
      hi = mid;
      c_hi = c;
    }
  }
  int quota = a.budget - c_hi;  // blocks with key == lo to keep, lowest ids first (none after an exact stop)
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
          const int at = (pos + __popc(tm & below)) * a.ratio, g = lane + 32 * m;
          for (int j = 0; j < a.ratio; ++j) out[at + j] = g * a.ratio + j;
        }
        pos += __popc(tm);
      }
    }
  }
  const int head = pos * a.ratio;
  for (int i = head + lane; i < a.topK; i += 32) {
    const int j = n_c * a.ratio + (i - head);
    out[i] = j <= t ? j : -1;
  }
}

template <int DI>
cudaError_t launch_score(const SelArgs& a, int B, cudaStream_t st) {
  constexpr size_t smem = score_smem_bytes<DI>();
  static const cudaError_t attr = cudaFuncSetAttribute(
      prefill_score_kernel<DI>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (attr != cudaSuccess) return attr;
  dim3 grid((a.S + kSRows - 1) / kSRows, B);
  prefill_score_kernel<DI><<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

template <int VPT>
cudaError_t launch_topk(const SelArgs& a, int B, cudaStream_t st) {
  dim3 grid((a.S + kRows - 1) / kRows, B);
  prefill_topk_kernel<VPT><<<grid, kThreads, 0, st>>>(a);
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
