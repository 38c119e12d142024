// qsa_rope.cu -- the upstream step of a QSA attention layer ("Qsa Attention
// Plugin", fused step 1: packed-QKV split, per-head qk-norm with the gammas
// folded as (1 + w), partial RoPE, paged-KV write and dense K/V mirrors).
//
// A persistent grid of 128-thread CTAs walks the tokens (b, s).  A token's
// packed heads are moved as 16-byte chunks of 8 halves by cp.async into a ring
// of three token slots in shared memory, so each SM keeps the loads of the
// next two tokens of every resident CTA in flight while it computes.  Each
// warp forms the token's RoPE cos/sin itself: the angle is reduced modulo a
// turn exactly in 64-bit integer arithmetic (the frequency as a fixed-point
// fraction of a turn), then evaluated in fp32, so no step needs FP64 or a
// CTA barrier.  The D/8 lanes that hold one head reduce its sum of squares
// with shuffles.  Because rotDim is a multiple of 16, the rotation partner of
// a chunk (rotDim/2 dims away) is a whole chunk held by another lane of the
// same group, fetched with shuffles.  q/k values are rounded once to fp16; v
// chunks are copied bit for bit.  Outputs: q (always), the dense K/V mirrors
// (optional) and the leading D columns of the token's K and V pool rows
// (optional; the indexer tails are never touched).
#include <cmath>

#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

struct RopeArgs {
  const __half* qkv;
  const float* qw;
  const float* kw;
  const int32_t* ctx;
  __half* qout;
  __half* kout;  // may be null
  __half* vout;  // may be null
  __half* pool;  // may be null
  const int32_t* pageTable;
  int S, Hq, Hkv, rot, poolHeadDim, numFlatPages, maxPagesPerSeq;
  float eps;
  unsigned long long turn[64];  // inv_freq of pair i as a 64-bit fixed-point fraction of a turn
};

constexpr int kRopeThreads = 128;
constexpr int kRopeStages = 3;  // token slots of the cp.async ring

__device__ __forceinline__ uint4 pack8(const uint64_t (&v)[4]) {
  return make_uint4(pack_half2(lo_f2(v[0]), hi_f2(v[0])), pack_half2(lo_f2(v[1]), hi_f2(v[1])),
                    pack_half2(lo_f2(v[2]), hi_f2(v[2])), pack_half2(lo_f2(v[3]), hi_f2(v[3])));
}

__device__ __forceinline__ void unpack8(const uint4 r, uint64_t (&v)[4]) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    v[i] = pack_f2(f.x, f.y);
  }
}

// 1 / sqrt(m): the hardware estimate refined by one Newton-Raphson step, r <- r (3 - m r^2) / 2, which
// leaves a relative error of a few units of 2^-24.
__device__ __forceinline__ float rsqrt_nr(float m) {
  const float r = rsqrtf(m);
  return r * fmaf(-0.5f * m * r, r, 1.5f);
}

// The D/8 lanes of one aligned group hold the consecutive 16-byte chunks of one head; y is this lane's
// chunk as 4 float pairs, w its 8 values of (1 + w) as pairs, partner the lane holding the rotation
// partner chunk (itself for chunks past rotDim) and cs / sn this chunk's rotation coefficients, elements
// 0-3 at cs[0..3] and 4-7 at cs[4 G..4 G + 3]: y' = y cs + partner sn, where sn carries the sign and
// chunks past rotDim have cs = 1, sn = 0.  On return y holds the normed, rotated values.  Elementwise
// work runs on f32x2 pairs (round-to-nearest, as the scalar operations).
template <int D>
__device__ __forceinline__ void norm_rotate(uint64_t (&y)[4], int partner, const uint64_t (&w)[4], float eps,
                                            const float* cs, const float* sn) {
  constexpr int G = D / 8;
  uint64_t acc = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) acc = ffma2(y[k], y[k], acc);
  float ss = lo_f2(acc) + hi_f2(acc);
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
  const float inv = rsqrt_nr(ss * (1.0f / D) + eps);
  const uint64_t inv2 = pack_f2(inv, inv);
  const ulonglong2 ca = *reinterpret_cast<const ulonglong2*>(cs), cb = *reinterpret_cast<const ulonglong2*>(cs + 4 * G);
  const ulonglong2 sa = *reinterpret_cast<const ulonglong2*>(sn), sb = *reinterpret_cast<const ulonglong2*>(sn + 4 * G);
  const uint64_t cv[4] = {ca.x, ca.y, cb.x, cb.y}, sv[4] = {sa.x, sa.y, sb.x, sb.y};
#pragma unroll
  for (int k = 0; k < 4; ++k) y[k] = fmul2(fmul2(y[k], inv2), w[k]);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint64_t p = pack_f2(__shfl_sync(kFull, lo_f2(y[k]), partner), __shfl_sync(kFull, hi_f2(y[k]), partner));
    y[k] = ffma2(p, sv[k], fmul2(y[k], cv[k]));
  }
}

__device__ __forceinline__ void load_w(const float* p, int G, uint64_t (&w)[4]) {
  const ulonglong2 a = *reinterpret_cast<const ulonglong2*>(p), b = *reinterpret_cast<const ulonglong2*>(p + 4 * G);
  w[0] = a.x;
  w[1] = a.y;
  w[2] = b.x;
  w[3] = b.y;
}

// Position of a CTA's n-th token; advanced by the grid stride without a division.
struct TokenCursor {
  long long tok;
  int b, s;
  __device__ __forceinline__ void step(int grid, int gq, int gr, int S) {
    tok += grid;
    b += gq;
    s += gr;
    if (s >= S) {
      s -= S;
      ++b;
    }
  }
};

// Persistent: CTA x takes tokens x, x + grid, ...  Each thread copies, with cp.async, exactly the chunks
// c = threadIdx.x + kRopeThreads k of a token that it later reads, so the ring of kRopeStages token
// slots needs no barrier: the copies of the next kRopeStages - 1 tokens fly while this one is computed.
// Each warp forms its own rotation coefficients for the token, so warps never wait on one another.
template <int D>
__global__ void __launch_bounds__(kRopeThreads) rope_qkv_kernel(const RopeArgs a, int T) {
  constexpr int G = D / 8;  // chunks per head; 32 is a multiple of G, so lane l always holds chunk l % G
  constexpr int W = kRopeThreads / 32;
  extern __shared__ __align__(16) uint4 ring[];  // [kRopeStages][nchunk]
  // per warp: rotation coefficients of chunk j, element e at [e / 4][j][e % 4], so that the lanes of a
  // group read consecutive 16-byte words (see norm_rotate); (1 + w) of q and k heads, same layout
  __shared__ __align__(16) float cos_s[W][2][G][4];
  __shared__ __align__(16) float sin_s[W][2][G][4];
  __shared__ __align__(16) float w1_s[2][2][G][4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, j = lane & (G - 1);
  const int NH = a.Hq + 2 * a.Hkv, nchunk = NH * G, firstK = a.Hq * G, firstV = (a.Hq + a.Hkv) * G;
  const int half = a.rot >> 1, hl = half >> 3;
  const int partner = j < hl ? lane + hl : (j < 2 * hl ? lane - hl : lane);
  const int grid = static_cast<int>(gridDim.x), gq = grid / a.S, gr = grid - gq * a.S;
  const uint4* src = reinterpret_cast<const uint4*>(a.qkv);
  for (int i = threadIdx.x; i < 2 * D; i += kRopeThreads) {
    const int d = i % D;
    w1_s[i / D][(d & 7) >> 2][d >> 3][d & 3] = 1.0f + __ldg((i < D ? a.qw : a.kw) + d);
  }
  for (int i = lane + 16 * hl; i < 8 * G; i += 32) {  // chunks past rotDim pass through
    cos_s[warp][(i & 7) >> 2][i >> 3][i & 3] = 1.0f;
    sin_s[warp][(i & 7) >> 2][i >> 3][i & 3] = 0.0f;
  }
  __syncthreads();  // w1_s
  uint64_t w1q[4];  // this lane's chunk of (1 + w) for q heads, kept in registers
  load_w(&w1_s[0][0][j][0], G, w1q);
  const float* w1k = &w1_s[1][0][j][0];
  const float* cs = &cos_s[warp][0][j][0];
  const float* sn = &sin_s[warp][0][j][0];
  TokenCursor cur{blockIdx.x, static_cast<int>(blockIdx.x) / a.S, static_cast<int>(blockIdx.x) % a.S};
  TokenCursor ahead = cur;
  auto issue = [&](int n) {  // one commit group per token slot, empty past the end or for padding rows
    if (ahead.tok < T) {
      const int L = __ldg(a.ctx + ahead.b);
      if (a.S == 1 ? L >= 1 : ahead.s < L) {
        const uint4* g = src + static_cast<size_t>(ahead.tok) * nchunk;
        uint4* d = ring + (n % kRopeStages) * nchunk;
        for (int c = threadIdx.x; c < nchunk; c += kRopeThreads) cp_async16(smem_addr(d + c), g + c, true);
      }
    }
    cp_async_commit();
    ahead.step(grid, gq, gr, a.S);
  };
#pragma unroll
  for (int n = 0; n < kRopeStages - 1; ++n) issue(n);
  for (int n = 0; cur.tok < T; ++n, cur.step(grid, gq, gr, a.S)) {
    issue(n + kRopeStages - 1);  // into the slot this thread read in iteration n - 1
    const int tok = static_cast<int>(cur.tok), L = __ldg(a.ctx + cur.b);
    const bool live = a.S == 1 ? L >= 1 : cur.s < L;
    __half* const qo = a.qout + static_cast<size_t>(tok) * a.Hq * D;
    __half* const ko = a.kout ? a.kout + static_cast<size_t>(tok) * a.Hkv * D : nullptr;
    __half* const vo = a.vout ? a.vout + static_cast<size_t>(tok) * a.Hkv * D : nullptr;
    if (!live) {  // padding row: zeros in the dense outputs, nothing in the pool
      for (int c = threadIdx.x; c < nchunk; c += kRopeThreads) {
        __half* dense = c < firstK ? qo + 8 * c : c < firstV ? (ko ? ko + 8 * (c - firstK) : nullptr)
                                                              : (vo ? vo + 8 * (c - firstV) : nullptr);
        if (dense) *reinterpret_cast<uint4*>(dense) = make_uint4(0u, 0u, 0u, 0u);
      }
      continue;
    }
    const int pos = a.S == 1 ? L - 1 : cur.s;
    __syncwarp();  // the warp is done with the previous token's coefficients
    for (int i = lane; i < half; i += 32) {  // pair (i, i + half): chunks i/8 and i/8 + hl
      float c, s;
      rope_cos_sin_turns(static_cast<unsigned>(pos), a.turn[i], c, s);
      const int e = i & 7, h4 = e >> 2, jc = i >> 3;
      cos_s[warp][h4][jc][e & 3] = c;
      sin_s[warp][h4][jc][e & 3] = -s;
      cos_s[warp][h4][jc + hl][e & 3] = c;
      sin_s[warp][h4][jc + hl][e & 3] = s;
    }
    // pool rows of this token (null when there is no pool or the page is outside it)
    __half* krow = nullptr;
    __half* vrow = nullptr;
    if (a.pool && pos < a.maxPagesPerSeq * kTokensPerPageHost) {
      const int32_t* pt = a.pageTable + static_cast<size_t>(cur.b) * 2 * a.maxPagesPerSeq;
      const int kp = __ldg(pt + (pos >> 7)), vp = __ldg(pt + a.maxPagesPerSeq + (pos >> 7));
      if (static_cast<unsigned>(kp) < static_cast<unsigned>(a.numFlatPages))
        krow = a.pool + (static_cast<size_t>(kp) * kTokensPerPageHost + (pos & 127)) * a.Hkv * a.poolHeadDim;
      if (static_cast<unsigned>(vp) < static_cast<unsigned>(a.numFlatPages))
        vrow = a.pool + (static_cast<size_t>(vp) * kTokensPerPageHost + (pos & 127)) * a.Hkv * a.poolHeadDim;
    }
    cp_async_wait<kRopeStages - 1>();  // this thread's chunks of token n have landed
    __syncwarp();                      // the warp's coefficients are visible
    const uint4* row = ring + (n % kRopeStages) * nchunk;
    // warp-uniform trip count: every lane takes part in the group shuffles; lanes past the end carry zeros.
    // Two chunks at a time interleave their shuffle chains.
#pragma unroll 2
    for (int c0 = warp * 32; c0 < nchunk; c0 += kRopeThreads) {
      const int c = c0 + lane;
      const bool in = c < nchunk;
      const uint4 raw = in ? row[c] : make_uint4(0u, 0u, 0u, 0u);
      if (c0 >= firstV) {  // the v heads come last: the whole warp copies
        if (in) {
          if (vo) *reinterpret_cast<uint4*>(vo + 8 * (c - firstV)) = raw;
          if (vrow) *reinterpret_cast<uint4*>(vrow + ((c - firstV) / G) * a.poolHeadDim + 8 * j) = raw;
        }
        continue;
      }
      uint64_t y[4];
      unpack8(raw, y);
      if (c0 + 32 <= firstK) {  // q heads only
        norm_rotate<D>(y, partner, w1q, a.eps, cs, sn);
        *reinterpret_cast<uint4*>(qo + 8 * c) = pack8(y);
        continue;
      }
      uint64_t wk[4];
      load_w(w1k, G, wk);
      if (c < firstK) {
#pragma unroll
        for (int k = 0; k < 4; ++k) wk[k] = w1q[k];
      }
      norm_rotate<D>(y, partner, wk, a.eps, cs, sn);
      if (!in) continue;
      const bool isq = c < firstK, isv = c >= firstV;
      const uint4 packed = isv ? raw : pack8(y);
      const int ck = isv ? c - firstV : c - firstK;  // chunk index within the k (or v) heads
      __half* dense = isq ? qo + 8 * c : (isv ? vo : ko) ? (isv ? vo : ko) + 8 * ck : nullptr;
      __half* prow = isq ? nullptr : (isv ? vrow : krow);
      if (dense) *reinterpret_cast<uint4*>(dense) = packed;
      if (prow) *reinterpret_cast<uint4*>(prow + (ck / G) * a.poolHeadDim + 8 * j) = packed;
    }
  }
  cp_async_wait<0>();  // the trailing groups are empty; nothing is left in flight at exit
}

}  // namespace

cudaError_t launch_rope_qkv(const QsaRopeQkvParams& p, const RopeFreqs& rf) {
  RopeArgs a;
  a.qkv = static_cast<const __half*>(p.qkv);
  a.qw = p.qNormW;
  a.kw = p.kNormW;
  a.ctx = p.contextLengths;
  a.qout = static_cast<__half*>(p.qOut);
  a.kout = static_cast<__half*>(p.kOut);
  a.vout = static_cast<__half*>(p.vOut);
  a.pool = static_cast<__half*>(p.kvPool);
  a.pageTable = p.pageTable;
  a.S = p.seqLen;
  a.Hq = p.numQHeads;
  a.Hkv = p.numKVHeads;
  a.rot = p.rotDim;
  a.poolHeadDim = p.poolHeadDim;
  a.numFlatPages = p.numFlatPages;
  a.maxPagesPerSeq = p.maxPagesPerSeq;
  a.eps = p.rmsNormEps;
  for (int i = 0; i < 64; ++i) a.turn[i] = rf.turn[i];
  const int T = p.batchSize * p.seqLen;  // validated <= INT_MAX
  const int nchunk = (p.numQHeads + 2 * p.numKVHeads) * (p.headDim / 8);
  const size_t smem = static_cast<size_t>(kRopeStages) * nchunk * 16;
  cudaStream_t st = static_cast<cudaStream_t>(p.stream);
  auto go = [&](auto kernel) -> cudaError_t {
    static const cudaError_t attr = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                         kRopeStages * kRopeMaxRowBytes);
    if (attr != cudaSuccess) return attr;
    int perSm = 0;
    const cudaError_t occ = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&perSm, kernel, kRopeThreads, smem);
    if (occ != cudaSuccess) return occ;
    const long long slots = static_cast<long long>(sm_count()) * (perSm > 0 ? perSm : 1);
    const unsigned grid = static_cast<unsigned>(T < slots ? T : slots);
    kernel<<<grid, kRopeThreads, smem, st>>>(a, T);
    return cudaGetLastError();
  };
  return p.headDim == 64 ? go(rope_qkv_kernel<64>) : go(rope_qkv_kernel<128>);
}

}  // namespace qsa
