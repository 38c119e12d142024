// qsa_attention.cu -- sparse GQA attention over QSA index lists.
//
//   sparse_prefill_kernel  one CTA per (query token, KV head) over dense padded
//                          BSND Q/K/V ("Cute Dsl Qsa Sparse Runner",
//                          QsaSparsePrefillParams)
//   sparse_decode_kernel   one CTA per (split, KV head, sequence) over the paged
//                          pool, up to 8 splits (fewer when they fit one wave
//                          of CTAs and 8 do not), fp32 partials, and the last
//                          split to finish merges them and resets its counter
//                          (QsaSparseDecodeParams, kMaxSplits = 8,
//                          kPartialRows = 16)
//
// Both stream the K/V rows named by the list through a cp.async ring in shared
// memory (16-byte copies, one 256-byte row per key, zero-filled for skipped
// entries).  The GQA head group is one MMA operand: each warp takes 16 keys of
// a 64-key tile and computes S^T = K Q^T with the keys as the M side and the
// group's heads as N (m16n8k16, no padding of the group to 16 rows), online
// softmax in fp32 (log2 domain), and O^T += V^T P^T with P^T formed from the S
// fragments by an in-register 8x8 transpose.  Warps keep independent running
// (m, l, O) and are merged once at the end.
#include <algorithm>
#include <atomic>

#include "qsa_device.cuh"
#include "qsa_internal.h"
#include "qsa_tcgen05.cuh"

namespace qsa {
namespace {

constexpr int kThreads = 128;  // 4 warps
constexpr int kKeys = 64;      // keys per tile (16 per warp)
constexpr int kD = 128;        // attention head dim
constexpr int kTileBytes = kKeys * kD * 2;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kOStride = 132;  // padded fp32 row of the warp-merge buffer

// Byte offset of 16-byte chunk `c` of row `r` in a [rows][256 B] tile (XOR swizzle
// over 8-row groups so ldmatrix reads are bank-conflict free).
__device__ __forceinline__ uint32_t swz(int r, int c) { return r * 256 + ((c ^ (r & 7)) << 4); }
// K and V tiles: two planes of 64 rows x 128 bytes (dims 0..63, then 64..127),
// chunk c & 7 of row r at 16-byte slot (c & 7) ^ (r & 7) of its 128-byte row;
// 8 consecutive rows of one chunk sit in 8 different bank groups.
__device__ __forceinline__ uint32_t kv_off(int r, int c) {
  return (c >> 3) * (kKeys * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// The element type of Q/K/V/O: fp16, or bf16 (kBf16).  Copies move the 16-bit
// values as they are; only the MMA, the rounding of P and the output differ.
template <bool kBf16>
__device__ __forceinline__ void mma_tile(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (kBf16)
    mma16816_bf16(d, a, b0, b1);
  else
    mma16816(d, a, b0, b1);
}
template <bool kBf16>
__device__ __forceinline__ uint32_t pack_p(float lo, float hi) {
  return kBf16 ? pack_bf162(lo, hi) : pack_half2(lo, hi);
}
template <bool kBf16>
__device__ __forceinline__ void store_pair(__half* dst, float x, float y) {
  *reinterpret_cast<uint32_t*>(dst) = pack_p<kBf16>(x, y);
}

// 2^x by the hardware approximation, results below the normal range flushed
// to zero (probabilities that small do not change an fp16 output).
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

template <int NT>
struct WarpAcc {
  float o[8][NT][4];  // O^T fragments: dims 16*mt + (g, g+8), heads 8*nt + (2q, 2q+1)
  float m[NT][2];     // running max (log2 units) of heads 8*nt + 2q, 8*nt + 2q + 1
  float l[NT][2];     // this thread's share of the running sum
};

template <int NT>
__device__ __forceinline__ void acc_init(WarpAcc<NT>& A) {
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) A.o[mt][nt][i] = 0.f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    A.m[nt][0] = A.m[nt][1] = -INFINITY;
    A.l[nt][0] = A.l[nt][1] = 0.f;
  }
}

// Q^T B-fragments of all 8 k-steps (128 dims) from the swizzled Q tile.
template <int NT>
__device__ __forceinline__ void load_q_frags(uint32_t q_tile, uint32_t (&qf)[NT][8][2]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int ks = 0; ks < 8; ks += 2) {
      const int row = 8 * nt + (lane & 7);
      const int chunk = 2 * ks + (lane >> 3);
      ldsm_x4(q_tile + swz(row, chunk), qf[nt][ks][0], qf[nt][ks][1], qf[nt][ks + 1][0], qf[nt][ks + 1][1]);
    }
}

// One warp, 16 keys (tile rows 16*warp ..): S^T = K Q^T, online softmax, O^T += V^T P^T.
template <int NT, bool kBf16>
__device__ __forceinline__ void attend16(WarpAcc<NT>& A, uint32_t k_tile, uint32_t v_tile,
                                         const uint32_t (&qf)[NT][8][2], bool valid0, bool valid1, float sl2) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int kr0 = warp * 16;
  const int mi = lane >> 3;
  float s[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    uint32_t a[4];
    ldsm_x4(k_tile + kv_off(kr0 + (lane & 7) + 8 * (mi & 1), 2 * ks + (mi >> 1)), a[0], a[1], a[2], a[3]);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mma_tile<kBf16>(s[nt], a, qf[nt][ks][0], qf[nt][ks][1]);
  }
  uint32_t pb[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const float x0 = valid0 ? s[nt][0] * sl2 : -INFINITY;  // key g,   head 2q
    const float x1 = valid0 ? s[nt][1] * sl2 : -INFINITY;  // key g,   head 2q+1
    const float x2 = valid1 ? s[nt][2] * sl2 : -INFINITY;  // key g+8, head 2q
    const float x3 = valid1 ? s[nt][3] * sl2 : -INFINITY;  // key g+8, head 2q+1
    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, o));
    }
    const float mn0 = fmaxf(A.m[nt][0], mx0), mn1 = fmaxf(A.m[nt][1], mx1);
    const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = ex2_ftz(A.m[nt][0] - mu0), al1 = ex2_ftz(A.m[nt][1] - mu1);
    A.m[nt][0] = mn0;
    A.m[nt][1] = mn1;
    const float p0 = ex2_ftz(x0 - mu0), p1 = ex2_ftz(x1 - mu1), p2 = ex2_ftz(x2 - mu0), p3 = ex2_ftz(x3 - mu1);
    A.l[nt][0] = A.l[nt][0] * al0 + (p0 + p2);
    A.l[nt][1] = A.l[nt][1] * al1 + (p1 + p3);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      A.o[mt][nt][0] *= al0;
      A.o[mt][nt][1] *= al1;
      A.o[mt][nt][2] *= al0;
      A.o[mt][nt][3] *= al1;
    }
    pb[nt][0] = movmatrix_t(pack_p<kBf16>(p0, p1));  // keys 0..7  -> (k = 2q..2q+1, n = g)
    pb[nt][1] = movmatrix_t(pack_p<kBf16>(p2, p3));  // keys 8..15
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    uint32_t a[4];
    ldsm_x4_t(v_tile + kv_off(kr0 + (lane & 7) + 8 * (mi >> 1), 2 * mt + (mi & 1)), a[0], a[1], a[2], a[3]);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mma_tile<kBf16>(A.o[mt][nt], a, pb[nt][0], pb[nt][1]);
  }
}

// Writes each warp's (m, l, O^T) to shared memory: mw/lw [4][16], ow [4][16][kOStride].
template <int NT>
__device__ __forceinline__ void stash_warp(const WarpAcc<NT>& A, float* mw, float* lw, float* ow) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float l = A.l[nt][j];
      l += __shfl_xor_sync(kFull, l, 4);
      l += __shfl_xor_sync(kFull, l, 8);
      l += __shfl_xor_sync(kFull, l, 16);
      if (g == 0) {
        mw[warp * 16 + 8 * nt + 2 * q + j] = A.m[nt][j];
        lw[warp * 16 + 8 * nt + 2 * q + j] = l;
      }
    }
  float* o = ow + warp * 16 * kOStride;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int h = 8 * nt + 2 * q, d = 16 * mt + g;
      o[h * kOStride + d] = A.o[mt][nt][0];
      o[(h + 1) * kOStride + d] = A.o[mt][nt][1];
      o[h * kOStride + d + 8] = A.o[mt][nt][2];
      o[(h + 1) * kOStride + d + 8] = A.o[mt][nt][3];
    }
}

// Merged (M, L) of one head over the 4 warps, and the warps' weights 2^(m_w - M).
__device__ __forceinline__ float merge_weights(const float* mw, const float* lw, int h, float (&f)[4], float& L) {
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < 4; ++w) M = fmaxf(M, mw[w * 16 + h]);
  L = 0.f;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float m = mw[w * 16 + h];
    f[w] = m == -INFINITY ? 0.f : exp2f(m - M);
    L += f[w] * lw[w * 16 + h];
  }
  return M;
}

// ------------------------------------------------------------------ prefill
// The staged list is permuted within each 64-key tile so that the 8 rows one
// gathering thread copies (keys 8r + c, r < 8, for its row-in-group c) sit in 8
// consecutive ints: slot 8c + r of the tile holds key 8r + c.
__device__ __forceinline__ int perm_slot(int i) {
  const int k = i & (kKeys - 1);
  return (i & ~(kKeys - 1)) | ((k & 7) << 3) | (k >> 3);
}

struct PrefillArgs {
  const __half* q;
  const __half* k;
  const __half* v;
  __half* o;
  const int32_t* indices;
  const int32_t* ctx;
  int32_t* status;  // optional error word
  int S, Hq, Hkv, G, topK, topKpad;
  float sl2;  // attentionScale * log2(e)
};

template <int NT, int STAGES, bool kBf16>
__global__ void __launch_bounds__(kThreads, STAGES == 1 ? 5 : 3) sparse_prefill_kernel(const PrefillArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t ring = smem_addr(smem);                       // [STAGES][K 16 KB | V 16 KB]
  const uint32_t q_tile = ring + STAGES * 2 * kTileBytes;      // [8*NT][256 B]
  int* idx_s = reinterpret_cast<int*>(smem + STAGES * 2 * kTileBytes + NT * 8 * 256);
  uint32_t* vmask = reinterpret_cast<uint32_t*>(idx_s + a.topKpad);  // bit k of word w: slot 32 w + k is valid
  int* misc = reinterpret_cast<int*>(vmask + a.topKpad / 32);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Within a sequence the CTAs run the rows from the last position down: the
  // longest lists start first and the sequence ends on short ones.  Sequences
  // follow one another, so one sequence's K/V is the L2 working set.
  const long long bid = blockIdx.x;
  const int kvh = static_cast<int>(bid % a.Hkv);
  const long long rowid = bid / a.Hkv;
  const int b = static_cast<int>(rowid / a.S);
  const int t = a.S - 1 - static_cast<int>(rowid % a.S);
  const long long bt = static_cast<long long>(b) * a.S + t;
  const int L = max(0, min(a.ctx[b], a.S));
  __half* out = a.o + (static_cast<size_t>(bt) * a.Hq + static_cast<size_t>(kvh) * a.G) * kD;
  if (t >= L) {  // rows at or past the live length are exact zeros
    for (int e = tid; e < a.G * kD / 8; e += kThreads) reinterpret_cast<uint4*>(out)[e] = make_uint4(0, 0, 0, 0);
    return;
  }
  // Q rows of the group (rows >= G zero), copied while the list is staged.
  const __half* qsrc = a.q + (static_cast<size_t>(bt) * a.Hq + static_cast<size_t>(kvh) * a.G) * kD;
  for (int e = tid; e < NT * 8 * 16; e += kThreads) {
    const int r = e >> 4, c = e & 15;
    const bool ok = r < a.G;
    cp_async16(q_tile + swz(r, c), qsrc + (ok ? r : 0) * kD + c * 8, ok);
  }
  cp_async_commit();
  // Stage the list, eight loads per thread in flight; entries outside [0, L) are skipped.
  const int32_t* lst = a.indices + static_cast<size_t>(bt) * a.topK;
  int last = -1;
  bool bad = false;
  for (int i0 = tid; i0 < a.topKpad; i0 += 8 * kThreads) {
    int jv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * kThreads;
      jv[u] = i < a.topK ? __ldg(lst + i) : -1;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * kThreads;
      if (i < a.topKpad) {
        const bool ok = static_cast<unsigned>(jv[u]) < static_cast<unsigned>(L);
        idx_s[perm_slot(i)] = ok ? jv[u] : -1;
        const unsigned m = __ballot_sync(kFull, ok);  // the warp holds 32 consecutive slots
        if (lane == 0) vmask[i >> 5] = m;
        last = ok ? i : last;
        bad |= !ok && jv[u] != -1;
      }
    }
  }
  if (__any_sync(kFull, bad) && lane == 0 && a.status) atomicOr(a.status, kErrBadIndex);
  last = __reduce_max_sync(kFull, last);
  if (lane == 0) misc[warp] = last;
  __syncthreads();
  const int nslots = max(max(misc[0], misc[1]), max(misc[2], misc[3])) + 1;
  const int ntiles = (nslots + kKeys - 1) / kKeys;

  // 16 consecutive lanes copy one 256-byte row, so every warp instruction reads
  // whole 128-byte lines (two rows of K, then the same two rows of V).  A
  // thread's chunk, its sequence, head and swizzled slot are fixed, so a key
  // costs one offset multiply-add from the per-thread bases.
  const int ch = tid & 15;
  const size_t head_off = (static_cast<size_t>(b) * a.S * a.Hkv + kvh) * kD + ch * 8;
  const __half* kbase = a.k + head_off;
  const __half* vbase = a.v + head_off;
  const int tok_stride = a.Hkv * kD;                   // elements between consecutive tokens
  const uint32_t slot0 = kv_off(tid >> 4, ch);        // key r*8 + tid/16 sits at slot0 + r * 1024
  auto issue = [&](int tile, int stage) {
    const uint32_t kdst = ring + stage * 2 * kTileBytes + slot0;
    const uint32_t vdst = kdst + kTileBytes;
    const int4* ids4 = reinterpret_cast<const int4*>(idx_s + tile * kKeys + (tid >> 4) * 8);
    const int4 i0 = ids4[0], i1 = ids4[1];
    const int idv[8] = {i0.x, i0.y, i0.z, i0.w, i1.x, i1.y, i1.z, i1.w};
#pragma unroll
    for (int r = 0; r < kKeys / 8; ++r) {
      const int j = idv[r];
      const bool ok = j >= 0;
      const size_t off = static_cast<size_t>(ok ? j : 0) * tok_stride;
      cp_async16(kdst + r * 8 * 128, kbase + off, ok);
      cp_async16(vdst + r * 8 * 128, vbase + off, ok);
    }
  };
  uint32_t qf[NT][8][2];
  WarpAcc<NT> A;
  acc_init(A);
  if constexpr (STAGES == 1) {
    // One tile in shared memory per CTA: a small CTA (42 KB), so 5 share an
    // SM and each one's gather latency is covered by the others' arithmetic.
    cp_async_wait<0>();  // Q
    __syncthreads();
    load_q_frags<NT>(q_tile, qf);
    for (int i = 0; i < ntiles; ++i) {
      __syncthreads();  // every warp is done with tile i-1
      issue(i, 0);
      cp_async_commit();
      cp_async_wait<0>();
      __syncthreads();
      const uint2 vm = *reinterpret_cast<const uint2*>(vmask + 2 * i);  // the tile's 64 validity bits
      const int k0 = warp * 16 + (lane >> 2);
      const uint32_t w0 = k0 < 32 ? vm.x : vm.y, w1 = k0 + 8 < 32 ? vm.x : vm.y;
      attend16<NT, kBf16>(A, ring, ring + kTileBytes, qf, (w0 >> (k0 & 31)) & 1u, (w1 >> ((k0 + 8) & 31)) & 1u,
                          a.sl2);
    }
  } else {
#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
      if (s < ntiles) issue(s, s);
      cp_async_commit();
    }
    cp_async_wait<STAGES - 1>();  // the Q group (oldest) has landed
    __syncthreads();
    load_q_frags<NT>(q_tile, qf);
    for (int i = 0; i < ntiles; ++i) {
      cp_async_wait<STAGES - 2>();
      __syncthreads();
      if (i + STAGES - 1 < ntiles) issue(i + STAGES - 1, (i + STAGES - 1) % STAGES);
      cp_async_commit();
      const int stage = i % STAGES;
      const uint2 vm = *reinterpret_cast<const uint2*>(vmask + 2 * i);
      const int k0 = warp * 16 + (lane >> 2);
      const uint32_t w0 = k0 < 32 ? vm.x : vm.y, w1 = k0 + 8 < 32 ? vm.x : vm.y;
      attend16<NT, kBf16>(A, ring + stage * 2 * kTileBytes, ring + stage * 2 * kTileBytes + kTileBytes, qf,
                   (w0 >> (k0 & 31)) & 1u, (w1 >> ((k0 + 8) & 31)) & 1u, a.sl2);
    }
  }
  cp_async_wait<0>();
  __syncthreads();
  float* mw = reinterpret_cast<float*>(smem);
  float* lw = mw + 64;
  float* ow = lw + 64;
  stash_warp<NT>(A, mw, lw, ow);
  __syncthreads();
  for (int e = tid; e < a.G * (kD / 2); e += kThreads) {
    const int h = e / (kD / 2), d = 2 * (e % (kD / 2));
    float f[4], Lsum;
    merge_weights(mw, lw, h, f, Lsum);
    float o0 = 0.f, o1 = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      o0 += f[w] * ow[(w * 16 + h) * kOStride + d];
      o1 += f[w] * ow[(w * 16 + h) * kOStride + d + 1];
    }
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    store_pair<kBf16>(out + h * kD + d, o0 * inv, o1 * inv);
  }
}

// ------------------------------------------------------------------- decode
struct DecodeArgs {
  const __half* q;
  const __half* pool;
  const int32_t* pageTable;
  const int32_t* indices;
  const int32_t* ctx;
  __half* o;
  float* partialO;
  float* partialStats;
  int32_t* counters;
  int32_t* status;  // optional error word
  int Hq, Hkv, G, poolHeadDim, numFlatPages, maxPagesPerSeq, topK;
  int nsplit;                     // slices per (sequence, KV head), 1..kMaxSplits
  int tilesPerSplit, extraTiles;  // split s owns tilesPerSplit (+1 for s < extraTiles) whole 64-key tiles
  int slicePad;                   // slots of the longest slice
  float sl2;
};

template <int NT, int STAGES, bool kBf16>
__global__ void __launch_bounds__(kThreads, STAGES == 1 ? 5 : 3) sparse_decode_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t ring = smem_addr(smem);
  const uint32_t q_tile = ring + STAGES * 2 * kTileBytes;
  long long* kofs = reinterpret_cast<long long*>(smem + STAGES * 2 * kTileBytes + NT * 8 * 256);
  long long* vofs = kofs + a.slicePad;
  int* misc = reinterpret_cast<int*>(vofs + a.slicePad);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int L = max(0, min(a.ctx[b], a.maxPagesPerSeq * kTokensPerPage));
  // Slices are whole 64-key tiles of the list, so no split ends on a nearly
  // empty tile: the ceil(topK / 64) tiles are dealt out evenly, the first
  // extraTiles splits taking one more.
  const int s0 = kKeys * (split * a.tilesPerSplit + min(split, a.extraTiles));
  const int s1 = min(a.topK, s0 + kKeys * (a.tilesPerSplit + (split < a.extraTiles ? 1 : 0)));
  const int32_t* lst = a.indices + static_cast<size_t>(b) * a.topK;
  const int32_t* ptK = a.pageTable + static_cast<size_t>(b) * 2 * a.maxPagesPerSeq;
  const int32_t* ptV = ptK + a.maxPagesPerSeq;
  // Resolve the slice's entries to pool offsets, four per thread per pass with
  // their list loads, then their page-table loads, in flight together.
  int last = -1, bad = 0;
  for (int i0 = tid; i0 < a.slicePad; i0 += 4 * kThreads) {
    int jv[4], kp[4], vp[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int slot = s0 + i0 + u * kThreads;
      jv[u] = i0 + u * kThreads < a.slicePad && slot < s1 ? __ldg(lst + slot) : -1;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool live = static_cast<unsigned>(jv[u]) < static_cast<unsigned>(L);
      kp[u] = live ? __ldg(ptK + (jv[u] >> 7)) : -1;
      vp[u] = live ? __ldg(ptV + (jv[u] >> 7)) : -1;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * kThreads;
      if (i >= a.slicePad) continue;
      const int j = jv[u];
      const bool ok = static_cast<unsigned>(j) < static_cast<unsigned>(L) &&
                      static_cast<unsigned>(kp[u]) < static_cast<unsigned>(a.numFlatPages) &&
                      static_cast<unsigned>(vp[u]) < static_cast<unsigned>(a.numFlatPages);
      const long long within = static_cast<long long>((j & 127) * a.Hkv + kvh) * a.poolHeadDim;
      kofs[perm_slot(i)] = ok ? static_cast<long long>(kp[u]) * kTokensPerPage * a.Hkv * a.poolHeadDim + within : -1;
      vofs[perm_slot(i)] = ok ? static_cast<long long>(vp[u]) * kTokensPerPage * a.Hkv * a.poolHeadDim + within : -1;
      last = ok ? i : last;
      const bool live = static_cast<unsigned>(j) < static_cast<unsigned>(L);
      bad |= !live && j != -1 ? kErrBadIndex : 0;
      bad |= live && !ok ? kErrBadPage : 0;
    }
  }
  bad = __reduce_or_sync(kFull, static_cast<unsigned>(bad));
  if (bad && lane == 0 && a.status) atomicOr(a.status, bad);
  last = __reduce_max_sync(kFull, last);
  if (lane == 0) misc[warp] = last;
  const __half* qsrc = a.q + (static_cast<size_t>(b) * a.Hq + static_cast<size_t>(kvh) * a.G) * kD;
  for (int e = tid; e < NT * 8 * 16; e += kThreads) {
    const int r = e >> 4, c = e & 15;
    const bool ok = r < a.G;
    cp_async16(q_tile + swz(r, c), qsrc + (ok ? r : 0) * kD + c * 8, ok);
  }
  cp_async_commit();
  __syncthreads();
  const int nslots = max(max(misc[0], misc[1]), max(misc[2], misc[3])) + 1;
  const int ntiles = (nslots + kKeys - 1) / kKeys;

  auto issue = [&](int tile, int stage) {  // one 256-byte row per 16 lanes, as in prefill
    const uint32_t kdst = ring + stage * 2 * kTileBytes;
    const uint32_t vdst = kdst + kTileBytes;
    const int ch = tid & 15;
    // this thread's 8 rows (keys 8r + tid/16) sit in 8 consecutive slots of the permuted offsets
    const longlong2* k2 = reinterpret_cast<const longlong2*>(kofs + tile * kKeys + (tid >> 4) * 8);
    const longlong2* v2 = reinterpret_cast<const longlong2*>(vofs + tile * kKeys + (tid >> 4) * 8);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {  // rows 4 hf .. 4 hf + 3: four offsets of each kind live at a time
      const longlong2 ka = k2[2 * hf], kb = k2[2 * hf + 1], va = v2[2 * hf], vb = v2[2 * hf + 1];
      const long long kov[4] = {ka.x, ka.y, kb.x, kb.y}, vov[4] = {va.x, va.y, vb.x, vb.y};
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int key = (4 * hf + rr) * 8 + (tid >> 4);
        const long long ko = kov[rr], vo = vov[rr];
        const bool ok = ko >= 0;
        cp_async16(kdst + kv_off(key, ch), a.pool + (ok ? ko : 0) + ch * 8, ok);
        cp_async16(vdst + kv_off(key, ch), a.pool + (ok ? vo : 0) + ch * 8, ok);
      }
    }
  };
  uint32_t qf[NT][8][2];
  WarpAcc<NT> A;
  acc_init(A);
  if constexpr (STAGES == 1) {  // one tile per CTA, 5 CTAs per SM (as in prefill)
    if (ntiles > 0) issue(0, 0);  // the first tile's copies travel with Q's
    cp_async_commit();
    cp_async_wait<1>();  // Q
    __syncthreads();
    load_q_frags<NT>(q_tile, qf);
    for (int i = 0; i < ntiles; ++i) {
      if (i > 0) {
        __syncthreads();  // every warp is done with tile i-1
        issue(i, 0);
        cp_async_commit();
      }
      cp_async_wait<0>();
      __syncthreads();
      const int slot = i * kKeys + warp * 16 + (lane >> 2);
      attend16<NT, kBf16>(A, ring, ring + kTileBytes, qf, kofs[perm_slot(slot)] >= 0,
                          kofs[perm_slot(slot + 8)] >= 0, a.sl2);
    }
  } else {
#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
      if (s < ntiles) issue(s, s);
      cp_async_commit();
    }
    cp_async_wait<STAGES - 1>();
    __syncthreads();
    load_q_frags<NT>(q_tile, qf);
    for (int i = 0; i < ntiles; ++i) {
      cp_async_wait<STAGES - 2>();
      __syncthreads();
      if (i + STAGES - 1 < ntiles) issue(i + STAGES - 1, (i + STAGES - 1) % STAGES);
      cp_async_commit();
      const int stage = i % STAGES;
      const int slot = i * kKeys + warp * 16 + (lane >> 2);
      attend16<NT, kBf16>(A, ring + stage * 2 * kTileBytes, ring + stage * 2 * kTileBytes + kTileBytes, qf,
                   kofs[perm_slot(slot)] >= 0, kofs[perm_slot(slot + 8)] >= 0, a.sl2);
    }
  }
  cp_async_wait<0>();
  __syncthreads();
  float* mw = reinterpret_cast<float*>(smem);
  float* lw = mw + 64;
  float* ow = lw + 64;
  stash_warp<NT>(A, mw, lw, ow);
  __syncthreads();

  // This split's partial: O unnormalised relative to its max M, stats (M, L).
  const size_t part = (static_cast<size_t>(b) * a.Hkv + kvh) * kMaxSplits + split;
  float* pO = a.partialO + part * kPartialRows * kD;
  float* pS = a.partialStats + part * 2 * kPartialRows;
  // Only the group's G rows are written; the combine reads no others.
  for (int e = tid; e < a.G * (kD / 2); e += kThreads) {
    const int h = e / (kD / 2), d = 2 * (e % (kD / 2));
    float f[4], Lsum;
    const float M = merge_weights(mw, lw, h, f, Lsum);
    float o0 = 0.f, o1 = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      o0 += f[w] * ow[(w * 16 + h) * kOStride + d];
      o1 += f[w] * ow[(w * 16 + h) * kOStride + d + 1];
    }
    reinterpret_cast<float2*>(pO + h * kD)[d / 2] = make_float2(o0, o1);
    if (d == 0) {
      pS[h] = M;
      pS[kPartialRows + h] = Lsum;
    }
  }
  // Last split to arrive merges the nsplit partials and re-arms the counter.
  __threadfence();
  __syncthreads();
  if (tid == 0) misc[4] = atomicAdd(a.counters + b * a.Hkv + kvh, 1) == a.nsplit - 1;
  __syncthreads();
  if (!misc[4]) return;
  __threadfence();
  const float* pO0 = a.partialO + (static_cast<size_t>(b) * a.Hkv + kvh) * kMaxSplits * kPartialRows * kD;
  const float* pS0 = a.partialStats + (static_cast<size_t>(b) * a.Hkv + kvh) * kMaxSplits * 2 * kPartialRows;
  __half* out = a.o + (static_cast<size_t>(b) * a.Hq + static_cast<size_t>(kvh) * a.G) * kD;
  for (int e = tid; e < a.G * (kD / 2); e += kThreads) {
    const int h = e / (kD / 2), d = 2 * (e % (kD / 2));
    // Every slot's loads are issued unconditionally (slots past nsplit re-read
    // the last one and are weighted 0), so they are all in flight together.
    float m[kMaxSplits];
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s) {
      const float v = __ldcg(pS0 + min(s, a.nsplit - 1) * 2 * kPartialRows + h);
      m[s] = s < a.nsplit ? v : -INFINITY;
    }
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s) M = fmaxf(M, m[s]);
    float Lsum = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s) {
      const int sc = min(s, a.nsplit - 1);
      const float f = m[s] == -INFINITY ? 0.f : exp2f(m[s] - M);
      Lsum += f * __ldcg(pS0 + sc * 2 * kPartialRows + kPartialRows + h);
      const float2 ov = __ldcg(reinterpret_cast<const float2*>(pO0 + (sc * kPartialRows + h) * kD + d));
      o0 += f * ov.x;
      o1 += f * ov.y;
    }
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    store_pair<kBf16>(out + h * kD + d, o0 * inv, o1 * inv);
  }
  if (tid == 0) a.counters[b * a.Hkv + kvh] = 0;
}


// ------------------------------------------------- prefill on tcgen05 / TMEM
// The same contract as sparse_prefill_kernel, with S = q.k on the
// 5th-generation tensor cores.  One CTA of 4 warps (one warpgroup, TMEM lanes
// 0..127) per (query token, KV head); tiles of 64 keys.  Per tile:
//   - the K and V rows the list names are gathered (16 lanes per 256-byte row,
//     cp.async, zero-filled for skipped entries) into two 16 KB tiles in the
//     SW128 layout, the 128 dims of a row split into two 64-dim halves;
//   - one thread issues S^T = K Q^T (M = 64 keys, N = 8 heads, eight MMAs of
//     16 dims, both operands read from shared memory by descriptor) into TMEM
//     and commits it to an mbarrier: no thread loads K into registers;
//   - an M = 64 accumulator puts key 16w + l in lane l of warp w's quadrant,
//     so warp w reads the scores of exactly its 16 keys (tcgen05.ld) and runs
//     its own online softmax over them, as the mma.sync kernel's warps do:
//     a warp max per head (redux on order-preserving integers), rescale, P
//     rounded to the element type and stored as 16-byte rows [key][8 heads];
//   - the warp multiplies P into V with mma.sync (O^T += V^T P^T, V^T by
//     ldmatrix.trans from the SW128 tile, P^T by ldmatrix.trans), keeping
//     (m, l, O) in registers; the four warps merge once at the end.
// Per gathered byte shared memory sees the cp.async write and the V read,
// not the K read.  A CTA needs 37 KB, so six share an SM.  A head group of
// 9..16 runs as two groups of 8.
constexpr int kTcKeys = 64;
constexpr int kTcHalf = kTcKeys * 128;          // bytes of one 64-dim half of a tile (8 KB)
constexpr int kTcTile = 2 * kTcHalf;            // 16 KB
constexpr uint64_t kTcWaitNs = 200ull * 1000 * 1000;

template <int NT>
constexpr size_t tc_prefill_smem() {  // + 1 KB to align the base to 1024 bytes
  return 1024 + 2 * kTcTile + NT * 2048 /*Q*/ + 4 * NT * 256 /*P per warp*/ + 64 /*barrier, TMEM slot, counts*/;
}

// Order-preserving map between fp32 and int32 (and back).
__device__ __forceinline__ int f2ord(float x) {
  const int i = __float_as_int(x);
  return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float ord2f(int o) { return __int_as_float(o >= 0 ? o : o ^ 0x7fffffff); }

// The tcgen05 tiles use the same two-plane SW128 layout as the mma.sync kernels (kv_off, kTcKeys == kKeys).
static_assert(kTcKeys == kKeys && kTcHalf == kKeys * 128, "one K/V tile layout for both prefill kernels");

template <int NT, bool kBf16>
__global__ void __launch_bounds__(kThreads, NT == 1 ? 6 : 5) sparse_prefill_tc_kernel(const PrefillArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  uint8_t* base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t kt = smem_addr(base);               // K tile [2 halves][64 keys][128 B], SW128
  const uint32_t vt = kt + kTcTile;                  // V tile, same layout
  const uint32_t qt = vt + kTcTile;                  // Q: NT x [2 halves][8 heads][128 B], SW128
  const uint32_t pt = qt + NT * 2048;                // P: [4 warps][NT][16 keys][8 heads] (16 B rows)
  uint64_t* bar = reinterpret_cast<uint64_t*>(base + 2 * kTcTile + NT * 2048 + 4 * NT * 256);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
  int* misc = reinterpret_cast<int*>(tslot + 1);     // [4] last valid slot per warp

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long bid = blockIdx.x;
  const int kvh = static_cast<int>(bid % a.Hkv);
  const long long rowid = bid / a.Hkv;
  const int b = static_cast<int>(rowid / a.S);
  const int t = a.S - 1 - static_cast<int>(rowid % a.S);  // longest lists first within a sequence
  const long long bt = static_cast<long long>(b) * a.S + t;
  const int L = max(0, min(a.ctx[b], a.S));
  __half* out = a.o + (static_cast<size_t>(bt) * a.Hq + static_cast<size_t>(kvh) * a.G) * kD;
  if (t >= L) {  // rows at or past the live length are exact zeros
    for (int e = tid; e < a.G * kD / 8; e += kThreads) reinterpret_cast<uint4*>(out)[e] = make_uint4(0, 0, 0, 0);
    return;
  }
  // Q rows of the group (heads >= G zero), in the SW128 K-major layout.
  const __half* qsrc = a.q + (static_cast<size_t>(bt) * a.Hq + static_cast<size_t>(kvh) * a.G) * kD;
  for (int e = tid; e < NT * 8 * 16; e += kThreads) {
    const int h = e >> 4, c = e & 15, hr = h & 7;
    const bool ok = h < a.G;
    cp_async16(qt + (h >> 3) * 2048 + (c >> 3) * 1024 + hr * 128 + (((c & 7) ^ hr) << 4), qsrc + (ok ? h : 0) * kD + c * 8,
               ok);
  }
  cp_async_commit();
  // The list's last valid slot fixes the tile count (entries outside [0, L) are skipped).
  const int32_t* lst = a.indices + static_cast<size_t>(bt) * a.topK;
  int last = -1;
  bool bad = false;
  for (int i = tid; i < a.topK; i += kThreads) {
    const int j = __ldg(lst + i);
    const bool ok = static_cast<unsigned>(j) < static_cast<unsigned>(L);
    last = ok ? i : last;
    bad |= !ok && j != -1;
  }
  if (__any_sync(kFull, bad) && lane == 0 && a.status) atomicOr(a.status, kErrBadIndex);
  last = __reduce_max_sync(kFull, last);
  if (lane == 0) misc[warp] = last;
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(tslot, 32);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;  // columns [0, 8 NT): this tile's S^T
  const int nslots = max(max(misc[0], misc[1]), max(misc[2], misc[3])) + 1;
  const int ntiles = (nslots + kTcKeys - 1) / kTcKeys;

  // Gathers: 16 lanes per 256-byte row, rows r*8 + tid/16 (r < 8); the chunk's
  // swizzled slot depends only on the thread.  A tile's row ids are loaded
  // one tile ahead and serve both the K and the V copies.
  const int ch = tid & 15, rsub = tid >> 4;
  const size_t head_off = (static_cast<size_t>(b) * a.S * a.Hkv + kvh) * kD + ch * 8;
  const __half* kbase = a.k + head_off;
  const __half* vbase = a.v + head_off;
  const int tok_stride = a.Hkv * kD;
  const uint32_t slot0 = kv_off(rsub, ch);
  int rows[kTcKeys / 8];  // token ids of this thread's rows of a tile, -1 when skipped
  int key_id;             // lanes 0..15: the id of key 16 w + lane of a tile
  auto load_ids = [&](int tile) {
#pragma unroll
    for (int r = 0; r < kTcKeys / 8; ++r) {
      const int slot = tile * kTcKeys + r * 8 + rsub;
      const int j = slot < a.topK ? __ldg(lst + slot) : -1;
      rows[r] = static_cast<unsigned>(j) < static_cast<unsigned>(L) ? j : -1;
    }
    const int ks = tile * kTcKeys + 16 * warp + (lane & 15);
    key_id = ks < a.topK ? __ldg(lst + ks) : -1;
  };
  auto issue = [&]() {
#pragma unroll
    for (int r = 0; r < kTcKeys / 8; ++r) {
      const size_t off = static_cast<size_t>(rows[r] >= 0 ? rows[r] : 0) * tok_stride;
      cp_async16(kt + slot0 + r * 1024, kbase + off, rows[r] >= 0);
      cp_async16(vt + slot0 + r * 1024, vbase + off, rows[r] >= 0);
    }
  };

  const float sl2 = a.sl2;
  const int g = lane >> 2, q = lane & 3, mi = lane >> 3;
  float o[8][NT][4];  // O^T fragments: dims 16*mt + (g, g+8), heads 8*nt + (2q, 2q+1)
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) o[mt][nt][i] = 0.f;
  float m_run[NT][8], l_part[NT][8];  // per warp (uniform) running max; this lane's key's share of l
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      m_run[nt][h] = -INFINITY;
      l_part[nt][h] = 0.f;
    }
  const uint32_t lane_addr = static_cast<uint32_t>(32 * warp) << 16;
  const uint32_t pw = pt + warp * NT * 256;  // this warp's P rows
  // A wait that runs out (a tensor-core fault) records a status bit; every
  // exit from the loop is decided at a barrier, so all threads leave together.
  bool ok = true, alive = true;
  if (ntiles > 0) {
    load_ids(0);
    issue();
  }
  cp_async_commit();
  for (int i = 0; i < ntiles; ++i) {
    const int my_key = key_id;
    cp_async_wait<0>();
    fence_proxy_async();  // cp.async writes -> the tensor cores' reads
    tc_fence_before();
    if (__syncthreads_or(!ok)) {
      alive = false;
      break;
    }
    tc_fence_after();
    if (tid == 0) {
      constexpr uint32_t idS = mma_idesc_f16(64, 8, kBf16, false, false);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint32_t koff = (s >> 2) * kTcHalf + (s & 3) * 32;
          umma_f16(tmem + nt * 8, smem_desc(kt + koff, 16, 1024, kSmemSwizzle128B),
                   smem_desc(qt + nt * 2048 + (s >> 2) * 1024 + (s & 3) * 32, 16, 1024, kSmemSwizzle128B), idS, s > 0);
        }
      umma_commit(bar);
    }
    __syncwarp();
    if (i + 1 < ntiles) load_ids(i + 1);  // the next tile's ids travel while S is computed
    ok = mbar_wait_bounded(bar, i & 1, kTcWaitNs);
    if (!ok && a.status) atomicOr(a.status, kErrWaitTimeout);
    tc_fence_after();
    const bool valid = lane < 16 && static_cast<unsigned>(my_key) < static_cast<unsigned>(L);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float sv[8];
      tmem_ld8(tmem + lane_addr + nt * 8, sv);
      float al[8];
      uint32_t pk[4];
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float x = valid ? sv[h] * sl2 : -INFINITY;
        const float tmax = ord2f(__reduce_max_sync(kFull, f2ord(x)));
        const float mn = fmaxf(m_run[nt][h], tmax);
        const float mu = mn == -INFINITY ? 0.f : mn;
        al[h] = ex2_ftz(m_run[nt][h] - mu);
        m_run[nt][h] = mn;
        const float p = ex2_ftz(x - mu);
        l_part[nt][h] = l_part[nt][h] * al[h] + p;
        sv[h] = p;
      }
#pragma unroll
      for (int h = 0; h < 4; ++h) pk[h] = pack_p<kBf16>(sv[2 * h], sv[2 * h + 1]);
      if (lane < 16)
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(pw + nt * 256 + lane * 16), "r"(pk[0]),
                     "r"(pk[1]), "r"(pk[2]), "r"(pk[3])
                     : "memory");
      // rescale this thread's O^T fragments (heads 2q, 2q+1 of group nt)
      const float a0 = q == 0 ? al[0] : q == 1 ? al[2] : q == 2 ? al[4] : al[6];
      const float a1 = q == 0 ? al[1] : q == 1 ? al[3] : q == 2 ? al[5] : al[7];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][nt][0] *= a0;
        o[mt][nt][1] *= a1;
        o[mt][nt][2] *= a0;
        o[mt][nt][3] *= a1;
      }
    }
    __syncwarp();
    uint32_t pb[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) ldsm_x2_t(pw + nt * 256 + (lane & 15) * 16, pb[nt][0], pb[nt][1]);
    // O^T += V^T P^T over the warp's 16 keys (rows 16 w .. 16 w + 15 of the V tile)
    const int kr0 = warp * 16;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      uint32_t av[4];
      ldsm_x4_t(vt + kv_off(kr0 + (lane & 7) + 8 * (mi >> 1), 2 * mt + (mi & 1)), av[0], av[1], av[2], av[3]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_tile<kBf16>(o[mt][nt], av, pb[nt][0], pb[nt][1]);
    }
    tc_fence_before();
    __syncthreads();  // every warp is done with the V tile and its P rows; S has been read
    if (i + 1 < ntiles) issue();
    cp_async_commit();
  }
  cp_async_wait<0>();
  alive = alive && __syncthreads_and(ok);
  if (warp == 0) tmem_dealloc(tmem, 32);
  if (!alive) return;
  // Each warp's (m, l, O^T) to shared memory (the tiles are free), then the
  // four warps merge: mw/lw [4][16], ow [4][16][kOStride].
  float* mw = reinterpret_cast<float*>(base);
  float* lw = mw + 64;
  float* ow = lw + 64;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      float v = lane < 16 ? l_part[nt][h] : 0.f;
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
      if (lane == 0) {
        mw[warp * 16 + 8 * nt + h] = m_run[nt][h];
        lw[warp * 16 + 8 * nt + h] = v;
      }
    }
  {
    float* ob = ow + warp * 16 * kOStride;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int h = 8 * nt + 2 * q, d = 16 * mt + g;
        ob[h * kOStride + d] = o[mt][nt][0];
        ob[(h + 1) * kOStride + d] = o[mt][nt][1];
        ob[h * kOStride + d + 8] = o[mt][nt][2];
        ob[(h + 1) * kOStride + d + 8] = o[mt][nt][3];
      }
  }
  __syncthreads();
  for (int e = tid; e < a.G * (kD / 2); e += kThreads) {
    const int h = e / (kD / 2), d = 2 * (e % (kD / 2));
    float f[4], Lsum;
    merge_weights(mw, lw, h, f, Lsum);
    float o0 = 0.f, o1 = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      o0 += f[w] * ow[(w * 16 + h) * kOStride + d];
      o1 += f[w] * ow[(w * 16 + h) * kOStride + d + 1];
    }
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    store_pair<kBf16>(out + h * kD + d, o0 * inv, o1 * inv);
  }
}

// Ring depth of both kernels: one 64-key tile (42 KB of shared memory, 5 CTAs
// per SM, each CTA's gather latency covered by the others) for a head group
// of up to 8; two (3 CTAs per SM, the register budget of the 16-head group)
// otherwise.
template <int NT>
constexpr int kRingStagesFor = NT == 1 ? 1 : 2;

template <int NT>
size_t prefill_smem(int topKpad) {
  return static_cast<size_t>(kRingStagesFor<NT>) * 2 * kTileBytes + NT * 8 * 256 +
         static_cast<size_t>(topKpad) * 4 + topKpad / 8 + 64;
}
template <int NT>
size_t decode_smem(int slicePad) {
  return static_cast<size_t>(kRingStagesFor<NT>) * 2 * kTileBytes + NT * 8 * 256 + static_cast<size_t>(slicePad) * 16 + 64;
}

constexpr int kMaxDynSmem = 227 * 1024;  // per-CTA opt-in limit; the launch asks only for what it uses

template <int NT, bool kBf16>
cudaError_t prefill_nt(const PrefillArgs& a, long long nblocks, cudaStream_t st) {
  const size_t smem = prefill_smem<NT>(a.topKpad);
  static const cudaError_t attr = cudaFuncSetAttribute(sparse_prefill_kernel<NT, kRingStagesFor<NT>, kBf16>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
  if (attr != cudaSuccess) return attr;
  sparse_prefill_kernel<NT, kRingStagesFor<NT>, kBf16><<<static_cast<unsigned>(nblocks), kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

// The list of a (sequence, KV head) is cut into nsplit slices of whole 64-key
// tiles.  nsplit is kMaxSplits unless that grid needs more than one wave of
// resident CTAs and a smaller count fits in one: a CTA's list resolution and
// its partial write take as long as a tile or two, so a second, partial wave
// of short CTAs costs more than longer slices in a single wave.  It is then
// lowered to the fewest slices with the same longest slice (33 tiles: 7
// slices of at most 5 rather than 8), which saves CTAs and partials without
// lengthening any CTA's chain.
template <int NT, bool kBf16>
cudaError_t decode_nt(DecodeArgs a, int B, cudaStream_t st) {
  auto kernel = sparse_decode_kernel<NT, kRingStagesFor<NT>, kBf16>;
  static const cudaError_t attr =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
  if (attr != cudaSuccess) return attr;
  const int tiles = (a.topK + kKeys - 1) / kKeys;  // <= kMaxTiles (the list width is validated)
  auto slice_pad = [&](int ns) { return kKeys * ((tiles + ns - 1) / ns); };
  // Resident CTAs per SM for a slice of n tiles (its list offsets live in
  // shared memory): 0 = not queried yet, -1 = does not fit.
  constexpr int kMaxTiles = 256;
  static std::atomic<int> per_sm[kMaxTiles + 1];
  auto slots = [&](int ns) -> long long {
    const int n = (tiles + ns - 1) / ns;
    if (n > kMaxTiles) return 0;
    int r = per_sm[n].load(std::memory_order_relaxed);
    if (r == 0) {
      const size_t smem = decode_smem<NT>(slice_pad(ns));
      int blocks = 0;
      if (smem > static_cast<size_t>(kMaxDynSmem)) {
        r = -1;
      } else if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kernel, kThreads, smem) != cudaSuccess) {
        (void)cudaGetLastError();  // a failed query is not the launch's error: this count is just not used
        r = -1;
      } else {
        r = blocks < 1 ? -1 : blocks;
      }
      per_sm[n].store(r, std::memory_order_relaxed);
    }
    return r > 0 ? static_cast<long long>(sm_count()) * r : 0;
  };
  const long long pairs = static_cast<long long>(B) * a.Hkv;
  int ns = std::min(kMaxSplits, tiles);
  if (pairs * ns > slots(ns))
    for (int c = ns - 1; c >= 1; --c)
      if (pairs * c <= slots(c)) {
        ns = c;
        break;
      }
  ns = (tiles + (tiles + ns - 1) / ns - 1) / ((tiles + ns - 1) / ns);
  a.nsplit = ns;
  a.tilesPerSplit = tiles / ns;
  a.extraTiles = tiles % ns;
  a.slicePad = slice_pad(ns);
  dim3 grid(ns, a.Hkv, B);
  kernel<<<grid, kThreads, decode_smem<NT>(a.slicePad), st>>>(a);
  return cudaGetLastError();
}

template <int NT, bool kBf16>
cudaError_t prefill_tc_nt(const PrefillArgs& a, long long nblocks, cudaStream_t st) {
  constexpr size_t smem = tc_prefill_smem<NT>();
  static const cudaError_t attr = cudaFuncSetAttribute(sparse_prefill_tc_kernel<NT, kBf16>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (attr != cudaSuccess) return attr;
  sparse_prefill_tc_kernel<NT, kBf16><<<static_cast<unsigned>(nblocks), kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sparse_prefill_tc(const QsaSparsePrefillParams& p, bool bf16) {
  PrefillArgs a;
  a.q = static_cast<const __half*>(p.qPtr);
  a.k = static_cast<const __half*>(p.kPtr);
  a.v = static_cast<const __half*>(p.vPtr);
  a.o = static_cast<__half*>(p.oPtr);
  a.indices = p.indices;
  a.ctx = p.contextLengths;
  a.status = p.status;
  a.S = p.seqLen;
  a.Hq = p.numQHeads;
  a.Hkv = p.numKVHeads;
  a.G = p.numQHeads / p.numKVHeads;
  a.topK = p.topK;
  a.topKpad = (p.topK + kTcKeys - 1) / kTcKeys * kTcKeys;
  a.sl2 = p.attentionScale * kLog2e;
  const long long nblocks = static_cast<long long>(p.batchSize) * p.seqLen * p.numKVHeads;
  cudaStream_t st = static_cast<cudaStream_t>(p.stream);
  if (bf16) return a.G <= 8 ? prefill_tc_nt<1, true>(a, nblocks, st) : prefill_tc_nt<2, true>(a, nblocks, st);
  return a.G <= 8 ? prefill_tc_nt<1, false>(a, nblocks, st) : prefill_tc_nt<2, false>(a, nblocks, st);
}

cudaError_t launch_sparse_prefill(const QsaSparsePrefillParams& p, bool bf16) {
  PrefillArgs a;
  a.q = static_cast<const __half*>(p.qPtr);
  a.k = static_cast<const __half*>(p.kPtr);
  a.v = static_cast<const __half*>(p.vPtr);
  a.o = static_cast<__half*>(p.oPtr);
  a.indices = p.indices;
  a.ctx = p.contextLengths;
  a.status = p.status;
  a.S = p.seqLen;
  a.Hq = p.numQHeads;
  a.Hkv = p.numKVHeads;
  a.G = p.numQHeads / p.numKVHeads;
  a.topK = p.topK;
  a.topKpad = (p.topK + kKeys - 1) / kKeys * kKeys;
  a.sl2 = p.attentionScale * kLog2e;
  const long long nblocks = static_cast<long long>(p.batchSize) * p.seqLen * p.numKVHeads;
  cudaStream_t st = static_cast<cudaStream_t>(p.stream);
  if (bf16) return a.G <= 8 ? prefill_nt<1, true>(a, nblocks, st) : prefill_nt<2, true>(a, nblocks, st);
  return a.G <= 8 ? prefill_nt<1, false>(a, nblocks, st) : prefill_nt<2, false>(a, nblocks, st);
}

cudaError_t launch_sparse_decode(const QsaSparseDecodeParams& p, bool bf16) {
  DecodeArgs a;
  a.q = static_cast<const __half*>(p.qPtr);
  a.pool = static_cast<const __half*>(p.kvPoolPtr);
  a.pageTable = p.pageTable;
  a.indices = p.indices;
  a.ctx = p.contextLengths;
  a.o = static_cast<__half*>(p.oPtr);
  a.partialO = p.partialO;
  a.partialStats = p.partialStats;
  a.counters = p.splitCounters;
  a.status = p.status;
  a.Hq = p.numQHeads;
  a.Hkv = p.numKVHeads;
  a.G = p.numQHeads / p.numKVHeads;
  a.poolHeadDim = p.poolHeadDim;
  a.numFlatPages = p.numFlatPages;
  a.maxPagesPerSeq = p.maxPagesPerSeq;
  a.topK = p.topK;
  a.sl2 = p.attentionScale * kLog2e;
  cudaStream_t st = static_cast<cudaStream_t>(p.stream);
  if (bf16) return a.G <= 8 ? decode_nt<1, true>(a, p.batchSize, st) : decode_nt<2, true>(a, p.batchSize, st);
  return a.G <= 8 ? decode_nt<1, false>(a, p.batchSize, st) : decode_nt<2, false>(a, p.batchSize, st);
}

}  // namespace qsa
