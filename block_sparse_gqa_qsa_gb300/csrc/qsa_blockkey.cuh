// qsa_blockkey.cuh -- the block key of the QSA indexer ("spark_model/layers/ops/qsa.rs",
// qsa_block_pool: mean of r raw index keys -> RMSNorm*(1+w) -> partial RoPE at the
// block start; "Qsa Attention Plugin": the key is stored fp16), computed by one warp
// with the FP64 unit used for one multiply per rotated dim only.
//
// GB300 issues an FP64 instruction at roughly 1/64 of the fp32 rate (a dependent
// DFMA costs ~70 cycles), and its 64-bit integer <-> float conversions run on
// the same unit, so a key computed in f64 takes microseconds.  Here:
//   - the sum of the r raw keys is exact (fp16 values are multiples of 2^-24
//     below 2^16, so the sum fits the ~48 bits of a double-float);
//   - the norm, the scale and the rotation run in double-float arithmetic (a value
//     kept as an unevaluated sum hi + lo of two fp32 numbers, ~48 significant
//     bits, error-free sums and products by the usual Knuth/Dekker transformations
//     with fma);
//   - the rotation angle is the f64 product pos * inv_freq (one DMUL, the same
//     value an f64 evaluation forms), reduced modulo a full turn exactly in
//     integer arithmetic against a 128-bit fixed-point 1/(2 pi), then evaluated
//     as a table angle (a multiple of 2 pi / 128, cos/sin formed on the host in
//     f64) plus a short Taylor series of the remainder (|x| <= pi / 128);
//   - the result is rounded once to fp16 (round to nearest even) from hi + lo.
// The result agrees with a direct f64 evaluation rounded to fp16 unless the f64
// value lies within ~1e-13 (relative) of an fp16 rounding boundary.
#pragma once

#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {

struct f2x {
  float hi, lo;
};

// The rotation tables of RopeFreqs that the block key reads, copied to shared
// memory once per CTA: a kernel parameter indexed by lane is a constant-bank
// load that serialises over the distinct addresses of the warp.
struct RopeSmem {
  double inv_freq[64];
  float qcos_hi[33];
  float qcos_lo[33];
};
// All threads of the CTA take part; the caller synchronises before use.
__device__ __forceinline__ void stage_rope(const RopeFreqs& rf, RopeSmem& rs) {
  for (int e = threadIdx.x; e < 64 + 33; e += blockDim.x) {
    if (e < 64) {
      rs.inv_freq[e] = rf.inv_freq[e];
    } else {
      rs.qcos_hi[e - 64] = rf.qcos_hi[e - 64];
      rs.qcos_lo[e - 64] = rf.qcos_lo[e - 64];
    }
  }
}

__device__ __forceinline__ f2x two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}
// a + b when |a| >= |b| (or a == 0).
__device__ __forceinline__ f2x quick_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ f2x df_neg(f2x x) { return {-x.hi, -x.lo}; }
__device__ __forceinline__ f2x df_add(f2x x, f2x y) {
  f2x s = two_sum(x.hi, y.hi);
  const f2x t = two_sum(x.lo, y.lo);
  s = quick_two_sum(s.hi, __fadd_rn(s.lo, t.hi));
  return quick_two_sum(s.hi, __fadd_rn(s.lo, t.lo));
}
__device__ __forceinline__ f2x df_add_f(f2x x, float y) {
  const f2x s = two_sum(x.hi, y);
  return quick_two_sum(s.hi, __fadd_rn(s.lo, x.lo));
}
__device__ __forceinline__ f2x df_mul(f2x x, f2x y) {
  const float p = __fmul_rn(x.hi, y.hi);
  float e = __fmaf_rn(x.hi, y.hi, -p);
  e = __fmaf_rn(x.hi, y.lo, e);
  e = __fmaf_rn(x.lo, y.hi, e);
  return quick_two_sum(p, e);
}
__device__ __forceinline__ f2x df_mul_f(f2x x, float y) {
  const float p = __fmul_rn(x.hi, y);
  float e = __fmaf_rn(x.hi, y, -p);
  e = __fmaf_rn(x.lo, y, e);
  return quick_two_sum(p, e);
}
__device__ __forceinline__ f2x df_sqr(f2x x) {
  const float p = __fmul_rn(x.hi, x.hi);
  float e = __fmaf_rn(x.hi, x.hi, -p);
  e = __fmaf_rn(__fmul_rn(2.f, x.hi), x.lo, e);
  return quick_two_sum(p, e);
}

// 1 / sqrt(x) for x > 0: the fp32 estimate, one Newton step with an exact
// residual, then a second step in double-float.
__device__ __forceinline__ f2x df_rsqrt(f2x x) {
  const float y0 = rsqrtf(x.hi);
  const f2x one = {1.f, 0.f};
  f2x r = df_add(one, df_neg(df_mul(x, df_sqr({y0, 0.f}))));
  const f2x y1 = quick_two_sum(y0, __fmul_rn(__fmul_rn(y0, r.hi), 0.5f));
  r = df_add(one, df_neg(df_mul(x, df_sqr(y1))));
  return df_add(y1, df_mul_f(y1, __fmul_rn(r.hi, 0.5f)));
}

// Round hi + lo to fp16, to nearest even.  fp16 rounding boundaries are fp32
// numbers and |lo| <= ulp(hi) / 2, so hi alone decides unless hi sits exactly
// on a boundary; then the sign of lo does.
__device__ __forceinline__ __half df_to_half(f2x v) {
  __half h = __float2half_rn(v.hi);
  if (v.lo != 0.f) {
    const __half dn = __float2half_rd(v.hi), up = __float2half_ru(v.hi);
    const float fd = __half2float(dn), fu = __half2float(up);
    if (fd != fu && __fsub_rn(v.hi, fd) == __fsub_rn(fu, v.hi)) h = v.lo > 0.f ? up : dn;
  }
  return h;
}

// frac(a / (2 pi)) * 2^64 for a finite a >= 0 below 2^52, exact up to the
// truncation of 1/(2 pi) at 128 bits: a = M * 2^(e - 1075) with a 53-bit M, and
// a / (2 pi) * 2^64 = M * C * 2^-(1139 - e), C = floor(2^128 / (2 pi)).
__device__ __forceinline__ unsigned long long turns_of(double a) {
  const unsigned long long bits = static_cast<unsigned long long>(__double_as_longlong(a));
  const int e = static_cast<int>(bits >> 52) & 0x7ff;
  if (e == 0) return 0ull;
  const unsigned long long M = (bits & 0xfffffffffffffull) | 0x10000000000000ull;
  const int sh = 1139 - e;  // >= 88 for a < 2^52
  if (sh >= 192) return 0ull;
  constexpr unsigned long long C1 = 0x7f09d5f47d4d3770ull, C2 = 0x28be60db9391054aull;  // C = C2 * 2^64 + C1
  const unsigned long long h1 = __umul64hi(M, C1);
  const unsigned long long l2 = M * C2, h2 = __umul64hi(M, C2);
  const unsigned long long p1 = h1 + l2;                   // bits 64..127 of M * C
  const unsigned long long p2 = h2 + (p1 < h1 ? 1ull : 0ull);  // bits 128.. of M * C
  if (sh >= 128) return p2 >> (sh - 128);
  return (p1 >> (sh - 64)) | (p2 << (128 - sh));
}

// cos and sin of the angle u * 2 pi / 2^64 in double-float: u is split into the
// nearest multiple k of 2^57 (k / 128 of a turn, from the quarter-turn table
// cos(pi j / 64), j = 0..32) and a remainder x of at most pi / 128 radians,
// whose sin and cos are Taylor series (the leading terms in double-float, the
// rest, below 1e-8, in fp32), and the two are joined by the angle-sum identity.
__device__ __forceinline__ void df_cos_sin_turns(unsigned long long u, const RopeSmem& rf, f2x& c, f2x& s) {
  const unsigned k = static_cast<unsigned>((u + (1ull << 56)) >> 57) & 127u;
  const long long rho = static_cast<long long>(u - (static_cast<unsigned long long>(k) << 57));
  // rho (|rho| <= 2^56) as hi * 2^32 + lo from its 32-bit halves: the high half
  // (below 2^24 in magnitude) converts exactly, the low half to within 2^8
  // units of 2^-64 turn.  32-bit conversions stay off the FP64 unit, which also
  // executes the 64-bit ones.
  const f2x r = two_sum(__fmul_rn(__int2float_rn(static_cast<int>(rho >> 32)), 0x1p32f),
                        __uint2float_rn(static_cast<unsigned>(rho & 0xffffffffll)));
  const f2x x = df_mul(r, {0x1.921fb6p-62f, -0x1.777a5cp-87f});  // rho * 2 pi / 2^64
  const f2x x2 = df_sqr(x);
  const float t = x2.hi, t2 = __fmul_rn(t, t);
  f2x ps = df_mul(x2, {-0x1.555556p-3f, 0x1.555556p-28f});  // -x^2 / 6
  ps = df_add_f(ps, __fmul_rn(t2, __fmaf_rn(-t, 0x1.a01a02p-13f, 0x1.111112p-7f)));  // + x^4/120 - x^6/5040
  const f2x sx = df_add(x, df_mul(x, ps));
  f2x cx = df_add({1.f, 0.f}, {-0.5f * x2.hi, -0.5f * x2.lo});  // 1 - x^2 / 2
  cx = df_add_f(cx, __fmul_rn(t2, __fmaf_rn(t, __fmaf_rn(t, 0x1.a01a02p-16f, -0x1.6c16c2p-10f), 0x1.555556p-5f)));
  const int q = static_cast<int>(k >> 5), j = static_cast<int>(k & 31);
  const f2x C = {rf.qcos_hi[j], rf.qcos_lo[j]}, S = {rf.qcos_hi[32 - j], rf.qcos_lo[32 - j]};
  const f2x ca = q == 0 ? C : q == 1 ? df_neg(S) : q == 2 ? df_neg(C) : S;
  const f2x sa = q == 0 ? S : q == 1 ? C : q == 2 ? df_neg(S) : df_neg(C);
  c = df_add(df_mul(ca, cx), df_neg(df_mul(sa, sx)));
  s = df_add(df_mul(sa, cx), df_mul(ca, sx));
}

// NW warps compute one block key of DI dims and store it fp16 to out[0, DI):
// warp wi (0 <= wi < NW) handles dims 32 (wi + NW p) + lane.  load(j, i)
// returns dim i of raw key j (j < ratio) of the block; pos is the block's first
// token; rf holds the staged rotation tables (stage_rope); y_s (DI entries) and,
// for NW > 1, part_s (NW entries) are shared-memory scratch of these warps,
// which synchronise on named barrier `bar` when NW > 1.
template <int DI, int NW, class Load>
__device__ __forceinline__ void block_key(const Load& load, int ratio, const float* __restrict__ wk, float eps, int rot,
                                          int pos, const RopeSmem& rf, f2x* y_s, f2x* part_s, int wi, int bar,
                                          __half* out) {
  constexpr int PER = DI / 32 / NW;
  static_assert(PER >= 1 && PER * 32 * NW == DI, "warps must split the dims evenly");
  const int lane = threadIdx.x & 31;
  auto dim = [&](int p) { return 32 * (wi + NW * p) + lane; };
  auto sync = [&]() {
    if constexpr (NW > 1)
      asm volatile("bar.sync %0, %1;\n" ::"r"(bar), "r"(NW * 32) : "memory");
    else
      __syncwarp();
  };
  // 1 / ratio in double-float (exact for a power of two)
  const float rinv = __frcp_rn(static_cast<float>(ratio));
  const f2x inv_r = {rinv, __fdiv_rn(__fmaf_rn(-rinv, static_cast<float>(ratio), 1.f), static_cast<float>(ratio))};
  float w[PER];  // issued with the key loads: the norm weights are needed only at the end
  f2x m[PER];    // sums of the raw keys, then their mean
#pragma unroll
  for (int p = 0; p < PER; ++p) {
    w[p] = wk[dim(p)];
    m[p] = {0.f, 0.f};
  }
  // The sums are exact: fp16 values are multiples of 2^-24 below 2^16 and a
  // partial sum of up to 2^8 of them needs at most 48 significant bits, which
  // hi + lo holds; the lo parts being added stay multiples of 2^-24 below 2^0.
  for (int j0 = 0; j0 < ratio; j0 += 4) {  // 4 keys x PER dims of loads in flight at once
    __half v[4][PER];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
      for (int p = 0; p < PER; ++p) v[jj][p] = j0 + jj < ratio ? load(j0 + jj, dim(p)) : __ushort_as_half(0);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
      for (int p = 0; p < PER; ++p) m[p] = df_add_f(m[p], __half2float(v[jj][p]));
  }
  f2x ss = {0.f, 0.f};
#pragma unroll
  for (int p = 0; p < PER; ++p) {
    m[p] = df_mul(m[p], inv_r);
    ss = df_add(ss, df_sqr(m[p]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss = df_add(ss, {__shfl_xor_sync(kFull, ss.hi, o), __shfl_xor_sync(kFull, ss.lo, o)});
  ss = {__shfl_sync(kFull, ss.hi, 0), __shfl_sync(kFull, ss.lo, 0)};  // one value for every lane
  if constexpr (NW > 1) {
    if (lane == 0) part_s[wi] = ss;
    sync();
    ss = part_s[0];
#pragma unroll
    for (int k = 1; k < NW; ++k) ss = df_add(ss, part_s[k]);  // the same order in every warp
  }
  const f2x inv = df_rsqrt(df_add_f({__fmul_rn(ss.hi, 1.f / DI), __fmul_rn(ss.lo, 1.f / DI)}, eps));
#pragma unroll
  for (int p = 0; p < PER; ++p) {
    m[p] = df_mul(df_mul(m[p], inv), two_sum(1.f, w[p]));
    y_s[dim(p)] = m[p];
  }
  sync();
  const int half = rot >> 1;
  const double posd = static_cast<double>(pos);
#pragma unroll
  for (int p = 0; p < PER; ++p) {
    const int i = dim(p);
    f2x r = m[p];
    if (i < rot) {
      const int kf = i < half ? i : i - half;
      f2x c, s;
      df_cos_sin_turns(turns_of(__dmul_rn(posd, rf.inv_freq[kf])), rf, c, s);
      const f2x ys = df_mul(y_s[i < half ? i + half : i - half], s);
      r = df_add(df_mul(m[p], c), i < half ? df_neg(ys) : ys);
    }
    out[i] = df_to_half(r);
  }
  sync();
}

}  // namespace qsa
