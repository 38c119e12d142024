// qsa_oracle.cpp -- plain fp64 CPU oracle for QSA (Qwen Sparse Attention)
// block-sparse GQA: the weight-free block indexer and sparse GQA attention.
//
// TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
// baseline leg of the benchmark may load this library.  It shares no code,
// header, table or helper with the CUDA library and is never called by it.
//
// Every step is written as the pages state it, in f64, with no blocking,
// fusion or reordering.  Sources (page title, then section):
//   [RS]  "spark_model/layers/ops/qsa.rs" (Atlas Inference API docs), doc
//         comments of qsa_block_pool, qsa_qprep, qsa_qprep_rows, qsa_score,
//         qsa_score_rows.
//   [PL]  "Qsa Attention Plugin" (TensorRT-Edge-LLM C++ API), class
//         QsaAttentionPlugin: fused steps 2-3 and the "KV pool contract".
//   [SR]  "Cute Dsl Qsa Sparse Runner" (TensorRT-Edge-LLM C++ API), structs
//         QsaSparsePrefillParams and QsaSparseDecodeParams.
//
// Readings where the pages are silent (each is also listed in the design notes):
//   - complete blocks visible to row t: n_c(t) = floor((t+1)/r); the list width
//     topK = beta*r + r - 1 leaves room for exactly r-1 tail tokens.
//   - partial RoPE is the half-split form on dims [0, rot): the pair
//     (i, i + rot/2) is rotated by pos * theta^(-2i/rot), i < rot/2; dims
//     [rot, di) pass through.  Angles, cos and sin are taken in f64.
//   - RMSNorm: y = x / sqrt(mean(x^2) + eps) * (1 + w), one w shared by heads.
//   - one shared index-key head; block keys are stored as fp16 (round to
//     nearest even), in prefill as in decode.
//   - selection: all blocks when n_c <= beta, else the beta largest scores,
//     exact ties going to the lower block id.
//   - lists are written in ascending order; rows t >= L are all -1.
//   - GQA: query head h reads KV head h / (Hq/Hkv).
//   - an empty list (no valid entry) gives a zero output row.
//   - decode: t = L-1; when t completes a block, its key is computed from the
//     K-row tails of the block's first r-1 tokens plus the new raw key and is
//     stored in the V-row tail of the block's first token; otherwise the new
//     raw key is stored in token t's K-row tail.
//
// Pins: every function here is checked by the CPU tests (tests/test_oracle_*)
// against closed forms, hand-worked examples (tests/golden/), brute force,
// a library routine (numpy float16, torch scaled_dot_product_attention) and
// invariants.  The exact constants of the indexer that the pages leave open
// (RoPE convention, eps placement) are pinned to the readings above, not to a
// printed example: the pages print none.

#include "qsa_oracle.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

// ----------------------------------------------------------------- fp16 bits
// IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.

double half_to_double(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int e = (h >> 10) & 0x1f;
  const int f = h & 0x3ff;
  double mag;
  if (e == 0) {
    mag = std::ldexp(static_cast<double>(f), -24);  // subnormal: f * 2^-24
  } else if (e == 31) {
    mag = f ? std::numeric_limits<double>::quiet_NaN() : std::numeric_limits<double>::infinity();
  } else {
    mag = std::ldexp(static_cast<double>(1024 + f), e - 25);  // (1.f) * 2^(e-15)
  }
  return sign ? -mag : mag;
}

// The same widening for all 65536 patterns, built once; the passes below read
// fp16 tensors through it.
const double* half_table() {
  static const std::vector<double> tab = [] {
    std::vector<double> t(65536);
    for (int h = 0; h < 65536; ++h) t[h] = half_to_double(static_cast<uint16_t>(h));
    return t;
  }();
  return tab.data();
}

// bfloat16: the upper 16 bits of a binary32 (1 sign, 8 exponent, 7 fraction
// bits), so widening is exact: place the bits on top of a float.
double bf16_to_double(uint16_t h) {
  const uint32_t u = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &u, sizeof(f));
  return static_cast<double>(f);
}

const double* bf16_table() {
  static const std::vector<double> tab = [] {
    std::vector<double> t(65536);
    for (int h = 0; h < 65536; ++h) t[h] = bf16_to_double(static_cast<uint16_t>(h));
    return t;
  }();
  return tab.data();
}

// Round-to-nearest-even of a double to binary16.
uint16_t double_to_half(double x) {
  if (std::isnan(x)) return 0x7e00;
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  double a = std::fabs(x);
  if (a == 0.0) return sign;
  // Quantum of the binade holding a; below 2^-14 the subnormal quantum 2^-24.
  int e2;
  std::frexp(a, &e2);  // a = m * 2^e2, m in [0.5, 1)  =>  floor(log2 a) = e2 - 1
  int E = e2 - 1;
  if (E < -14) E = -14;
  const double quantum = std::ldexp(1.0, E - 10);
  // a / quantum is exact (power-of-two scaling); nearbyint rounds half to even.
  double n = std::nearbyint(a / quantum);
  if (E == -14 && n < 1024.0) {
    return static_cast<uint16_t>(sign | static_cast<uint16_t>(n));  // subnormal (n may be 0)
  }
  if (n >= 2048.0) {  // rounded up into the next binade
    n = 1024.0;
    E += 1;
  }
  if (E + 15 >= 31) return static_cast<uint16_t>(sign | 0x7c00);  // overflow to inf
  return static_cast<uint16_t>(sign | ((E + 15) << 10) | (static_cast<int>(n) - 1024));
}

// ------------------------------------------------------------ small helpers

// y = x / sqrt(mean(x^2) + eps) * (1 + w)   ([RS] qsa_block_pool, qsa_qprep)
void rms_norm_one_plus_w(const double* x, const float* w, int n, double eps, double* y) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  const double inv = 1.0 / std::sqrt(ss / n + eps);
  for (int i = 0; i < n; ++i) y[i] = x[i] * inv * (1.0 + static_cast<double>(w[i]));
}

// Half-split rotary embedding of dims [0, rot) at position pos.
void partial_rope(double* y, int rot, int64_t pos, double theta) {
  const int half = rot / 2;
  for (int i = 0; i < half; ++i) {
    const double inv_freq = std::pow(theta, -2.0 * i / rot);
    const double a = static_cast<double>(pos) * inv_freq;
    const double c = std::cos(a), s = std::sin(a);
    const double x0 = y[i], x1 = y[i + half];
    y[i] = x0 * c - x1 * s;
    y[i + half] = x1 * c + x0 * s;
  }
}

bool rope_args_ok(int di, int rot) { return di > 0 && di <= 512 && rot >= 0 && rot <= di && rot % 2 == 0; }

// Index query of one (row, head): RMSNorm*(1+w), then RoPE at pos.
void index_q(const uint16_t* x, const float* w, int di, int rot, int64_t pos, double theta,
             double eps, double* q) {
  const double* H = half_table();
  std::vector<double> xd(di);
  for (int i = 0; i < di; ++i) xd[i] = H[x[i]];
  rms_norm_one_plus_w(xd.data(), w, di, eps, q);
  partial_rope(q, rot, pos, theta);
}

// Block key: mean of r raw keys -> RMSNorm*(1+w) -> RoPE at the block start pos -> fp16.
void block_key(const uint16_t* raw, int r, const float* w, int di, int rot, int64_t pos,
               double theta, double eps, uint16_t* kbar, double* y64) {
  const double* H = half_table();
  std::vector<double> m(di, 0.0), y(di);
  for (int j = 0; j < r; ++j)
    for (int i = 0; i < di; ++i) m[i] += H[raw[static_cast<size_t>(j) * di + i]];
  for (int i = 0; i < di; ++i) m[i] /= r;
  rms_norm_one_plus_w(m.data(), w, di, eps, y.data());
  partial_rope(y.data(), rot, pos, theta);
  for (int i = 0; i < di; ++i) kbar[i] = double_to_half(y[i]);
  if (y64) std::memcpy(y64, y.data(), sizeof(double) * di);
}

// sum_h relu(q_h . kbar) / sqrt(di)   ([RS] qsa_score)
double block_score(const double* q, const uint16_t* kbar, int Hi, int di) {
  const double* H = half_table();
  double k[512];
  for (int i = 0; i < di; ++i) k[i] = H[kbar[i]];
  double s = 0.0;
  for (int h = 0; h < Hi; ++h) {
    double dot = 0.0;
    for (int i = 0; i < di; ++i) dot += q[static_cast<size_t>(h) * di + i] * k[i];
    s += dot > 0.0 ? dot : 0.0;
  }
  return s / std::sqrt(static_cast<double>(di));
}

// Top-beta by (score desc, id asc); output ascending ids.  ([PL] step 2/B3)
int select_blocks(const double* s, int n_c, int budget, int32_t* sel) {
  std::vector<int32_t> ids(n_c);
  for (int g = 0; g < n_c; ++g) ids[g] = g;
  if (n_c > budget) {
    std::sort(ids.begin(), ids.end(), [s](int32_t a, int32_t b) {
      if (s[a] != s[b]) return s[a] > s[b];
      return a < b;
    });
    ids.resize(budget);
    std::sort(ids.begin(), ids.end());
  }
  std::copy(ids.begin(), ids.end(), sel);
  return static_cast<int>(ids.size());
}

// Selected blocks -> tokens {r g .. r g + r-1}, plus the tail {r n_c .. t}, ascending, -1 padded.
int expand(const int32_t* sel, int nsel, int n_c, int64_t t, int r, int topK, int32_t* list) {
  std::vector<int32_t> toks;
  toks.reserve(static_cast<size_t>(nsel) * r + r);
  for (int k = 0; k < nsel; ++k)
    for (int j = 0; j < r; ++j) toks.push_back(sel[k] * r + j);
  for (int64_t j = static_cast<int64_t>(n_c) * r; j <= t; ++j) toks.push_back(static_cast<int32_t>(j));
  std::sort(toks.begin(), toks.end());
  if (static_cast<int>(toks.size()) > topK) return -1;
  for (int i = 0; i < topK; ++i) list[i] = i < static_cast<int>(toks.size()) ? toks[i] : -1;
  return static_cast<int>(toks.size());
}

// Softmax attention of one query head over n rows: o = sum_j p_j v_j,
// p = softmax(scale * q . k_j).  Empty -> zeros.  ([SR] QsaSparsePrefillParams)
// H widens the 16-bit inputs to f64: half_table() or bf16_table().
void attend_head(const uint16_t* q, const uint16_t* const* krows, const uint16_t* const* vrows,
                 int64_t n, int D, double scale, double* o, const double* H) {
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  if (n == 0) return;
  std::vector<double> qd(D), s(n);
  for (int d = 0; d < D; ++d) qd[d] = H[q[d]];
  double m = -std::numeric_limits<double>::infinity();
  for (int64_t j = 0; j < n; ++j) {
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += qd[d] * H[krows[j][d]];
    s[j] = scale * dot;
    m = std::max(m, s[j]);
  }
  double l = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    const double p = std::exp(s[j] - m);
    l += p;
    for (int d = 0; d < D; ++d) o[d] += p * H[vrows[j][d]];
  }
  for (int d = 0; d < D; ++d) o[d] /= l;
}

template <class F>
void parallel_for(int64_t n, int nthreads, F f) {
  if (nthreads <= 0) nthreads = static_cast<int>(std::max(1u, std::thread::hardware_concurrency()));
  if (n <= 1 || nthreads == 1) {
    for (int64_t i = 0; i < n; ++i) f(i);
    return;
  }
  const int T = static_cast<int>(std::min<int64_t>(nthreads, n));
  std::vector<std::thread> pool;
  pool.reserve(T);
  for (int k = 0; k < T; ++k) {
    pool.emplace_back([=, &f]() {
      for (int64_t i = k; i < n; i += T) f(i);  // static round-robin: deterministic outputs
    });
  }
  for (auto& th : pool) th.join();
}

constexpr int kTokensPerPage = 128;  // [SR] QsaSparseDecodeParams: pool [2*numPages, 128, Hkv, poolHeadDim]

}  // namespace

// =============================================================== C entry points
extern "C" {

double qsa_oracle_half_to_double(uint16_t h) { return half_to_double(h); }
uint16_t qsa_oracle_double_to_half(double x) { return double_to_half(x); }

int32_t qsa_oracle_index_q(const uint16_t* x, const float* w, int32_t di, int32_t rot, int64_t pos,
                           double theta, double eps, double* y) {
  if (!x || !w || !y || !rope_args_ok(di, rot) || pos < 0) return -1;
  index_q(x, w, di, rot, pos, theta, eps, y);
  return 0;
}

int32_t qsa_oracle_block_key(const uint16_t* raw, int32_t r, const float* w, int32_t di, int32_t rot,
                             int64_t pos, double theta, double eps, uint16_t* kbar, double* y64) {
  if (!raw || !w || !kbar || r <= 0 || !rope_args_ok(di, rot) || pos < 0) return -1;
  block_key(raw, r, w, di, rot, pos, theta, eps, kbar, y64);
  return 0;
}

double qsa_oracle_block_score(const double* q, const uint16_t* kbar, int32_t Hi, int32_t di) {
  return block_score(q, kbar, Hi, di);
}

int32_t qsa_oracle_select(const double* scores, int32_t n_c, int32_t budget, int32_t* sel) {
  if (n_c < 0 || budget <= 0 || (n_c > 0 && (!scores || !sel))) return -1;
  return select_blocks(scores, n_c, budget, sel);
}

int32_t qsa_oracle_expand(const int32_t* sel, int32_t nsel, int32_t n_c, int64_t t, int32_t r,
                          int32_t topK, int32_t* list) {
  if (!list || r <= 0 || topK <= 0 || nsel < 0 || (nsel > 0 && !sel)) return -1;
  return expand(sel, nsel, n_c, t, r, topK, list);
}

int32_t qsa_oracle_indexer_prefill(const uint16_t* idxQ, const uint16_t* idxK, const float* wq,
                                   const float* wk, const int32_t* ctx, int32_t B, int32_t S,
                                   int32_t Hi, int32_t di, int32_t rot, int32_t ratio, int32_t budget,
                                   int32_t topK, double theta, double eps, const int64_t* rows,
                                   int64_t nrows, int32_t* indices, uint16_t* kbar_out,
                                   double* scores_out, int32_t nthreads) {
  if (!idxQ || !idxK || !wq || !wk || !ctx || !indices) return -1;
  if (B <= 0 || S <= 0 || Hi <= 0 || ratio <= 0 || budget <= 0 || !rope_args_ok(di, rot)) return -1;
  if (topK < budget * ratio + ratio - 1) return -1;
  for (int b = 0; b < B; ++b)
    if (ctx[b] < 0 || ctx[b] > S) return -1;
  const int64_t nr = rows ? nrows : static_cast<int64_t>(B) * S;
  for (int64_t i = 0; rows && i < nr; ++i)
    if (rows[i] < 0 || rows[i] >= static_cast<int64_t>(B) * S) return -1;
  const int nbmax = S / ratio;

  // Block keys of every complete block of every sequence (g < floor(L/r)).
  std::vector<uint16_t> kbar(static_cast<size_t>(B) * nbmax * di, 0);
  parallel_for(static_cast<int64_t>(B) * nbmax, nthreads, [&](int64_t bg) {
    const int b = static_cast<int>(bg / nbmax), g = static_cast<int>(bg % nbmax);
    if (g >= ctx[b] / ratio) return;
    const uint16_t* raw = idxK + (static_cast<size_t>(b) * S + static_cast<size_t>(g) * ratio) * di;
    block_key(raw, ratio, wk, di, rot, static_cast<int64_t>(g) * ratio, theta, eps,
              kbar.data() + (static_cast<size_t>(b) * nbmax + g) * di, nullptr);
  });
  if (kbar_out) std::memcpy(kbar_out, kbar.data(), kbar.size() * sizeof(uint16_t));

  parallel_for(nr, nthreads, [&](int64_t i) {
    const int64_t row = rows ? rows[i] : i;
    const int b = static_cast<int>(row / S);
    const int64_t t = row % S;
    int32_t* list = indices + i * topK;
    double* srow = scores_out ? scores_out + i * nbmax : nullptr;
    if (srow)
      for (int g = 0; g < nbmax; ++g) srow[g] = -std::numeric_limits<double>::infinity();
    if (t >= ctx[b]) {  // rows at or past the live length: all -1
      for (int k = 0; k < topK; ++k) list[k] = -1;
      return;
    }
    std::vector<double> q(static_cast<size_t>(Hi) * di);
    for (int h = 0; h < Hi; ++h)
      index_q(idxQ + ((static_cast<size_t>(b) * S + t) * Hi + h) * di, wq, di, rot, t, theta, eps,
              q.data() + static_cast<size_t>(h) * di);
    const int n_c = static_cast<int>((t + 1) / ratio);
    std::vector<double> s(n_c);
    for (int g = 0; g < n_c; ++g)
      s[g] = block_score(q.data(), kbar.data() + (static_cast<size_t>(b) * nbmax + g) * di, Hi, di);
    if (srow)
      for (int g = 0; g < n_c; ++g) srow[g] = s[g];
    std::vector<int32_t> sel(std::max(n_c, 1));
    const int nsel = select_blocks(s.data(), n_c, budget, sel.data());
    expand(sel.data(), nsel, n_c, t, ratio, topK, list);
  });
  return 0;
}

int32_t sparse_prefill_impl(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* indices,
                            const int32_t* ctx, int32_t B, int32_t S, int32_t Hq, int32_t Hkv, int32_t D,
                            int32_t topK, double scale, const int64_t* rows, int64_t nrows, double* out,
                            int32_t nthreads, const double* H) {
  if (!q || !k || !v || !indices || !ctx || !out) return -1;
  if (B <= 0 || S <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || topK <= 0 || Hq % Hkv != 0) return -1;
  for (int b = 0; b < B; ++b)
    if (ctx[b] < 0 || ctx[b] > S) return -1;
  const int64_t nr = rows ? nrows : static_cast<int64_t>(B) * S;
  for (int64_t i = 0; rows && i < nr; ++i)
    if (rows[i] < 0 || rows[i] >= static_cast<int64_t>(B) * S) return -1;
  const int group = Hq / Hkv;
  std::atomic<int32_t> bad{0};
  parallel_for(nr * Hq, nthreads, [&](int64_t ih) {
    const int64_t i = ih / Hq;
    const int h = static_cast<int>(ih % Hq);
    const int64_t row = rows ? rows[i] : i;
    const int b = static_cast<int>(row / S);
    const int64_t t = row % S;
    double* o = out + (i * Hq + h) * D;
    if (t >= ctx[b]) {  // exact zeros at or past the live length
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      return;
    }
    const int g = h / group;
    const int32_t* list = indices + i * topK;
    std::vector<const uint16_t*> kr, vr;
    for (int e = 0; e < topK; ++e) {
      const int32_t j = list[e];
      if (j < 0) continue;  // -1 padding
      if (j >= ctx[b]) {    // a list may only name live tokens
        bad = 1;
        continue;
      }
      kr.push_back(k + ((static_cast<size_t>(b) * S + j) * Hkv + g) * D);
      vr.push_back(v + ((static_cast<size_t>(b) * S + j) * Hkv + g) * D);
    }
    attend_head(q + ((static_cast<size_t>(b) * S + t) * Hq + h) * D, kr.data(), vr.data(),
                static_cast<int64_t>(kr.size()), D, scale, o, H);
  });
  return bad ? -2 : 0;
}

int32_t qsa_oracle_indexer_decode_state(const uint16_t* idxQ, const uint16_t* idxK, const float* wq,
                                        const float* wk, const uint16_t* kbar, const uint16_t* tail,
                                        int64_t L, int32_t Hi, int32_t di, int32_t rot, int32_t ratio,
                                        int32_t budget, int32_t topK, double theta, double eps,
                                        int32_t* indices, uint16_t* kbar_new, double* scores_out) {
  if (!indices || Hi <= 0 || ratio <= 0 || budget <= 0 || !rope_args_ok(di, rot)) return -1;
  if (topK < budget * ratio + ratio - 1 || L < 0) return -1;
  if (L == 0) {  // no token: empty list, no state change
    for (int k = 0; k < topK; ++k) indices[k] = -1;
    return 0;
  }
  if (!idxQ || !idxK || !wq || !wk) return -1;
  const int64_t t = L - 1;
  const int64_t n_prev = t / ratio;  // blocks complete before this token
  const int64_t n_c = L / ratio;     // blocks complete including it
  if (n_prev > 0 && !kbar) return -1;
  if (t % ratio > 0 && !tail) return -1;
  const bool completes = n_c > n_prev;
  if (completes && !kbar_new) return -1;

  // B1: q prep at pos t; compress the block t completes (its first r-1 raw keys
  // come from the K-row tails, the last is the new raw key).
  std::vector<double> q(static_cast<size_t>(Hi) * di);
  for (int h = 0; h < Hi; ++h)
    index_q(idxQ + static_cast<size_t>(h) * di, wq, di, rot, t, theta, eps, q.data() + static_cast<size_t>(h) * di);
  if (completes) {
    std::vector<uint16_t> raw(static_cast<size_t>(ratio) * di);
    if (ratio > 1) std::memcpy(raw.data(), tail, sizeof(uint16_t) * static_cast<size_t>(ratio - 1) * di);
    std::memcpy(raw.data() + static_cast<size_t>(ratio - 1) * di, idxK, sizeof(uint16_t) * di);
    block_key(raw.data(), ratio, wk, di, rot, n_prev * ratio, theta, eps, kbar_new, nullptr);
  }
  // B2: block scores over every complete block.
  std::vector<double> s(n_c);
  for (int64_t g = 0; g < n_c; ++g) {
    const uint16_t* kg = g < n_prev ? kbar + g * di : kbar_new;
    s[g] = block_score(q.data(), kg, Hi, di);
  }
  if (scores_out)
    for (int64_t g = 0; g < n_c; ++g) scores_out[g] = s[g];
  // B3: top-beta + expand.
  std::vector<int32_t> sel(std::max<int64_t>(n_c, 1));
  const int nsel = select_blocks(s.data(), static_cast<int>(n_c), budget, sel.data());
  if (expand(sel.data(), nsel, static_cast<int>(n_c), t, ratio, topK, indices) < 0) return -1;
  return completes ? 1 : 0;
}

int32_t qsa_oracle_indexer_decode(const uint16_t* idxQ, const uint16_t* idxK, const float* wq,
                                  const float* wk, uint16_t* pool, const int32_t* pageTable,
                                  const int32_t* ctx, int32_t B, int32_t Hkv, int32_t D,
                                  int32_t poolHeadDim, int32_t numFlatPages, int32_t maxPagesPerSeq,
                                  int32_t Hi, int32_t di, int32_t rot, int32_t ratio, int32_t budget,
                                  int32_t topK, double theta, double eps, int32_t* indices,
                                  double* scores_out, int32_t nthreads) {
  if (!idxQ || !idxK || !wq || !wk || !pool || !pageTable || !ctx || !indices) return -1;
  if (B <= 0 || Hkv <= 0 || D <= 0 || di <= 0 || poolHeadDim < D + di || numFlatPages <= 0 ||
      maxPagesPerSeq <= 0 || ratio <= 0 || kTokensPerPage % ratio != 0)
    return -1;
  for (int b = 0; b < B; ++b)
    if (ctx[b] < 0 || ctx[b] > static_cast<int64_t>(maxPagesPerSeq) * kTokensPerPage) return -1;
  const int64_t nbmax = static_cast<int64_t>(maxPagesPerSeq) * kTokensPerPage / ratio;
  // Address of column c of token j's row, head 0, in plane p (0 = K pages, 1 = V pages).
  auto row_ptr = [&](int b, int plane, int64_t j) -> uint16_t* {
    const int32_t page = pageTable[(static_cast<size_t>(b) * 2 + plane) * maxPagesPerSeq + j / kTokensPerPage];
    return pool + ((static_cast<size_t>(page) * kTokensPerPage + j % kTokensPerPage) * Hkv) * poolHeadDim;
  };
  int32_t bad = 0;
  for (int b = 0; b < B; ++b)
    for (int p = 0; p < 2; ++p)
      for (int64_t pg = 0; pg * kTokensPerPage < ctx[b]; ++pg) {
        const int32_t page = pageTable[(static_cast<size_t>(b) * 2 + p) * maxPagesPerSeq + pg];
        if (page < 0 || page >= numFlatPages) bad = 1;
      }
  if (bad) return -1;

  parallel_for(B, nthreads, [&](int64_t bi) {
    const int b = static_cast<int>(bi);
    const int64_t L = ctx[b];
    int32_t* list = indices + static_cast<size_t>(b) * topK;
    double* srow = scores_out ? scores_out + b * nbmax : nullptr;
    if (srow)
      for (int64_t g = 0; g < nbmax; ++g) srow[g] = -std::numeric_limits<double>::infinity();
    if (L == 0) {
      for (int k = 0; k < topK; ++k) list[k] = -1;
      return;
    }
    const int64_t t = L - 1, n_prev = t / ratio, first_tail = n_prev * ratio;
    // Gather the indexer state held in the pool tails (head 0, columns [D, D+di)).
    std::vector<uint16_t> kb(static_cast<size_t>(std::max<int64_t>(n_prev, 1)) * di);
    for (int64_t g = 0; g < n_prev; ++g)
      std::memcpy(kb.data() + g * di, row_ptr(b, 1, g * ratio) + D, sizeof(uint16_t) * di);
    std::vector<uint16_t> tl(static_cast<size_t>(std::max<int64_t>(t - first_tail, 1)) * di);
    for (int64_t j = first_tail; j < t; ++j)
      std::memcpy(tl.data() + (j - first_tail) * di, row_ptr(b, 0, j) + D, sizeof(uint16_t) * di);
    std::vector<uint16_t> knew(di);
    const int32_t rc = qsa_oracle_indexer_decode_state(
        idxQ + static_cast<size_t>(b) * Hi * di, idxK + static_cast<size_t>(b) * di, wq, wk, kb.data(),
        tl.data(), L, Hi, di, rot, ratio, budget, topK, theta, eps, list, knew.data(), srow);
    // Write back the state update.
    if (rc == 1)
      std::memcpy(row_ptr(b, 1, first_tail) + D, knew.data(), sizeof(uint16_t) * di);
    else if (rc == 0)
      std::memcpy(row_ptr(b, 0, t) + D, idxK + static_cast<size_t>(b) * di, sizeof(uint16_t) * di);
  });
  return 0;
}

int32_t attend_rows_impl(const uint16_t* q, const uint16_t* krows, const uint16_t* vrows, int64_t n, int32_t Hq,
                         int32_t Hkv, int32_t D, double scale, double* out, const double* H) {
  if (!q || !out || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0 || n < 0 || (n > 0 && (!krows || !vrows)))
    return -1;
  const int group = Hq / Hkv;
  for (int h = 0; h < Hq; ++h) {
    const int g = h / group;
    std::vector<const uint16_t*> kr(n), vr(n);
    for (int64_t j = 0; j < n; ++j) {
      kr[j] = krows + (j * Hkv + g) * D;
      vr[j] = vrows + (j * Hkv + g) * D;
    }
    attend_head(q + static_cast<size_t>(h) * D, kr.data(), vr.data(), n, D, scale, out + static_cast<size_t>(h) * D,
                H);
  }
  return 0;
}

int32_t sparse_decode_impl(const uint16_t* q, const uint16_t* pool, const int32_t* pageTable,
                           const int32_t* indices, const int32_t* ctx, int32_t B, int32_t Hq, int32_t Hkv,
                           int32_t D, int32_t poolHeadDim, int32_t numFlatPages, int32_t maxPagesPerSeq,
                           int32_t topK, double scale, double* out, int32_t nthreads, const double* H) {
  if (!q || !pool || !pageTable || !indices || !ctx || !out) return -1;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0 || poolHeadDim < D || topK <= 0) return -1;
  const int group = Hq / Hkv;
  std::atomic<int32_t> bad{0};
  parallel_for(static_cast<int64_t>(B) * Hq, nthreads, [&](int64_t bh) {
    const int b = static_cast<int>(bh / Hq), h = static_cast<int>(bh % Hq), g = h / group;
    double* o = out + bh * D;
    const int32_t* list = indices + static_cast<size_t>(b) * topK;
    std::vector<const uint16_t*> kr, vr;
    for (int e = 0; e < topK; ++e) {
      const int32_t j = list[e];
      if (j < 0) continue;
      if (j >= ctx[b]) {
        bad = 1;
        continue;
      }
      const int32_t kp = pageTable[(static_cast<size_t>(b) * 2 + 0) * maxPagesPerSeq + j / kTokensPerPage];
      const int32_t vp = pageTable[(static_cast<size_t>(b) * 2 + 1) * maxPagesPerSeq + j / kTokensPerPage];
      if (kp < 0 || kp >= numFlatPages || vp < 0 || vp >= numFlatPages) {
        bad = 1;
        continue;
      }
      kr.push_back(pool + ((static_cast<size_t>(kp) * kTokensPerPage + j % kTokensPerPage) * Hkv + g) * poolHeadDim);
      vr.push_back(pool + ((static_cast<size_t>(vp) * kTokensPerPage + j % kTokensPerPage) * Hkv + g) * poolHeadDim);
    }
    attend_head(q + bh * D, kr.data(), vr.data(), static_cast<int64_t>(kr.size()), D, scale, o, H);
  });
  return bad ? -2 : 0;
}

int32_t qsa_oracle_sparse_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                  const int32_t* indices, const int32_t* ctx, int32_t B, int32_t S,
                                  int32_t Hq, int32_t Hkv, int32_t D, int32_t topK, double scale,
                                  const int64_t* rows, int64_t nrows, double* out, int32_t nthreads) {
  return sparse_prefill_impl(q, k, v, indices, ctx, B, S, Hq, Hkv, D, topK, scale, rows, nrows, out, nthreads,
                             half_table());
}
int32_t qsa_oracle_sparse_prefill_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                       const int32_t* indices, const int32_t* ctx, int32_t B, int32_t S,
                                       int32_t Hq, int32_t Hkv, int32_t D, int32_t topK, double scale,
                                       const int64_t* rows, int64_t nrows, double* out, int32_t nthreads) {
  return sparse_prefill_impl(q, k, v, indices, ctx, B, S, Hq, Hkv, D, topK, scale, rows, nrows, out, nthreads,
                             bf16_table());
}
int32_t qsa_oracle_attend_rows(const uint16_t* q, const uint16_t* krows, const uint16_t* vrows, int64_t n,
                               int32_t Hq, int32_t Hkv, int32_t D, double scale, double* out) {
  return attend_rows_impl(q, krows, vrows, n, Hq, Hkv, D, scale, out, half_table());
}
int32_t qsa_oracle_attend_rows_bf16(const uint16_t* q, const uint16_t* krows, const uint16_t* vrows, int64_t n,
                                    int32_t Hq, int32_t Hkv, int32_t D, double scale, double* out) {
  return attend_rows_impl(q, krows, vrows, n, Hq, Hkv, D, scale, out, bf16_table());
}
int32_t qsa_oracle_sparse_decode(const uint16_t* q, const uint16_t* pool, const int32_t* pageTable,
                                 const int32_t* indices, const int32_t* ctx, int32_t B, int32_t Hq,
                                 int32_t Hkv, int32_t D, int32_t poolHeadDim, int32_t numFlatPages,
                                 int32_t maxPagesPerSeq, int32_t topK, double scale, double* out,
                                 int32_t nthreads) {
  return sparse_decode_impl(q, pool, pageTable, indices, ctx, B, Hq, Hkv, D, poolHeadDim, numFlatPages,
                            maxPagesPerSeq, topK, scale, out, nthreads, half_table());
}
int32_t qsa_oracle_sparse_decode_bf16(const uint16_t* q, const uint16_t* pool, const int32_t* pageTable,
                                      const int32_t* indices, const int32_t* ctx, int32_t B, int32_t Hq,
                                      int32_t Hkv, int32_t D, int32_t poolHeadDim, int32_t numFlatPages,
                                      int32_t maxPagesPerSeq, int32_t topK, double scale, double* out,
                                      int32_t nthreads) {
  return sparse_decode_impl(q, pool, pageTable, indices, ctx, B, Hq, Hkv, D, poolHeadDim, numFlatPages,
                            maxPagesPerSeq, topK, scale, out, nthreads, bf16_table());
}
double qsa_oracle_bf16_to_double(uint16_t h) { return bf16_to_double(h); }

// Upstream step of the attention layer ("Qsa Attention Plugin", fused step 1):
// split a packed QKV row into heads; q and k heads get the per-head RMSNorm
// with (1 + w) and the partial RoPE at the row's position (the same two
// operations as the index-query prep), v heads pass through; every output is
// rounded once to fp16.  Row s is at position s when S > 1 (prefill from 0) and
// at L - 1 when S == 1 (one new token); rows at or past L are zeros.
int32_t qsa_oracle_rope_qkv(const uint16_t* qkv, const float* qw, const float* kw, const int32_t* ctx, int32_t B,
                            int32_t S, int32_t Hq, int32_t Hkv, int32_t D, int32_t rot, double theta, double eps,
                            uint16_t* qout, uint16_t* kout, uint16_t* vout, int32_t nthreads) {
  if (!qkv || !qw || !kw || !ctx || !qout || !kout || !vout) return -1;
  if (B <= 0 || S <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || rot < 0 || rot > D || (rot & 1)) return -1;
  const int NH = Hq + 2 * Hkv;
  parallel_for(static_cast<int64_t>(B) * S * NH, nthreads, [&](int64_t i) {
    const int h = static_cast<int>(i % NH);
    const int64_t bs = i / NH;
    const int b = static_cast<int>(bs / S), s = static_cast<int>(bs % S);
    const int L = ctx[b];
    const bool live = S == 1 ? L >= 1 : s < L;
    const int64_t pos = S == 1 ? static_cast<int64_t>(L) - 1 : s;
    const uint16_t* x = qkv + (bs * NH + h) * D;
    uint16_t* dst = h < Hq ? qout + (bs * Hq + h) * D
                  : h < Hq + Hkv ? kout + (bs * Hkv + (h - Hq)) * D
                                 : vout + (bs * Hkv + (h - Hq - Hkv)) * D;
    if (!live) {
      for (int d = 0; d < D; ++d) dst[d] = 0;
      return;
    }
    if (h >= Hq + Hkv) {
      for (int d = 0; d < D; ++d) dst[d] = x[d];
      return;
    }
    std::vector<double> y(D);
    index_q(x, h < Hq ? qw : kw, D, rot, pos, theta, eps, y.data());
    for (int d = 0; d < D; ++d) dst[d] = double_to_half(y[d]);
  });
  return 0;
}

}  // extern "C"
