/*
 * qsa_oracle.h -- C entry points of the plain fp64 CPU oracle for QSA
 * (Qwen Sparse Attention) block-sparse GQA.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or helper with the CUDA library; the product path never
 * calls it and never falls back to it.
 *
 * Conventions (all arrays host memory, row-major, innermost index last):
 *   - fp16 tensors are passed as their raw IEEE binary16 bit patterns (uint16).
 *   - ratio r, budget beta, topK = list width, t = 0-based token position,
 *     L = live length of a sequence, n_c(t) = floor((t+1)/r) complete blocks.
 *   - Every function returns 0 on success and a negative value on invalid
 *     arguments (nothing is written then).
 *   - nthreads <= 0 means "all hardware threads".
 */
#ifndef QSA_ORACLE_H
#define QSA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* IEEE 754 binary16 <-> binary64 (exact widening; round-to-nearest-even narrowing). */
double qsa_oracle_half_to_double(uint16_t h);
uint16_t qsa_oracle_double_to_half(double x);

/* Index-query prep of one (row, head) vector: RMSNorm*(1+w) then partial RoPE
 * at position pos.  x: fp16 [di]; w: fp32 [di]; y: f64 [di]. */
int32_t qsa_oracle_index_q(const uint16_t* x, const float* w, int32_t di, int32_t rot,
                           int64_t pos, double theta, double eps, double* y);

/* Block key of one block from its r raw index keys (fp16 [r][di], contiguous):
 * mean -> RMSNorm*(1+w) -> partial RoPE at pos -> fp16 (RNE).  y64 (optional)
 * receives the f64 value before rounding. */
int32_t qsa_oracle_block_key(const uint16_t* raw, int32_t r, const float* w, int32_t di,
                             int32_t rot, int64_t pos, double theta, double eps,
                             uint16_t* kbar, double* y64);

/* Block score sum_h relu(q_h . kbar) / sqrt(di); q f64 [Hi][di], kbar fp16 [di]. */
double qsa_oracle_block_score(const double* q, const uint16_t* kbar, int32_t Hi, int32_t di);

/* Top-beta selection of blocks [0, n_c) by (score desc, block id asc).
 * sel receives the selected ids in ascending order; returns their count. */
int32_t qsa_oracle_select(const double* scores, int32_t n_c, int32_t budget, int32_t* sel);

/* Expansion of the selected blocks plus the causal tail {r*n_c .. t} into a
 * -1-padded ascending list of width topK. */
int32_t qsa_oracle_expand(const int32_t* sel, int32_t nsel, int32_t n_c, int64_t t,
                          int32_t r, int32_t topK, int32_t* list);

/* Prefill indexer.
 *   idxQ fp16 [B][S][Hi][di], idxK fp16 [B][S][di], wq/wk fp32 [di], ctx int32 [B].
 *   rows: optional flat row ids (b*S + t); NULL means all B*S rows in order.
 *   indices: int32 [nrows][topK] (row-compact when rows != NULL).
 *   kbar_out: optional fp16 [B][S/r][di] (blocks g < floor(L/r) written, rest 0).
 *   scores_out: optional f64 [nrows][S/r]; -inf where g >= n_c(t) or t >= L. */
int32_t qsa_oracle_indexer_prefill(const uint16_t* idxQ, const uint16_t* idxK,
                                   const float* wq, const float* wk, const int32_t* ctx,
                                   int32_t B, int32_t S, int32_t Hi, int32_t di, int32_t rot,
                                   int32_t ratio, int32_t budget, int32_t topK,
                                   double theta, double eps,
                                   const int64_t* rows, int64_t nrows,
                                   int32_t* indices, uint16_t* kbar_out, double* scores_out,
                                   int32_t nthreads);

/* Sparse GQA prefill attention over given index lists.
 *   q fp16 [B][S][Hq][D], k/v fp16 [B][S][Hkv][D], ctx int32 [B].
 *   indices int32 [nrows][topK] (row-compact when rows != NULL, else [B*S][topK]).
 *   out f64 [nrows][Hq][D]; rows t >= L are 0, an empty list gives 0. */
int32_t qsa_oracle_sparse_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                  const int32_t* indices, const int32_t* ctx,
                                  int32_t B, int32_t S, int32_t Hq, int32_t Hkv, int32_t D,
                                  int32_t topK, double scale,
                                  const int64_t* rows, int64_t nrows, double* out,
                                  int32_t nthreads);

/* Decode indexer for one sequence from its compact state (no pool):
 *   L = total length including the new token, t = L-1.
 *   idxQ fp16 [Hi][di] (new token), idxK fp16 [di] (new token raw key).
 *   kbar fp16 [floor(t/r)][di]: block keys of the blocks complete before t.
 *   tail fp16 [t mod r][di]: raw keys of tokens r*floor(t/r) .. t-1.
 *   indices int32 [topK]; kbar_new fp16 [di] written when t completes a block
 *   (return value 1), else untouched (return value 0); scores_out optional f64
 *   [floor(L/r)]. */
int32_t qsa_oracle_indexer_decode_state(const uint16_t* idxQ, const uint16_t* idxK,
                                        const float* wq, const float* wk,
                                        const uint16_t* kbar, const uint16_t* tail, int64_t L,
                                        int32_t Hi, int32_t di, int32_t rot, int32_t ratio,
                                        int32_t budget, int32_t topK, double theta, double eps,
                                        int32_t* indices, uint16_t* kbar_new, double* scores_out);

/* Decode indexer over the paged pool.
 *   pool fp16 [numFlatPages][128][Hkv][poolHeadDim]; tails of head 0 are read and
 *   updated in place.  pageTable int32 [B][2][maxPagesPerSeq] (row 0 K pages,
 *   row 1 V pages, both absolute pool page ids).  ctx int32 [B] = total lengths.
 *   idxQ fp16 [B][Hi][di]; idxK fp16 [B][di]; indices int32 [B][topK].
 *   scores_out optional f64 [B][maxPagesPerSeq*128/r]. */
int32_t qsa_oracle_indexer_decode(const uint16_t* idxQ, const uint16_t* idxK,
                                  const float* wq, const float* wk, uint16_t* pool,
                                  const int32_t* pageTable, const int32_t* ctx,
                                  int32_t B, int32_t Hkv, int32_t D, int32_t poolHeadDim,
                                  int32_t numFlatPages, int32_t maxPagesPerSeq,
                                  int32_t Hi, int32_t di, int32_t rot, int32_t ratio,
                                  int32_t budget, int32_t topK, double theta, double eps,
                                  int32_t* indices, double* scores_out, int32_t nthreads);

/* Attention of one query token over n gathered rows (no pool):
 *   q fp16 [Hq][D], krows/vrows fp16 [n][Hkv][D]; out f64 [Hq][D]. */
int32_t qsa_oracle_attend_rows(const uint16_t* q, const uint16_t* krows, const uint16_t* vrows,
                               int64_t n, int32_t Hq, int32_t Hkv, int32_t D, double scale,
                               double* out);

/* Sparse GQA decode attention over the paged pool (columns [0, D) of each row).
 *   q fp16 [B][Hq][D]; indices int32 [B][topK]; out f64 [B][Hq][D]. */
int32_t qsa_oracle_sparse_decode(const uint16_t* q, const uint16_t* pool, const int32_t* pageTable,
                                 const int32_t* indices, const int32_t* ctx,
                                 int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t poolHeadDim,
                                 int32_t numFlatPages, int32_t maxPagesPerSeq, int32_t topK,
                                 double scale, double* out, int32_t nthreads);

/* bf16 variants of the three attention passes: the same arguments, with every
 * 16-bit tensor (q, k, v, krows, vrows, pool) read as bfloat16 bit patterns
 * ("Cute Dsl Qsa Sparse Runner": Q/K/V are fp16 or bf16). */
int32_t qsa_oracle_sparse_prefill_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                       const int32_t* indices, const int32_t* ctx,
                                       int32_t B, int32_t S, int32_t Hq, int32_t Hkv, int32_t D,
                                       int32_t topK, double scale,
                                       const int64_t* rows, int64_t nrows, double* out,
                                       int32_t nthreads);
int32_t qsa_oracle_attend_rows_bf16(const uint16_t* q, const uint16_t* krows, const uint16_t* vrows,
                                    int64_t n, int32_t Hq, int32_t Hkv, int32_t D, double scale,
                                    double* out);
int32_t qsa_oracle_sparse_decode_bf16(const uint16_t* q, const uint16_t* pool, const int32_t* pageTable,
                                      const int32_t* indices, const int32_t* ctx,
                                      int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t poolHeadDim,
                                      int32_t numFlatPages, int32_t maxPagesPerSeq, int32_t topK,
                                      double scale, double* out, int32_t nthreads);
/* Upstream step of the attention layer: packed QKV fp16 [B][S][Hq + 2*Hkv][D]
 * (q heads, then k heads, then v heads) -> qout fp16 [B][S][Hq][D] and
 * kout / vout fp16 [B][S][Hkv][D].  q and k heads: RMSNorm*(1+w) (qw, kw fp32
 * [D]) then partial RoPE on [0, rot) at the row's position, rounded once to
 * fp16; v heads copied.  Row s is at position s when S > 1, at ctx[b]-1 when
 * S == 1; rows at or past the live length are zeros. */
int32_t qsa_oracle_rope_qkv(const uint16_t* qkv, const float* qw, const float* kw, const int32_t* ctx,
                            int32_t B, int32_t S, int32_t Hq, int32_t Hkv, int32_t D, int32_t rot,
                            double theta, double eps, uint16_t* qout, uint16_t* kout, uint16_t* vout,
                            int32_t nthreads);

/* bfloat16 -> binary64 (exact widening). */
double qsa_oracle_bf16_to_double(uint16_t h);

#ifdef __cplusplus
}
#endif

#endif /* QSA_ORACLE_H */
