/*
 * qsa.h -- C ABI of libqsa.so: QSA (Qwen Sparse Attention) block-sparse GQA
 * on one GB300 (sm_103a).
 *
 * Four entry points make up the hot path:
 *   qsa_indexer_prefill  -- weight-free block indexer over a padded prefill batch
 *   qsa_indexer_decode   -- the same indexer for one new token per sequence,
 *                           reading and updating its state in the paged KV pool
 *   qsa_sparse_prefill   -- sparse GQA attention over dense padded BSND Q/K/V
 *   qsa_sparse_decode    -- split-K sparse GQA decode attention over the pool
 *
 * Where each operation is defined (page title, then section):
 *   "Cute Dsl Qsa Sparse Runner" (TensorRT-Edge-LLM C++ API): the runner
 *       classes, struct QsaSparsePrefillParams, struct QsaSparseDecodeParams,
 *       kMaxSplits = 8, kPartialRows = 16.
 *   "Qsa Attention Plugin" (TensorRT-Edge-LLM C++ API): class
 *       QsaAttentionPlugin -- fused step 2 (prefill indexer, top-512 blocks,
 *       expand + causal tail, [B, S, 2051] lists), step 3 (decode indexer
 *       B1/B2/B3), the attributes of the constructor, and the "KV pool
 *       contract" (widened rows, tail state of head 0).
 *   "spark_model/layers/ops/qsa.rs" (Atlas Inference API docs): doc comments
 *       of qsa_block_pool, qsa_qprep, qsa_qprep_rows, qsa_score, qsa_score_rows
 *       (block pooling, query prep, block score sum_h relu(q_h . k_b)/sqrt(hd)).
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers (cudaMalloc'd or equivalent) of
 *     the GPU that is current on the calling thread; the caller owns every
 *     buffer.  The library allocates nothing and never synchronises the host:
 *     each call only enqueues kernels on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream).
 *   - fp16 means IEEE binary16.  Layouts are row-major, innermost index last.
 *   - Parameters are validated on the host before anything is launched.  A
 *     non-QSA_OK status means nothing was enqueued, except QSA_ERR_CUDA, which
 *     reports a failed launch (the CUDA error is left for cudaGetLastError and
 *     described by qsa_last_error_message()).
 *   - No C++ exception crosses this boundary.
 */
#ifndef QSA_H
#define QSA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QSA_API __attribute__((visibility("default")))
#else
#define QSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QSA_OK = 0,
  QSA_ERR_INVALID_ARG = 1, /* null pointer, negative or inconsistent size        */
  QSA_ERR_UNSUPPORTED = 2, /* valid shape that these kernels do not implement   */
  QSA_ERR_WORKSPACE = 3,   /* workspace missing, too small or misaligned        */
  QSA_ERR_CUDA = 4         /* a kernel launch failed                            */
} qsa_status_t;

/* ------------------------------------------------------------------ indexer */

/* Prefill indexer ("Qsa Attention Plugin", fused step 2; "qsa.rs",
 * qsa_block_pool / qsa_qprep_rows / qsa_score_rows).  Normal prefill from
 * position 0 (no chunked prefill).  For each sequence b with live length
 * L = contextLengths[b] and each row t < L it writes the -1-padded list
 *   { r*g .. r*g + r-1 : g among the top-`budget` complete blocks }
 *     U { r*n_c .. t },      n_c = floor((t+1)/r),
 * where block keys are mean(r raw keys) -> RMSNorm*(1+kNormW) -> RoPE at r*g
 * (stored fp16), queries are RMSNorm*(1+qNormW) -> RoPE at t (fp32), and the
 * score of block g is sum_h relu(q_h . kbar_g) / sqrt(headDim).  When
 * n_c <= budget every block is kept; exact score ties go to the lower block
 * id.  Lists are written in ascending token order; rows t >= L are all -1.
 * Limits: seqLen <= qsa_indexer_prefill_max_seq_len() (2^24), batchSize *
 * seqLen < 2^31, batchSize <= 65535; other shapes return QSA_ERR_UNSUPPORTED.
 * Calls that share one workspace must not run concurrently (one stream). */
typedef struct {
  const void* idxQ;              /* fp16 [B, S, numHeads, headDim] raw index queries     */
  const void* idxK;              /* fp16 [B, S, headDim] raw index keys (one shared head)  */
  const float* qNormW;           /* fp32 [headDim]; the norm multiplies by (1 + w)         */
  const float* kNormW;           /* fp32 [headDim]                                          */
  const int32_t* contextLengths; /* int32 [B], 0 <= L <= S                                  */
  int32_t* indices;              /* out int32 [B, S, topK]                                  */
  void* workspace;               /* >= qsa_indexer_prefill_workspace_size(), 256-B aligned,
                                    no initial contents required: status word, block keys
                                    fp16 [B, S/r, headDim], a work counter, and 320 score
                                    slots of 8 x S/r fp32 (the rows being selected), i.e.
                                    ~(2*B*headDim/r + 2560/r*4) bytes per row of S: 21 MB
                                    at B = 1, S = 8192, 336 MB at S = 131072. Linear in S */
  size_t workspaceBytes;
  int32_t batchSize;             /* B                                                       */
  int32_t seqLen;                /* S (padded length)                                       */
  int32_t numHeads;              /* indexer heads Hi, 1..8                                  */
  int32_t headDim;               /* indexer head dim di: 64 or 128                          */
  int32_t rotDim;                /* rotated dims: even, <= headDim                           */
  int32_t compressRatio;         /* r (tokens per block); 4 on the pages                    */
  int32_t budget;                /* blocks kept per row; 512 on the pages                    */
  int32_t topK;                  /* list width, >= budget*r + r - 1 (2051 on the pages)      */
  float ropeTheta;               /* RoPE base                                                */
  float rmsNormEps;              /* RMSNorm epsilon                                          */
  void* stream;                  /* cudaStream_t                                             */
} QsaIndexerPrefillParams;

/* Decode indexer ("Qsa Attention Plugin", step 3: B1 fused q-prep + predicated
 * tail write / compress, B2 block scores from the kbar tails, B3 deterministic
 * top-`budget` + expand).  One new token per sequence at t = L-1 where
 * L = contextLengths[b] is the TOTAL length including that token.  Indexer
 * state lives in head 0 of the pool rows, columns [kvHeadDim, kvHeadDim+headDim)
 * ("KV pool contract"): block g's key in the V-row tail of token r*g, the raw
 * index key of each token of the trailing incomplete block in its K-row tail.
 * This call (B1) stores the new raw key in the K-row tail of token t when t
 * leaves its block incomplete; when t completes block g = (t+1)/r - 1 it
 * instead computes that block's key from the K-row tails of tokens
 * r*g .. t-1 plus the new raw key and stores it in the V-row tail of token r*g.
 * No other pool byte is written.  Then it scores every complete block and
 * writes the row's list exactly as the prefill indexer would for row t.
 * A sequence with L == 0 gets an all -1 list and no pool write.
 * Device-side errors do not fault: the first int32 of the workspace is a
 * status word that the kernels OR bits into and never clear -- bit 0: a
 * wait on a TMA copy ran past 0.2 s and the scorer stopped early (the lists
 * of that call are then not valid); bit 1: a page id outside
 * [0, numFlatPages) was met and skipped.  Limits: batchSize <= 1024,
 * budget <= 4096, compressRatio 4, 8 or 16. */
typedef struct {
  const void* idxQ;              /* fp16 [B, numHeads, headDim] raw index query of the new token */
  const void* idxK;              /* fp16 [B, headDim] raw index key of the new token             */
  const float* qNormW;           /* fp32 [headDim]                                                */
  const float* kNormW;           /* fp32 [headDim]                                                */
  void* kvPool;                  /* fp16 [numFlatPages, 128, numKVHeads, poolHeadDim]; tails R/W  */
  const int32_t* pageTable;      /* int32 [B, 2, maxPagesPerSeq]: row 0 K page ids, row 1 V page
                                    ids (absolute pool page ids, i.e. pre-offset by numPages)     */
  const int32_t* contextLengths; /* int32 [B], total lengths, 0 <= L <= 128*maxPagesPerSeq        */
  int32_t* indices;              /* out int32 [B, 1, topK]                                        */
  void* workspace;               /* >= qsa_indexer_decode_workspace_size(), 256-B aligned, and
                                    ZERO-FILLED before its first use; every call leaves its
                                    counters at zero again                                         */
  size_t workspaceBytes;
  int32_t batchSize;             /* B                                                              */
  int32_t numKVHeads;            /* Hkv of the pool                                                */
  int32_t kvHeadDim;             /* attention head dim D: the tail starts at column D              */
  int32_t poolHeadDim;           /* >= kvHeadDim + headDim                                         */
  int32_t numFlatPages;          /* pages in the pool (both planes)                                */
  int32_t maxPagesPerSeq;        /* page-table row length                                          */
  int32_t numHeads;              /* indexer heads Hi, 1..8                                         */
  int32_t headDim;               /* indexer head dim di: 64 or 128                                 */
  int32_t rotDim;
  int32_t compressRatio;         /* r: 4, 8 or 16 (divides the 128-token page)                     */
  int32_t budget;                /* 1..4096                                                        */
  int32_t topK;                  /* >= budget*r + r - 1                                            */
  float ropeTheta;
  float rmsNormEps;
  void* stream;
} QsaIndexerDecodeParams;

/* Prefill -> decode hand-off of the indexer state ("Qsa Attention Plugin",
 * "KV pool contract").  After qsa_indexer_prefill has run on a batch, this
 * call writes that batch's indexer state into a paged KV pool, so that
 * qsa_indexer_decode can continue each sequence at position L =
 * contextLengths[b]:
 *   - the key of every complete block g < floor(L/r) (the fp16 key the
 *     prefill call left in its workspace) goes to the V-row tail of token r*g;
 *   - the raw index key of every token of the trailing incomplete block
 *     (r*floor(L/r) .. L-1) goes to that token's K-row tail.
 * Tails are head 0, columns [kvHeadDim, kvHeadDim + headDim) of a pool row; no
 * other pool byte is written.  A decode step at t = L then selects what the
 * prefill indexer selects for row t of the same sequence extended by one token.
 * Pages are read from pageTable rows 0 (K) and 1 (V) for tokens < L; a page id
 * outside [0, numFlatPages) is skipped and sets bit 1 of the status word at the
 * head of the workspace. */
typedef struct {
  const void* idxK;              /* fp16 [B, S, headDim] raw index keys (the prefill call's input)   */
  const int32_t* contextLengths; /* int32 [B], as given to the prefill call                           */
  void* workspace;               /* the qsa_indexer_prefill workspace after that call                 */
  size_t workspaceBytes;
  void* kvPool;                  /* fp16 [numFlatPages, 128, numKVHeads, poolHeadDim]                 */
  const int32_t* pageTable;      /* int32 [B, 2, maxPagesPerSeq] (row 1 pre-offset by numPages)       */
  int32_t batchSize;             /* B                                                                 */
  int32_t seqLen;                /* S of the prefill call                                             */
  int32_t headDim;               /* indexer head dim di (64 or 128)                                   */
  int32_t compressRatio;         /* r of the prefill call                                             */
  int32_t numKVHeads;            /* Hkv of the pool                                                   */
  int32_t kvHeadDim;             /* attention head dim D: the tail starts at column D                 */
  int32_t poolHeadDim;           /* >= kvHeadDim + headDim                                            */
  int32_t numFlatPages;
  int32_t maxPagesPerSeq;        /* 128 * maxPagesPerSeq >= S                                         */
  void* stream;
} QsaIndexerHandoffParams;

/* Upstream step of a QSA attention layer ("Qsa Attention Plugin", fused step
 * 1: packed-QKV split, per-head qk-norm with (1 + w), partial RoPE, paged-KV
 * write, dense K/V mirrors).  The projections stay with the caller: this call
 * takes their packed output.  For every live row and head:
 *   q/k heads: y = x / sqrt(mean(x^2) + eps) * (1 + w), then the half-split
 *              RoPE of dims [0, rotDim) at the row's position, rounded to fp16;
 *   v heads:   copied.
 * Row s is at position s when seqLen > 1 (a prefill from position 0; rows
 * s >= contextLengths[b] are padding) and at contextLengths[b] - 1 when
 * seqLen == 1 (one new token, contextLengths = total length including it).
 * Outputs: qOut (always; zeros for padding rows), kOut / vOut dense mirrors
 * when non-NULL (zeros for padding rows), and, when kvPool is non-NULL, the
 * leading headDim columns of the token's K row (page table row 0) and V row
 * (row 1) for every KV head.  Pool tails and padding rows' pool rows are not
 * written; a page id outside [0, numFlatPages) is skipped.
 * Errors: QSA_ERR_INVALID_ARG for NULL required pointers, sizes < 1, an odd
 * rotDim or rotDim > headDim, theta <= 0, eps < 0, or a pool without its page
 * table; QSA_ERR_UNSUPPORTED for headDim not 64/128, rotDim not a multiple of
 * 16, poolHeadDim not a multiple of 8, a tensor pointer not 16-byte aligned,
 * or a packed token row (numQHeads + 2 numKVHeads) * headDim * 2 above 64 KiB.  Ownership: every buffer is the caller's; nothing is allocated. */
typedef struct {
  const void* qkv;               /* fp16 [B, S, numQHeads + 2*numKVHeads, headDim]: q, then k, then v heads */
  const float* qNormW;           /* fp32 [headDim]                                                          */
  const float* kNormW;           /* fp32 [headDim]                                                          */
  const int32_t* contextLengths; /* int32 [B]                                                               */
  void* qOut;                    /* out fp16 [B, S, numQHeads, headDim]                                     */
  void* kOut;                    /* out fp16 [B, S, numKVHeads, headDim], or NULL                           */
  void* vOut;                    /* out fp16 [B, S, numKVHeads, headDim], or NULL                           */
  void* kvPool;                  /* fp16 [numFlatPages, 128, numKVHeads, poolHeadDim], or NULL              */
  const int32_t* pageTable;      /* int32 [B, 2, maxPagesPerSeq] (needed with kvPool)                       */
  int32_t batchSize;
  int32_t seqLen;
  int32_t numQHeads;
  int32_t numKVHeads;
  int32_t headDim;               /* 64 or 128                                                               */
  int32_t rotDim;                /* multiple of 16, <= headDim                                              */
  int32_t poolHeadDim;           /* >= headDim, multiple of 8 (with kvPool)                                 */
  int32_t numFlatPages;
  int32_t maxPagesPerSeq;
  float ropeTheta;
  float rmsNormEps;
  void* stream;
} QsaRopeQkvParams;

/* --------------------------------------------------------------- attention */

/* Sparse GQA prefill ("Cute Dsl Qsa Sparse Runner", struct
 * QsaSparsePrefillParams, field for field).  For each live row t < L and query
 * head h (KV head g = h / (numQHeads/numKVHeads)):
 *   o[b,t,h] = sum_{j in list} softmax_j(attentionScale * q[b,t,h] . k[b,j,g]) v[b,j,g]
 * over the entries j >= 0 of indices[b,t,:].  Causality lives entirely in the
 * list: no positional mask is applied.  Output rows t >= L are exact zeros;
 * a live row whose list has no valid entry is zero too.  K/V rows are only
 * read where a list names them; an entry outside [0, L) is skipped (a list
 * must only name live tokens).
 * status (not on the pages; may be NULL): a device int32 that the kernel ORs
 * error bits into and never clears -- bit 2 (value 4): an entry other than -1
 * fell outside [0, L) and was skipped.  Zero it before the calls it should
 * cover; read it once the stream has reached them (qsa_last_device_error
 * reads it as well).  A NULL status records nothing; the entries are
 * skipped all the same. */
typedef struct {
  const void* qPtr;              /* fp16 [B, S, numQHeads, headDim]  */
  const void* kPtr;              /* fp16 [B, S, numKVHeads, headDim] */
  const void* vPtr;              /* fp16 [B, S, numKVHeads, headDim] */
  void* oPtr;                    /* out fp16 [B, S, numQHeads, headDim] */
  const int32_t* indices;        /* int32 [B, S, topK], -1 padded on the right */
  const int32_t* contextLengths; /* int32 [B], 0 <= L <= S */
  int32_t batchSize;
  int32_t seqLen;
  int32_t numQHeads;
  int32_t numKVHeads;            /* numQHeads / numKVHeads must be 1..16 */
  int32_t headDim;               /* 128 */
  int32_t topK;
  float attentionScale;          /* multiplier of q . k (not assumed 1/sqrt(D)) */
  void* stream;
  int32_t* status;               /* optional device error word (see above), or NULL */
} QsaSparsePrefillParams;

/* Split-K sparse GQA decode ("Cute Dsl Qsa Sparse Runner", struct
 * QsaSparseDecodeParams, field for field).  One query token per sequence;
 * K/V rows come from the pool through the page table, and only columns
 * [0, headDim) of a pool row are read.  The list of each (sequence, KV head)
 * is cut into at most kMaxSplits = 8 contiguous slices of whole 64-entry
 * tiles (fewer when B * numKVHeads * 8 CTAs would not fit in one wave on the
 * GPU and a smaller count does); each slice writes an fp32 partial (O, m, l)
 * and the last slice to finish merges the partials into oPtr and resets its
 * counter to zero.  The slice count depends only on the shapes and the GPU,
 * so repeated calls give identical bits.  splitCounters MUST be zero on
 * entry (zero-fill the buffer once; every call leaves it zeroed).
 * status (not on the pages; may be NULL): a device int32 that the kernels OR
 * error bits into and never clear -- bit 1 (value 2): a list entry's page id
 * fell outside [0, numFlatPages); bit 2 (value 4): an entry other than -1
 * fell outside [0, L).  Such entries are skipped (never read) whether or not
 * status is given. */
typedef struct {
  const void* qPtr;              /* fp16 [B, 1, numQHeads, headDim] */
  const void* kvPoolPtr;         /* fp16 [numFlatPages, 128, numKVHeads, poolHeadDim] */
  const int32_t* pageTable;      /* int32 [B, 2, maxPagesPerSeq] (row 1 pre-offset by numPages) */
  const int32_t* indices;        /* int32 [B, 1, topK], -1 padded */
  const int32_t* contextLengths; /* int32 [B], total lengths including the new token */
  void* oPtr;                    /* out fp16 [B, 1, numQHeads, headDim] */
  float* partialO;               /* fp32 [B*numKVHeads*8, 16, headDim] */
  float* partialStats;           /* fp32 [B*numKVHeads*8, 2, 16] */
  int32_t* splitCounters;        /* int32 [B*numKVHeads], zero on entry */
  int32_t batchSize;
  int32_t numQHeads;
  int32_t numKVHeads;            /* numQHeads / numKVHeads must be 1..16 */
  int32_t headDim;               /* 128 */
  int32_t poolHeadDim;           /* >= headDim, multiple of 8 */
  int32_t numFlatPages;          /* 2 * numPages (both planes) */
  int32_t maxPagesPerSeq;
  int32_t topK;
  float attentionScale;
  void* stream;
  int32_t* status;               /* optional device error word (see above), or NULL */
} QsaSparseDecodeParams;

/* ------------------------------------------------------------ entry points */

QSA_API qsa_status_t qsa_indexer_prefill(const QsaIndexerPrefillParams* params);
QSA_API qsa_status_t qsa_indexer_decode(const QsaIndexerDecodeParams* params);
QSA_API qsa_status_t qsa_sparse_prefill(const QsaSparsePrefillParams* params);
QSA_API qsa_status_t qsa_sparse_decode(const QsaSparseDecodeParams* params);
QSA_API qsa_status_t qsa_indexer_prefill_handoff(const QsaIndexerHandoffParams* params);
QSA_API qsa_status_t qsa_rope_qkv(const QsaRopeQkvParams* params);

/* The two attention calls with bfloat16 tensors ("Cute Dsl Qsa Sparse Runner":
 * the runners take fp16 or bf16): the same params structs, contract and
 * checks, with qPtr/kPtr/vPtr/oPtr (prefill) and qPtr/kvPoolPtr/oPtr (decode)
 * holding bf16 instead of fp16.  Arithmetic: products in fp32, softmax in fp32,
 * P rounded to bf16 for the PV product, fp32 accumulation, output rounded to
 * bf16.  The decode indexer keeps its fp16 tails in a bf16 pool's columns
 * [kvHeadDim, kvHeadDim + headDim): the attention never reads them. */
QSA_API qsa_status_t qsa_sparse_prefill_bf16(const QsaSparsePrefillParams* params);
QSA_API qsa_status_t qsa_sparse_decode_bf16(const QsaSparseDecodeParams* params);

/* The sparse prefill attention ("Cute Dsl Qsa Sparse Runner",
 * QsaSparsePrefillParams: per-row gathers, one CTA per (query token, KV
 * head)) on the 5th-generation tensor cores: tcgen05.mma with its operands
 * read from shared memory by descriptor and its accumulators in tensor memory,
 * over tiles of 128 keys.  Same params, contract, checks and errors as
 * qsa_sparse_prefill / qsa_sparse_prefill_bf16 (fp16 or bf16 tensors);
 * arithmetic: q.k products accumulated in fp32, softmax in fp32, P rounded to
 * the element type for the PV product, fp32 accumulation, output rounded once.
 * The result differs from qsa_sparse_prefill only by rounding order.
 * status bit 0 (value 1), added to the bits above: a wait on the tensor cores
 * ran past 0.2 s and the row was left unwritten. */
QSA_API qsa_status_t qsa_sparse_prefill_tcgen05(const QsaSparsePrefillParams* params);
QSA_API qsa_status_t qsa_sparse_prefill_tcgen05_bf16(const QsaSparsePrefillParams* params);

/* Split-K sparse decode with no caller workspace.  The pages have no
 * counterpart to this entry point.  It serves callers that cannot hand device
 * memory to a library call on their decode path: an engine whose memory is
 * planned once up front and offers plugins no workspace, or a serving loop
 * that must not reach an allocator per token (an allocator may synchronise
 * the device, or fail under memory pressure, in the middle of a step).
 *
 * It computes exactly what qsa_sparse_decode computes, with these differences:
 *   - partialO, partialStats and splitCounters must be NULL.  The fp32
 *     partials and the split counters live in one fixed scratch array inside
 *     the library (16.25 MiB of device memory per GPU, placed by the driver
 *     when the library's code is loaded onto that GPU).  It holds
 *     batchSize * numKVHeads <= 256 (sequence, KV head) pairs at headDim 128;
 *     larger shapes return QSA_ERR_UNSUPPORTED and launch nothing.
 *   - The first call in each CUDA context (per GPU: its primary context, which
 *     the runtime uses) looks up the scratch's address and clears its
 *     counters on `stream`.  Make that first call before any stream capture.
 *     Later calls in the same context only launch the kernels.  After
 *     cudaDeviceReset the next call sees a new context, where the library's
 *     code and scratch are loaded afresh, and does the set-up again (so that
 *     call too belongs before any capture).
 *   - All calls on one GPU within a process share that scratch.  Two calls
 *     whose kernels may run at the same time (different streams, or
 *     different threads) race and corrupt each other's outputs: issue them on
 *     one stream. */
QSA_API qsa_status_t qsa_sparse_decode_noalloc(const QsaSparseDecodeParams* params);

/* Gather-to-scratch form of the decode (qsa.rs, "qsa_gather" and the
 * scratch-as-paged-cache note): copies the K and V rows of the tokens that a
 * decode list names out of the paged pool into contiguous scratch, and
 * describes the scratch as a paged pool of its own, so that an unchanged
 * qsa_sparse_decode can consume it.  It is the A/B counterpart of the
 * decode's in-kernel page-table gathers: qsa_sparse_decode on
 * (scratch, scratchPageTable, scratchIndices, scratchLengths) with
 * numFlatPages = 2 * batchSize * P, maxPagesPerSeq = P, poolHeadDim = headDim
 * returns exactly, bit for bit, what qsa_sparse_decode returns on the pool
 * with the original list.
 *
 * P = qsa_gather_scratch_pages(topK) = ceil(topK / 128).  Slot n of sequence
 * b holds list entry n: its K row at scratch page b * P + n / 128, row n % 128,
 * and its V row at page (batchSize + b) * P + n / 128.  An entry outside
 * [0, contextLengths[b]) or on a page outside [0, numFlatPages) leaves its
 * slot unwritten (it is never read) and is -1 in scratchIndices.
 *
 * Errors: QSA_ERR_INVALID_ARG for a NULL pointer, sizes < 1 or
 * poolHeadDim < headDim; QSA_ERR_UNSUPPORTED for headDim not a multiple of 8,
 * numKVHeads * headDim above 1024, poolHeadDim not a multiple of 8, or kvPool
 * / scratch not 16-byte aligned.  Every buffer is the caller's; nothing is
 * allocated. */
typedef struct {
  const void* kvPool;            /* fp16 or bf16 [numFlatPages, 128, numKVHeads, poolHeadDim]               */
  const int32_t* pageTable;      /* int32 [B, 2, maxPagesPerSeq]                                            */
  const int32_t* indices;        /* int32 [B, 1, topK], -1 padded                                           */
  const int32_t* contextLengths; /* int32 [B]                                                               */
  void* scratch;                 /* out, same element type: [2 * B * P, 128, numKVHeads, headDim]           */
  int32_t* scratchPageTable;     /* out int32 [B, 2, P]                                                     */
  int32_t* scratchIndices;       /* out int32 [B, 1, topK]: n where entry n names a row, else -1            */
  int32_t* scratchLengths;       /* out int32 [B]: topK                                                     */
  int32_t batchSize;
  int32_t numKVHeads;
  int32_t headDim;               /* columns [0, headDim) of each pool row are copied                        */
  int32_t poolHeadDim;
  int32_t numFlatPages;
  int32_t maxPagesPerSeq;
  int32_t topK;
  void* stream;
} QsaGatherParams;

QSA_API qsa_status_t qsa_gather_selected(const QsaGatherParams* params);
QSA_API int32_t qsa_gather_scratch_pages(int32_t topK);
/* Elements (halves) of the scratch: 2 * batchSize * P * 128 * numKVHeads * headDim (0 when invalid). */
QSA_API size_t qsa_gather_scratch_elems(int32_t batchSize, int32_t numKVHeads, int32_t headDim, int32_t topK);

/* Workspace bytes of the indexers (0 when the sizes are invalid). */
QSA_API size_t qsa_indexer_prefill_workspace_size(int32_t batchSize, int32_t seqLen, int32_t headDim,
                                          int32_t compressRatio);
QSA_API size_t qsa_indexer_decode_workspace_size(int32_t batchSize, int32_t maxPagesPerSeq,
                                         int32_t compressRatio, int32_t budget);

/* Element counts of the split-K decode workspace ("Cute Dsl Qsa Sparse Runner",
 * QsaSparseDecodeParams: partialO, partialStats, splitCounters). */
QSA_API size_t qsa_sparse_decode_partial_o_elems(int32_t batchSize, int32_t numKVHeads, int32_t headDim);
QSA_API size_t qsa_sparse_decode_partial_stats_elems(int32_t batchSize, int32_t numKVHeads);
QSA_API size_t qsa_sparse_decode_counter_elems(int32_t batchSize, int32_t numKVHeads);
QSA_API int32_t qsa_sparse_decode_max_splits(void);   /* kMaxSplits = 8   */
QSA_API int32_t qsa_sparse_decode_partial_rows(void); /* kPartialRows = 16 */

/* Whether these kernels cover a shape (the runners' canImplement): 1 or 0. */
QSA_API int32_t qsa_sparse_prefill_can_implement(int32_t numQHeads, int32_t numKVHeads, int32_t headDim);
QSA_API int32_t qsa_sparse_decode_can_implement(int32_t numQHeads, int32_t numKVHeads, int32_t headDim,
                                        int32_t poolHeadDim);

/* Longest padded sequence the prefill indexer takes (2^24 rows; longer
 * seqLen returns QSA_ERR_UNSUPPORTED).  Its memory is linear in seqLen (the
 * workspace above); the bound keeps token and block ids in int32 with room.
 * qsa_indexer_prefill_max_blocks() returns the same number: the largest
 * floor(seqLen / compressRatio) a call can have (ratio 1). */
QSA_API int32_t qsa_indexer_prefill_max_seq_len(void);
QSA_API int32_t qsa_indexer_prefill_max_blocks(void);

/* Debug read of the status word at the head of an indexer workspace (the
 * device-side error bits: bit 0 a TMA wait that ran out, bit 1 a page id
 * outside the pool; see qsa_indexer_decode).  Enqueues a 4-byte copy of that
 * word into host memory *out on `stream` (a cudaStream_t) and returns without
 * waiting: *out is valid once the stream has reached the copy (for pageable
 * host memory CUDA completes the copy before the call returns).  The bits
 * accumulate; zero-fill the workspace to clear them.  Errors:
 * QSA_ERR_INVALID_ARG for a NULL pointer, QSA_ERR_CUDA if the copy cannot be
 * enqueued.  Nothing else is read or written. */
QSA_API qsa_status_t qsa_last_device_error(const void* workspace, void* stream, int32_t* out);

/* Testing hook for the device-side error path (process-wide, not for
 * production use): bounds every later qsa_indexer_decode call's waits on the
 * progress of its own page stream to `ns` nanoseconds instead of 0.2 s, so
 * that a test can make them run out and read bit 0 of the status word.  0
 * restores the 0.2 s bound.  The wait for copies already in flight before a
 * CTA exits keeps its 0.2 s bound whatever is set, so no copy outlives its
 * CTA.  The lists of a call whose waits ran out are not valid; zero-fill the
 * workspace before the next call. */
QSA_API void qsa_debug_set_wait_limit_ns(uint64_t ns);

/* Human-readable name of a status, and the detail of the last failure on the
 * calling thread (never NULL; empty when there was none). */
QSA_API const char* qsa_status_string(qsa_status_t status);
QSA_API const char* qsa_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H */
