// qsa_internal.h -- launch interface between the C ABI (qsa_api.cu) and the
// kernel translation units.  Host-side only; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/qsa.h"

namespace qsa {

constexpr int kTokensPerPageHost = 128;  // pool page size of the decode contract

// theta^(-2i/rot) for i < rot/2, formed in f64 on the host once per call, and
// the same frequencies as 64-bit fixed-point fractions of a turn:
// turn[i] = frac(inv_freq[i] / (2 pi)) * 2^64, so that pos * turn[i] mod 2^64
// is the angle pos * inv_freq[i] as an exact fraction of a full turn.
// qcos_hi[j] + qcos_lo[j] is cos(pi j / 64) for j = 0..32 (a quarter turn in
// steps of 1/128 of a turn) as a pair of fp32 numbers, formed in f64 on the host;
// the block-key rotation evaluates its angles from it.
struct RopeFreqs {
  double inv_freq[64];
  unsigned long long turn[64];
  float qcos_hi[33];
  float qcos_lo[33];
};

// Prefill indexer -----------------------------------------------------------
constexpr int kPrefillRowsPerCta = 8;      // query rows sharing one CTA's block-key tiles
constexpr int kPrefillScoreSlots = 320;    // CTAs of the persistent select kernel at most (2 per SM), one
                                           // workspace score slot of 8 rows x S/r floats each
constexpr int kPrefillMaxSeqLen = 1 << 24; // rows per sequence: int32 block and token ids with headroom
size_t indexer_prefill_workspace_bytes(int B, int S, int di, int ratio);
cudaError_t launch_indexer_prefill(const QsaIndexerPrefillParams& p, const RopeFreqs& rf);
cudaError_t launch_indexer_handoff(const QsaIndexerHandoffParams& p);

// Decode indexer ------------------------------------------------------------
constexpr int kDecodeMaxBatch = 1024;   // the streaming scorer keeps a per-sequence page prefix on chip
size_t indexer_decode_workspace_bytes(int B, int maxPagesPerSeq, int ratio, int budget);
cudaError_t launch_indexer_decode(const QsaIndexerDecodeParams& p, const RopeFreqs& rf,
                                  const CUtensorMap& kbarMap);
// Bound of the decode scorer's progress waits (0: the default 0.2 s); see qsa_debug_set_wait_limit_ns.
void set_decode_wait_limit_ns(uint64_t ns);

// Attention -----------------------------------------------------------------
// bf16: Q/K/V/O (prefill) or q/pool/o (decode) hold bfloat16 instead of fp16.
cudaError_t launch_sparse_prefill(const QsaSparsePrefillParams& p, bool bf16 = false);
cudaError_t launch_sparse_prefill_tc(const QsaSparsePrefillParams& p, bool bf16 = false);  // tcgen05 / TMEM
cudaError_t launch_sparse_decode(const QsaSparseDecodeParams& p, bool bf16 = false);

// Upstream q/k norm + RoPE ------------------------------------------------------
cudaError_t launch_rope_qkv(const QsaRopeQkvParams& p, const RopeFreqs& rf);
constexpr int kRopeMaxRowBytes = 64 * 1024;  // one token's packed heads, staged in shared memory

cudaError_t launch_gather(const QsaGatherParams& p);
int gather_scratch_pages(int topK);
int gather_max_row_chunks();  // 16-byte chunks of one K (or V) token row a warp copies

// SMs of the current device (cached per device).
int sm_count();


// Stores msg as the calling thread's qsa_last_error_message() and returns s.
qsa_status_t record_error(qsa_status_t s, const char* msg);

}  // namespace qsa
