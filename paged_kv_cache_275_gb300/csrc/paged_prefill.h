// Internal interface of the chunked prefill kernel (paged_prefill.cu), used by capi.cu.
#pragma once

#include "pkv_internal.h"

namespace pkv {

struct PrefillParams {
  const void* q;               // bf16 [T][num_q_heads][head_dim]
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;  // prefix + chunk
  const int32_t* query_start;   // [num_seqs + 1]
  void* out;                    // bf16 [T][num_q_heads][head_dim]
  unsigned* err;
  int64_t num_blocks;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int max_blocks_per_seq;
  int max_query_len;  // host's bound on the chunk lengths (sizes the grid)
  float scale;
  // Split-K over the key steps: each (tile pair, kv head, sequence) runs as num_splits CTAs, each over
  // a contiguous share of the key steps.  With num_splits > 1 the CTAs write fp32 partial states
  // (O unnormalised, m in base 2, l) to ws and a merge kernel forms out.
  int num_splits = 1;
  int ws_rows = 0;     // chunk rows per sequence in ws (the grid's tiles x chunk tokens per CTA)
  float* ws = nullptr;  // [split][seq][ws_rows][num_q_heads]: D floats of O; then the same index: (m, l)
};

// Chunked prefill attention (tensor cores); grid covers max_query_len rows per sequence.
cudaError_t launch_paged_prefill(const PrefillParams& p, int head_dim, int group, int max_query_len,
                                 cudaStream_t stream);
// Chunk tokens one CTA covers (two 128-row tiles of 128 / group tokens).
inline int prefill_cta_tokens(int group) { return 256 / group; }
// Workspace bytes of a split call: partial states of every split.
inline size_t prefill_workspace_bytes(int num_seqs, int max_query_len, int num_q_heads, int num_kv_heads,
                                      int head_dim, int num_splits) {
  if (num_splits <= 1) return 0;
  const int cta = prefill_cta_tokens(num_q_heads / num_kv_heads);
  const size_t rows = static_cast<size_t>((max_query_len + cta - 1) / cta) * cta;
  return static_cast<size_t>(num_splits) * num_seqs * rows * num_q_heads * (head_dim + 2) * sizeof(float);
}

}  // namespace pkv
