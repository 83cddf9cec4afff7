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
};

// Chunked prefill attention (tensor cores); grid covers max_query_len rows per sequence.
cudaError_t launch_paged_prefill(const PrefillParams& p, int head_dim, int group, int max_query_len,
                                 cudaStream_t stream);

}  // namespace pkv
