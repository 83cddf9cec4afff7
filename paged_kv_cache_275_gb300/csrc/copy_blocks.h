// Internal interface of the block-copy kernel (copy_blocks.cu), used by capi.cu.
#pragma once

#include "pkv_internal.h"

namespace pkv {

struct CopyParams {
  void* k_cache;
  void* v_cache;
  const int64_t* src_dst;  // [num_pairs][2]
  unsigned* err;
  int64_t num_blocks;
  int64_t chunks_per_block;  // 16-byte chunks in one block (all kv heads)
};

// copy_blocks kernel launch (one CTA per pair and K/V).
cudaError_t launch_copy_blocks(const CopyParams& p, int num_pairs, cudaStream_t stream);

}  // namespace pkv
