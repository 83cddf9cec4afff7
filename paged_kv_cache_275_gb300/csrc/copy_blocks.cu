// copy_blocks: whole-block copies inside the KV pool, the copy half of
// copy-on-write for blocks shared between sequences ("v0版本介绍", section
// "为什么需要推理框架": requests may share the KV blocks of a common prompt).
//
// A block of the [block][kv head][16][head_dim] layout is one contiguous run
// of num_kv_heads * 16 * head_dim bf16 (64 KB at 8 kv heads, D 128), so a copy
// is a plain streaming memcpy: one CTA per (pair, K or V) moves the run with
// 16-byte loads and stores, four in flight per thread.
#include <cuda_runtime.h>

#include "copy_blocks.h"

namespace pkv {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kThreads) copy_blocks_kernel(const CopyParams p) {
  pdl_trigger();
  pdl_wait();
  const int pair = blockIdx.x >> 1;
  const int64_t src = p.src_dst[2 * pair];
  const int64_t dst = p.src_dst[2 * pair + 1];
  if (src < 0 || src >= p.num_blocks || dst < 0 || dst >= p.num_blocks) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrCopyRange);
    return;
  }
  uint4* base = static_cast<uint4*>((blockIdx.x & 1) ? p.v_cache : p.k_cache);
  const uint4* from = base + src * p.chunks_per_block;
  uint4* to = base + dst * p.chunks_per_block;
  const int64_t n = p.chunks_per_block;
  for (int64_t i = threadIdx.x; i < n; i += kThreads * kUnroll) {
    uint4 r[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (i + u * kThreads < n) r[u] = __ldg(from + i + u * kThreads);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (i + u * kThreads < n) to[i + u * kThreads] = r[u];
  }
}

}  // namespace

cudaError_t launch_copy_blocks(const CopyParams& p, int num_pairs, cudaStream_t stream) {
  return launch_pdl(copy_blocks_kernel, dim3(static_cast<unsigned>(num_pairs) * 2u), dim3(kThreads), 0, stream, p);
}

}  // namespace pkv
