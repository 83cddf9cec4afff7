// kv_append: scatter each new token's K and V into its paged slot.
//
// "从零实现一个 mini vLLM--开篇", section 2: in decode only the new token's K
// and V are computed and appended to the cache; "跟着 Claude Code，我用 Python
// 实现了一个轻量级的 vLLM", section "核心机制一：分页 KV Cache": the cache is
// made of fixed 16-token blocks.  Cache layout [block][kv head][16][head_dim].
//
// A pure copy, bound by launch latency at decode sizes (one token per
// sequence).  Each thread moves one 16-byte chunk of K and the matching chunk
// of V: reads are fully coalesced, writes land as 256-byte (D = 128) or
// 128-byte (D = 64) runs, one per (token, kv head) row.
#include <cuda_runtime.h>

#include "pkv_internal.h"

namespace pkv {
namespace {

__device__ __forceinline__ uint4 load_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__global__ void __launch_bounds__(256) kv_append_kernel(const AppendParams p) {
  pdl_trigger();
  pdl_wait();
  const int chunks_per_row = p.head_dim / 8;                    // 16-byte chunks per (token, head) row
  const int chunks_per_token = p.num_kv_heads * chunks_per_row;
  const int64_t total = p.num_tokens * chunks_per_token;
  const uint4* __restrict__ k = static_cast<const uint4*>(p.k);
  const uint4* __restrict__ v = static_cast<const uint4*>(p.v);
  uint4* __restrict__ kc = static_cast<uint4*>(p.k_cache);
  uint4* __restrict__ vc = static_cast<uint4*>(p.v_cache);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int64_t token = idx / chunks_per_token;
    const int rem = static_cast<int>(idx - token * chunks_per_token);
    const int64_t slot = __ldg(p.slot_mapping + token);
    if (slot < 0) continue;  // padding
    if (slot >= p.num_slots) {
      atomicOr(p.err, kErrSlot);
      continue;
    }
    const int64_t block = slot / kBlockTokens;
    const int offset = static_cast<int>(slot % kBlockTokens);
    const int head = rem / chunks_per_row;
    const int chunk = rem - head * chunks_per_row;
    const int64_t dst = ((block * p.num_kv_heads + head) * kBlockTokens + offset) * chunks_per_row + chunk;
    const uint4 kv_k = load_stream(k + idx);
    const uint4 kv_v = load_stream(v + idx);
    kc[dst] = kv_k;
    vc[dst] = kv_v;
  }
}

}  // namespace

cudaError_t launch_kv_append(const AppendParams& p, int num_sms, cudaStream_t stream) {
  const int64_t total = p.num_tokens * p.num_kv_heads * (p.head_dim / 8);
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(kv_append_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream, p);
}

}  // namespace pkv
