// Internal interface between the C ABI layer (capi.cu) and the kernel
// translation units.  Not installed; the public ABI is include/pagedkv.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

struct CUtensorMap_st;  // cuda.h's tensor-map type (CUtensorMap)

namespace pkv {

constexpr int kBlockTokens = 16;  // tokens per KV block

// Bits of the sticky device error word (same values as PKV_DEVERR_*).
constexpr unsigned kErrSlot = 0x1u;
constexpr unsigned kErrBlockId = 0x2u;
constexpr unsigned kErrLenNegative = 0x4u;
constexpr unsigned kErrLenTooLong = 0x8u;
constexpr unsigned kErrTimeout = 0x10u;
constexpr unsigned kErrCopyRange = 0x20u;
constexpr unsigned kErrPosition = 0x40u;
constexpr unsigned kErrSmemAlign = 0x80u;

struct AppendParams {
  const void* k;
  const void* v;
  const int64_t* slot_mapping;
  void* k_cache;
  void* v_cache;
  unsigned* err;
  int64_t num_tokens;
  int64_t num_slots;  // 16 * num_blocks
  int num_kv_heads;
  int head_dim;
};

struct DecodeParams {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  void* out;
  int32_t* ws_prefix;  // workspace: int32 [num_seqs + 1] block prefix over sequences
  int32_t* ws_pairs;   // workspace: int32 [num_seqs * num_kv_heads][2]: per (sequence, kv head) pair, the
                       // piece holding its first block (times 2, plus the state slot there) and the piece
                       // holding its last block
  float* ws_pieces;    // workspace: fp32 partial states, [num_partitions][2][piece_floats]
  unsigned* err;
  int64_t num_blocks;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int max_blocks_per_seq;
  int num_partitions;
  float qscale;  // scale * log2(e): scores are kept in base-2 units
  // Fused decode step (all null for plain attention): this step's token of every
  // (sequence, kv head), appended at position context_len - 1, and the rotary table.
  const void* k_new;     // bf16 [num_seqs][num_kv_heads][head_dim] or null
  const void* v_new;     // bf16 [num_seqs][num_kv_heads][head_dim]
  const float* cos_sin;  // fp32 [max_position][head_dim] (cos | sin) or null: no RoPE
  int64_t max_position;
};

// Programmatic dependent launch.  Every kernel of this library is launched with
// programmatic stream serialization: it may start (and run its prologue) while
// the previous kernel in the stream drains, and it executes pdl_wait() before
// its first access to global memory, which returns once that kernel has
// completed and its writes are visible.  Each kernel also calls pdl_trigger()
// on entry so that the next one can be scheduled early.  Launched after
// anything else (a copy, another library's kernel) the launch is an ordinary
// stream-ordered one.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem_bytes, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
#endif

// Set the per-host-thread message returned by pkv_last_error_message().
void set_error_message(const char* message);

// kv_append kernel launch.
cudaError_t launch_kv_append(const AppendParams& p, int num_sms, cudaStream_t stream);

// Number of fp32 values in one partial-state piece for these shapes.
int piece_floats(int head_dim, int group);
// Bytes of the workspace header (block prefix, then the pair records) for num_seqs sequences.
size_t workspace_prefix_bytes(int num_seqs);
size_t workspace_header_bytes(int num_seqs, int num_kv_heads);
// Pieces the partition kernel keeps in flight on the current device: one per warp
// (the default num_partitions).
cudaError_t resident_partition_pieces(int head_dim, int group, int num_seqs, int* pieces);
// Tensor map of a cache viewed as [rows = num_blocks * num_kv_heads * 16][head_dim] bf16, box 16 rows x
// 64 dims, 128-byte swizzle (the tensor-copy layout of the prefill kernel and of the decode tensor-core path).
cudaError_t encode_cache_map(CUtensorMap_st* map, const void* cache, int64_t rows, int head_dim);
// One warp waiting on a barrier that nothing completes, for at most limit_ns (the bounded-wait self-test).
cudaError_t launch_bounded_wait_selftest(unsigned* err, unsigned long long limit_ns, cudaStream_t stream);
// Decode kernels.  `group` = num_q_heads / num_kv_heads.
cudaError_t launch_decode_partition(const DecodeParams& p, int head_dim, int group, cudaStream_t stream);
cudaError_t launch_decode_merge(const DecodeParams& p, int head_dim, int group, cudaStream_t stream);

}  // namespace pkv
