// Decode attention for callers that cannot allocate device memory.
//
// The regular entry point needs a caller-owned workspace.  Some callers
// cannot provide one: a plugin loaded into a host process that owns every
// device allocation, or a serving loop where cudaMalloc would implicitly
// synchronise the device and stall other streams.  This file gives them
// pkv_paged_decode_attention_static, which uses a fixed scratch area built
// into the library instead.
//
// The scratch area is a file-scope __device__ array: every GPU that loads the
// library holds PKV_STATIC_WORKSPACE_BYTES of it until the process exits.  In
// host code the array's name is only a host-side stand-in, so its device
// address is looked up with cudaGetSymbolAddress, once per device, on the
// first call made with that device current; make that first call before
// any stream capture.  Nothing here calls cudaMalloc, cudaFree or any other
// allocating routine.
//
// Every call shares the one array, and the array keeps what the last call
// left in it.  The attention kernels need nothing in it to start at zero:
// the partition kernel writes the block prefix and every partial state
// before the merge kernel reads them.  Calls that can overlap on the GPU
// (different streams, different host threads) race on the array; serialise
// them on one stream.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "pagedkv.h"
#include "pkv_internal.h"

static __device__ __align__(256) unsigned char g_pkv_static_workspace[PKV_STATIC_WORKSPACE_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
pkv_status static_workspace_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  char msg[256];
  if (e != cudaSuccess) {
    snprintf(msg, sizeof msg, "cudaGetDevice: %s", cudaGetErrorString(e));
    pkv::set_error_message(msg);
    return PKV_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    snprintf(msg, sizeof msg, "device ordinal %d out of range", dev);
    pkv::set_error_message(msg);
    return PKV_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_addr[dev]) {
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_pkv_static_workspace);
    if (e != cudaSuccess || addr == nullptr) {
      snprintf(msg, sizeof msg, "cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(e));
      pkv::set_error_message(msg);
      return PKV_ERR_CUDA;
    }
    g_static_addr[dev] = addr;
  }
  *out = g_static_addr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_paged_decode_attention_static(const void* q, const void* k_cache, const void* v_cache,
                                                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                         const int32_t* context_lens, int32_t num_seqs,
                                                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                                         int64_t num_blocks, int32_t block_size, float scale,
                                                         void* out, pkv_stream_t stream) {
  // Same shapes, same default partition count and same kernels as pkv_paged_decode_attention.
  size_t need = 0;
  pkv_status st = pkv_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, 0,
                                            &need);
  if (st != PKV_OK) return st;
  if (need > PKV_STATIC_WORKSPACE_BYTES) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "these shapes need %zu bytes of scratch; the built-in static area holds %zu "
             "(PKV_STATIC_WORKSPACE_BYTES): use pkv_paged_decode_attention with a workspace",
             need, static_cast<size_t>(PKV_STATIC_WORKSPACE_BYTES));
    pkv::set_error_message(msg);
    return PKV_ERR_UNSUPPORTED;
  }
  void* ws = nullptr;
  if (num_seqs > 0) {
    st = static_workspace_address(&ws);
    if (st != PKV_OK) return st;
  }
  return pkv_paged_decode_attention_split(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                          num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size,
                                          scale, out, ws, PKV_STATIC_WORKSPACE_BYTES, 0, PKV_PHASE_ALL, stream);
}
