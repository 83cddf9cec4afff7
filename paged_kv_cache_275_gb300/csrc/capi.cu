// C ABI of the paged KV-cache hot path (declared in include/pagedkv.h).
//
// Host-side only: argument validation (every host-checkable error returns
// before anything is enqueued), workspace layout, the default partition
// count, kernel dispatch on the caller's stream, the per-device sticky error
// word, and the per-thread error message.  No call allocates device memory.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "pagedkv.h"
#include "copy_blocks.h"
#include "paged_prefill.h"
#include "pkv_internal.h"

// Sticky device error word; one instance per device (module-scope __device__).
static __device__ unsigned int g_pkv_device_error;

namespace {

thread_local char t_message[512] = "";
std::atomic<uint64_t> g_launches{0};

constexpr int kMaxDevices = 64;
std::mutex g_device_mu;
unsigned* g_error_word[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};

pkv_status fail(pkv_status status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_message, sizeof t_message, fmt, ap);
  va_end(ap);
  return status;
}

pkv_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

pkv_status ok() {
  t_message[0] = '\0';
  return PKV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Error word address and SM count of the current device, looked up once per device.
pkv_status device_state(unsigned** err, int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_device_mu);
  if (!g_error_word[dev]) {
    void* addr = nullptr;
    if ((e = cudaGetSymbolAddress(&addr, g_pkv_device_error)) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress(device error word)");
    int count = 0;
    if ((e = cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(multiProcessorCount)");
    g_sm_count[dev] = count;
    g_error_word[dev] = static_cast<unsigned*>(addr);
  }
  if (err) *err = g_error_word[dev];
  if (sms) *sms = g_sm_count[dev];
  return PKV_OK;
}

// Sequences of a decode call handled by one partition + merge launch pair (larger batches are
// cut on the host into consecutive slices of at most this many).
int32_t launch_seqs(int32_t num_seqs) { return num_seqs < PKV_MAX_SEQS ? num_seqs : PKV_MAX_SEQS; }

// Shape checks shared by the workspace query and the attention calls.  `per_launch` is the most
// sequences one kernel launch sees (decode slices the batch; prefill takes it whole).
pkv_status check_shapes(int32_t num_seqs, int32_t per_launch, int32_t num_q_heads, int32_t num_kv_heads,
                        int32_t head_dim, int32_t max_blocks_per_seq) {
  if (num_seqs < 0) return fail(PKV_ERR_INVALID_ARGUMENT, "num_seqs must be >= 0 (got %d)", num_seqs);
  if (num_q_heads <= 0 || num_kv_heads <= 0)
    return fail(PKV_ERR_INVALID_ARGUMENT, "head counts must be positive (q %d, kv %d)", num_q_heads, num_kv_heads);
  if (num_q_heads % num_kv_heads != 0)
    return fail(PKV_ERR_INVALID_ARGUMENT, "num_q_heads %d is not a multiple of num_kv_heads %d", num_q_heads,
                num_kv_heads);
  const int group = num_q_heads / num_kv_heads;
  if (group != 1 && group != 2 && group != 4 && group != 8)
    return fail(PKV_ERR_UNSUPPORTED, "GQA group %d not built (1, 2, 4 or 8)", group);
  if (head_dim != 64 && head_dim != 128)
    return fail(PKV_ERR_UNSUPPORTED, "head_dim %d not built (64 or 128)", head_dim);
  if (max_blocks_per_seq <= 0)
    return fail(PKV_ERR_INVALID_ARGUMENT, "max_blocks_per_seq must be positive (got %d)", max_blocks_per_seq);
  if (static_cast<int64_t>(per_launch) * max_blocks_per_seq * num_kv_heads >= (int64_t{1} << 31) ||
      static_cast<int64_t>(max_blocks_per_seq) * PKV_BLOCK_SIZE >= (int64_t{1} << 31))
    return fail(PKV_ERR_UNSUPPORTED, "sequences per launch * max_blocks_per_seq * num_kv_heads must stay below 2^31");
  return PKV_OK;
}
pkv_status check_decode_shapes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                               int32_t max_blocks_per_seq) {
  return check_shapes(num_seqs, launch_seqs(num_seqs), num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq);
}

constexpr int32_t kMaxPartitions = 1 << 20;

pkv_status default_partitions(int32_t num_seqs, int32_t num_kv_heads, int32_t head_dim, int32_t group,
                              int32_t max_blocks_per_seq, int32_t* out) {
  int pieces = 0;
  const cudaError_t e = pkv::resident_partition_pieces(head_dim, group, num_seqs, &pieces);
  if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
  // Never more pieces than the block stream can have items.
  const int64_t bound = static_cast<int64_t>(num_seqs) * num_kv_heads * max_blocks_per_seq;
  int64_t n = pieces;
  if (n > bound) n = bound;
  if (n > kMaxPartitions) n = kMaxPartitions;
  if (n < 1) n = 1;
  *out = static_cast<int32_t>(n);
  return PKV_OK;
}

size_t workspace_bytes_for(int32_t num_seqs, int32_t num_kv_heads, int32_t head_dim, int32_t group,
                           int32_t num_partitions) {
  return pkv::workspace_header_bytes(num_seqs, num_kv_heads) +
         static_cast<size_t>(num_partitions) * 2 * pkv::piece_floats(head_dim, group) * sizeof(float);
}

// Workspace one decode call needs: the most any of its slices needs (a slice of PKV_MAX_SEQS and,
// when the batch does not divide evenly, the shorter last one; each at its own default partition
// count unless one is given).
pkv_status decode_workspace_need(int32_t num_seqs, int32_t num_kv_heads, int32_t head_dim, int32_t group,
                                 int32_t max_blocks_per_seq, int32_t num_partitions, size_t* need) {
  *need = 0;
  const int32_t sizes[2] = {launch_seqs(num_seqs), num_seqs > PKV_MAX_SEQS ? num_seqs % PKV_MAX_SEQS : 0};
  for (int32_t n : sizes) {
    if (n == 0) continue;
    int32_t parts = num_partitions;
    if (parts == 0)
      if (pkv_status st = default_partitions(n, num_kv_heads, head_dim, group, max_blocks_per_seq, &parts);
          st != PKV_OK)
        return st;
    const size_t b = workspace_bytes_for(n, num_kv_heads, head_dim, group, parts);
    if (b > *need) *need = b;
  }
  return PKV_OK;
}

}  // namespace

// Fused-step inputs of decode_impl (null for plain attention).
struct FusedStep {
  const void* k_new;
  const void* v_new;
  const float* cos_sin;
  int64_t max_position;
};

static pkv_status decode_impl(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                              int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks,
                              int32_t block_size, float scale, void* out, void* workspace, size_t workspace_bytes,
                              int32_t num_partitions, int32_t phases, pkv_stream_t stream, const FusedStep* fused) {
  if (pkv_status st = check_decode_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq);
      st != PKV_OK)
    return st;
  if (block_size != PKV_BLOCK_SIZE)
    return fail(PKV_ERR_UNSUPPORTED, "block_size must be %d (got %d)", PKV_BLOCK_SIZE, block_size);
  if (num_blocks <= 0 || num_blocks > (int64_t{1} << 40))
    return fail(PKV_ERR_INVALID_ARGUMENT, "num_blocks out of range (got %lld)", (long long)num_blocks);
  if (!std::isfinite(scale)) return fail(PKV_ERR_INVALID_ARGUMENT, "scale must be finite");
  if (phases < 1 || phases > PKV_PHASE_ALL) return fail(PKV_ERR_INVALID_ARGUMENT, "phases must be 1, 2 or 3");
  if (num_partitions < 0 || num_partitions > kMaxPartitions)
    return fail(PKV_ERR_INVALID_ARGUMENT, "num_partitions out of range (got %d)", num_partitions);
  if (num_seqs == 0) return ok();
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out || !workspace)
    return fail(PKV_ERR_INVALID_ARGUMENT, "null pointer argument");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return fail(PKV_ERR_INVALID_ARGUMENT, "q, caches, out and workspace must be 16-byte aligned");
  const int group = num_q_heads / num_kv_heads;
  if (num_seqs > PKV_MAX_SEQS && phases != PKV_PHASE_ALL)
    return fail(PKV_ERR_UNSUPPORTED, "phases other than PKV_PHASE_ALL need num_seqs <= PKV_MAX_SEQS (%d)",
                PKV_MAX_SEQS);
  size_t need = 0;
  if (pkv_status st = decode_workspace_need(num_seqs, num_kv_heads, head_dim, group, max_blocks_per_seq,
                                            num_partitions, &need);
      st != PKV_OK)
    return st;
  if (workspace_bytes < need)
    return fail(PKV_ERR_INVALID_ARGUMENT, "workspace too small: %zu bytes given, %zu needed", workspace_bytes, need);

  unsigned* err = nullptr;
  if (pkv_status st = device_state(&err, nullptr); st != PKV_OK) return st;
  // A batch larger than PKV_MAX_SEQS runs as consecutive slices of at most that many sequences,
  // each a partition + merge pair on the same stream and workspace (a slice's merge has read the
  // workspace before the next slice's partition kernel, which waits for it, writes it).
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t q_row = static_cast<size_t>(num_q_heads) * head_dim * 2;  // bytes of one sequence's q / out
  const size_t kv_row = static_cast<size_t>(num_kv_heads) * head_dim * 2;
  for (int32_t s0 = 0; s0 < num_seqs; s0 += PKV_MAX_SEQS) {
    const int32_t n = launch_seqs(num_seqs - s0);
    int32_t parts = num_partitions;
    if (parts == 0)
      if (pkv_status st = default_partitions(n, num_kv_heads, head_dim, group, max_blocks_per_seq, &parts);
          st != PKV_OK)
        return st;
    pkv::DecodeParams p{};
    p.q = static_cast<const unsigned char*>(q) + s0 * q_row;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables + static_cast<size_t>(s0) * max_blocks_per_seq;
    p.context_lens = context_lens + s0;
    p.out = static_cast<unsigned char*>(out) + s0 * q_row;
    p.ws_prefix = static_cast<int32_t*>(workspace);
    p.ws_pairs = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(workspace) + pkv::workspace_prefix_bytes(n));
    p.ws_pieces = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) +
                                           pkv::workspace_header_bytes(n, num_kv_heads));
    p.err = err;
    p.num_blocks = num_blocks;
    p.num_seqs = n;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_partitions = parts;
    p.qscale = scale * 1.4426950408889634f;
    if (fused) {
      p.k_new = static_cast<const unsigned char*>(fused->k_new) + s0 * kv_row;
      p.v_new = static_cast<const unsigned char*>(fused->v_new) + s0 * kv_row;
      p.cos_sin = fused->cos_sin;
      p.max_position = fused->max_position;
    }
    if (phases & PKV_PHASE_PARTITION) {
      const cudaError_t e = pkv::launch_decode_partition(p, head_dim, group, s);
      if (e != cudaSuccess) return cuda_fail(e, "partition kernel launch");
      g_launches.fetch_add(1);
    }
    if (phases & PKV_PHASE_MERGE) {
      const cudaError_t e = pkv::launch_decode_merge(p, head_dim, group, s);
      if (e != cudaSuccess) return cuda_fail(e, "merge kernel launch");
      g_launches.fetch_add(1);
    }
  }
  return ok();
}


void pkv::set_error_message(const char* message) { snprintf(t_message, sizeof t_message, "%s", message); }

extern "C" {

const char* pkv_last_error_message(void) { return t_message; }

uint64_t pkv_kernel_launch_count(void) { return g_launches.load(); }

pkv_status pkv_kv_append(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                         int32_t num_kv_heads, int32_t head_dim, void* k_cache, void* v_cache, int64_t num_blocks,
                         int32_t block_size, pkv_stream_t stream) {
  if (num_tokens < 0) return fail(PKV_ERR_INVALID_ARGUMENT, "num_tokens must be >= 0 (got %lld)", (long long)num_tokens);
  if (num_kv_heads <= 0) return fail(PKV_ERR_INVALID_ARGUMENT, "num_kv_heads must be positive (got %d)", num_kv_heads);
  if (head_dim != 64 && head_dim != 128)
    return fail(PKV_ERR_UNSUPPORTED, "head_dim %d not built (64 or 128)", head_dim);
  if (block_size != PKV_BLOCK_SIZE)
    return fail(PKV_ERR_UNSUPPORTED, "block_size must be %d (got %d)", PKV_BLOCK_SIZE, block_size);
  if (num_blocks <= 0 || num_blocks > (int64_t{1} << 40))
    return fail(PKV_ERR_INVALID_ARGUMENT, "num_blocks out of range (got %lld)", (long long)num_blocks);
  if (num_tokens > (int64_t{1} << 32))
    return fail(PKV_ERR_UNSUPPORTED, "num_tokens %lld too large", (long long)num_tokens);
  if (num_tokens == 0) return ok();
  if (!k || !v || !slot_mapping || !k_cache || !v_cache)
    return fail(PKV_ERR_INVALID_ARGUMENT, "null pointer argument");
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return fail(PKV_ERR_INVALID_ARGUMENT, "k, v and the caches must be 16-byte aligned, slot_mapping 8-byte aligned");
  unsigned* err = nullptr;
  int sms = 0;
  if (pkv_status st = device_state(&err, &sms); st != PKV_OK) return st;
  pkv::AppendParams p{};
  p.k = k;
  p.v = v;
  p.slot_mapping = slot_mapping;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.err = err;
  p.num_tokens = num_tokens;
  p.num_slots = num_blocks * PKV_BLOCK_SIZE;
  p.num_kv_heads = num_kv_heads;
  p.head_dim = head_dim;
  const cudaError_t e = pkv::launch_kv_append(p, sms, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
  g_launches.fetch_add(1);
  return ok();
}

pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const int64_t* src_dst, int32_t num_pairs,
                           int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks, pkv_stream_t stream) {
  if (num_pairs < 0) return fail(PKV_ERR_INVALID_ARGUMENT, "num_pairs must be >= 0 (got %d)", num_pairs);
  if (num_pairs > (1 << 30)) return fail(PKV_ERR_UNSUPPORTED, "num_pairs %d too large", num_pairs);
  if (num_kv_heads <= 0) return fail(PKV_ERR_INVALID_ARGUMENT, "num_kv_heads must be positive (got %d)", num_kv_heads);
  if (head_dim != 64 && head_dim != 128)
    return fail(PKV_ERR_UNSUPPORTED, "head_dim %d not built (64 or 128)", head_dim);
  if (num_blocks <= 0 || num_blocks > (int64_t{1} << 40))
    return fail(PKV_ERR_INVALID_ARGUMENT, "num_blocks out of range (got %lld)", (long long)num_blocks);
  if (num_pairs == 0) return ok();
  if (!k_cache || !v_cache || !src_dst) return fail(PKV_ERR_INVALID_ARGUMENT, "null pointer argument");
  if (!aligned16(k_cache) || !aligned16(v_cache) || (reinterpret_cast<uintptr_t>(src_dst) & 7u))
    return fail(PKV_ERR_INVALID_ARGUMENT, "caches must be 16-byte aligned, src_dst 8-byte aligned");
  unsigned* err = nullptr;
  if (pkv_status st = device_state(&err, nullptr); st != PKV_OK) return st;
  pkv::CopyParams p{};
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.src_dst = src_dst;
  p.err = err;
  p.num_blocks = num_blocks;
  p.chunks_per_block = static_cast<int64_t>(num_kv_heads) * PKV_BLOCK_SIZE * head_dim / 8;
  const cudaError_t e = pkv::launch_copy_blocks(p, num_pairs, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "copy_blocks launch");
  g_launches.fetch_add(1);
  return ok();
}

pkv_status pkv_selftest_wait_timeout(uint64_t limit_ns, pkv_stream_t stream) {
  if (limit_ns < 1000 || limit_ns > 1000000000ull)
    return fail(PKV_ERR_INVALID_ARGUMENT, "limit_ns must lie in [1e3, 1e9] (got %llu)", (unsigned long long)limit_ns);
  unsigned* err = nullptr;
  if (pkv_status st = device_state(&err, nullptr); st != PKV_OK) return st;
  const cudaError_t e =
      pkv::launch_bounded_wait_selftest(err, limit_ns, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  g_launches.fetch_add(1);
  return ok();
}

namespace {
constexpr int32_t kMaxPrefillSplits = 32;  // the merge reads one split per lane

pkv_status prefill_impl(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                        int32_t max_blocks_per_seq, const int32_t* context_lens, const int32_t* query_start,
                        int32_t max_query_len, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                        int32_t head_dim, int64_t num_blocks, int32_t block_size, float scale, void* out,
                        int32_t num_splits, void* workspace, size_t workspace_bytes, pkv_stream_t stream) {
  if (num_splits < 1 || num_splits > kMaxPrefillSplits)
    return fail(PKV_ERR_INVALID_ARGUMENT, "num_splits must be in [1, %d] (got %d)", kMaxPrefillSplits, num_splits);
  if (static_cast<int64_t>(num_seqs) * num_splits > 65535)
    return fail(PKV_ERR_UNSUPPORTED, "num_seqs * num_splits = %lld exceeds 65535 (one grid row of CTAs each)",
                static_cast<long long>(num_seqs) * num_splits);
  if (pkv_status st = check_shapes(num_seqs, num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq);
      st != PKV_OK)
    return st;
  if (block_size != PKV_BLOCK_SIZE)
    return fail(PKV_ERR_UNSUPPORTED, "block_size must be %d (got %d)", PKV_BLOCK_SIZE, block_size);
  if (num_blocks <= 0 || num_blocks * num_kv_heads * PKV_BLOCK_SIZE >= (int64_t{1} << 31))
    return fail(PKV_ERR_UNSUPPORTED, "num_blocks * num_kv_heads * 16 must be in (0, 2^31) (got %lld blocks)",
                (long long)num_blocks);
  if (!std::isfinite(scale)) return fail(PKV_ERR_INVALID_ARGUMENT, "scale must be finite");
  if (max_query_len < 0) return fail(PKV_ERR_INVALID_ARGUMENT, "max_query_len must be >= 0 (got %d)", max_query_len);
  // A CTA takes two 128-row tiles of 128 / G chunk tokens each; its sequence's tiles are one grid dimension.
  const int32_t cta_tokens = 256 / (num_q_heads / num_kv_heads);
  if ((static_cast<int64_t>(max_query_len) + cta_tokens - 1) / cta_tokens > 65535)
    return fail(PKV_ERR_UNSUPPORTED, "max_query_len %d exceeds 65535 CTAs of %d chunk tokens", max_query_len,
                cta_tokens);
  if (num_seqs == 0 || max_query_len == 0) return ok();
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start || !out)
    return fail(PKV_ERR_INVALID_ARGUMENT, "null pointer argument");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(query_start) & 3u))
    return fail(PKV_ERR_INVALID_ARGUMENT, "q, caches and out must be 16-byte aligned");
  if (num_splits > 1) {
    const size_t need =
        pkv::prefill_workspace_bytes(num_seqs, max_query_len, num_q_heads, num_kv_heads, head_dim, num_splits);
    if (!workspace || workspace_bytes < need)
      return fail(PKV_ERR_INVALID_ARGUMENT, "workspace too small: %zu bytes given, %zu needed", workspace_bytes, need);
    if (!aligned16(workspace)) return fail(PKV_ERR_INVALID_ARGUMENT, "workspace must be 16-byte aligned");
  }
  unsigned* err = nullptr;
  if (pkv_status st = device_state(&err, nullptr); st != PKV_OK) return st;
  pkv::PrefillParams p{};
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.query_start = query_start;
  p.out = out;
  p.err = err;
  p.num_blocks = num_blocks;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.max_query_len = max_query_len;
  p.scale = scale;
  if (num_splits > 1) {
    p.num_splits = num_splits;
    p.ws = static_cast<float*>(workspace);
  }
  const cudaError_t e = pkv::launch_paged_prefill(p, head_dim, num_q_heads / num_kv_heads, max_query_len,
                                                  reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "prefill kernel launch");
  g_launches.fetch_add(num_splits > 1 ? 2 : 1);
  return ok();
}
}  // namespace

pkv_status pkv_paged_prefill_attention(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* context_lens, const int32_t* query_start,
                                       int32_t max_query_len, int32_t num_seqs, int32_t num_q_heads,
                                       int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks, int32_t block_size,
                                       float scale, void* out, pkv_stream_t stream) {
  return prefill_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, query_start, max_query_len,
                      num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale, out, 1, nullptr, 0,
                      stream);
}

pkv_status pkv_paged_prefill_attention_split(const void* q, const void* k_cache, const void* v_cache,
                                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                                             const int32_t* context_lens, const int32_t* query_start,
                                             int32_t max_query_len, int32_t num_seqs, int32_t num_q_heads,
                                             int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks,
                                             int32_t block_size, float scale, void* out, int32_t num_splits,
                                             void* workspace, size_t workspace_bytes, pkv_stream_t stream) {
  return prefill_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, query_start, max_query_len,
                      num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale, out, num_splits,
                      workspace, workspace_bytes, stream);
}

pkv_status pkv_prefill_default_splits(int32_t num_seqs, int32_t max_query_len, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t* num_splits) {
  if (!num_splits) return fail(PKV_ERR_INVALID_ARGUMENT, "num_splits is null");
  if (num_seqs < 0 || max_query_len < 0) return fail(PKV_ERR_INVALID_ARGUMENT, "num_seqs and max_query_len must be >= 0");
  if (pkv_status st = check_shapes(num_seqs, num_seqs, num_q_heads, num_kv_heads, 128, 1); st != PKV_OK) return st;
  int sms = 0;
  if (pkv_status st = device_state(nullptr, &sms); st != PKV_OK) return st;
  // The most splits that keep every CTA of the call in one wave (one CTA per SM), at most 32, and
  // within the 65535 grid rows; 1 when the call already fills the GPU.
  const int64_t cta = pkv::prefill_cta_tokens(num_q_heads / num_kv_heads);
  const int64_t ctas = static_cast<int64_t>(num_seqs) * num_kv_heads * ((max_query_len + cta - 1) / cta);
  int64_t n = ctas > 0 ? sms / ctas : 1;
  if (n > kMaxPrefillSplits) n = kMaxPrefillSplits;
  if (num_seqs > 0 && n > 65535 / num_seqs) n = 65535 / num_seqs;
  if (n < 1) n = 1;
  *num_splits = static_cast<int32_t>(n);
  return ok();
}

pkv_status pkv_prefill_workspace_size(int32_t num_seqs, int32_t max_query_len, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim, int32_t num_splits, size_t* bytes) {
  if (!bytes) return fail(PKV_ERR_INVALID_ARGUMENT, "bytes must not be null");
  if (num_seqs < 0 || max_query_len < 0) return fail(PKV_ERR_INVALID_ARGUMENT, "num_seqs and max_query_len must be >= 0");
  if (num_splits < 1 || num_splits > kMaxPrefillSplits)
    return fail(PKV_ERR_INVALID_ARGUMENT, "num_splits must be in [1, %d] (got %d)", kMaxPrefillSplits, num_splits);
  if (pkv_status st = check_shapes(num_seqs, num_seqs, num_q_heads, num_kv_heads, head_dim, 1); st != PKV_OK) return st;
  *bytes = pkv::prefill_workspace_bytes(num_seqs, max_query_len, num_q_heads, num_kv_heads, head_dim, num_splits);
  return ok();
}

pkv_status pkv_decode_default_partitions(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t max_blocks_per_seq, int32_t* num_partitions) {
  if (!num_partitions) return fail(PKV_ERR_INVALID_ARGUMENT, "num_partitions is null");
  if (pkv_status st = check_decode_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq);
      st != PKV_OK)
    return st;
  if (pkv_status st = default_partitions(launch_seqs(num_seqs), num_kv_heads, head_dim, num_q_heads / num_kv_heads,
                                         max_blocks_per_seq, num_partitions);
      st != PKV_OK)
    return st;
  return ok();
}

pkv_status pkv_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                     int32_t max_blocks_per_seq, int32_t num_partitions, size_t* bytes) {
  if (!bytes) return fail(PKV_ERR_INVALID_ARGUMENT, "bytes is null");
  if (pkv_status st = check_decode_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq);
      st != PKV_OK)
    return st;
  if (num_partitions < 0 || num_partitions > kMaxPartitions)
    return fail(PKV_ERR_INVALID_ARGUMENT, "num_partitions out of range (got %d)", num_partitions);
  size_t need = 0;
  if (pkv_status st = decode_workspace_need(num_seqs, num_kv_heads, head_dim, num_q_heads / num_kv_heads,
                                            max_blocks_per_seq, num_partitions, &need);
      st != PKV_OK)
    return st;
  *bytes = need;
  return ok();
}

pkv_status pkv_paged_decode_attention_split(const void* q, const void* k_cache, const void* v_cache,
                                            const int32_t* block_tables, int32_t max_blocks_per_seq,
                                            const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                                            int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks,
                                            int32_t block_size, float scale, void* out, void* workspace,
                                            size_t workspace_bytes, int32_t num_partitions, int32_t phases,
                                            pkv_stream_t stream) {
  return decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                     num_kv_heads, head_dim, num_blocks, block_size, scale, out, workspace, workspace_bytes,
                     num_partitions, phases, stream, nullptr);
}

pkv_status pkv_decode_step(const void* q, const void* k_new, const void* v_new, const float* cos_sin,
                           int64_t max_position, void* k_cache, void* v_cache, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                           int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks,
                           int32_t block_size, float scale, void* out, void* workspace, size_t workspace_bytes,
                           pkv_stream_t stream) {
  if (num_seqs > 0) {
    if (!k_new || !v_new) return fail(PKV_ERR_INVALID_ARGUMENT, "null pointer argument");
    if (!aligned16(k_new) || !aligned16(v_new) || (cos_sin && !aligned16(cos_sin)))
      return fail(PKV_ERR_INVALID_ARGUMENT, "k_new, v_new and cos_sin must be 16-byte aligned");
    if (cos_sin && max_position <= 0)
      return fail(PKV_ERR_INVALID_ARGUMENT, "max_position must be positive with a rotary table (got %lld)",
                  (long long)max_position);
  }
  const FusedStep fused{k_new, v_new, cos_sin, cos_sin ? max_position : 0};
  return decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                     num_kv_heads, head_dim, num_blocks, block_size, scale, out, workspace, workspace_bytes, 0,
                     PKV_PHASE_ALL, stream, &fused);
}

pkv_status pkv_paged_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks, int32_t block_size,
                                      float scale, void* out, void* workspace, size_t workspace_bytes,
                                      pkv_stream_t stream) {
  return pkv_paged_decode_attention_split(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                          num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size,
                                          scale, out, workspace, workspace_bytes, 0, PKV_PHASE_ALL, stream);
}

pkv_status pkv_get_and_clear_device_error(uint32_t* bits, pkv_stream_t stream) {
  if (!bits) return fail(PKV_ERR_INVALID_ARGUMENT, "bits is null");
  unsigned* err = nullptr;
  if (pkv_status st = device_state(&err, nullptr); st != PKV_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned host = 0;
  if ((e = cudaMemcpyAsync(&host, err, sizeof host, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_fail(e, "reading the device error word");
  if ((e = cudaMemsetAsync(err, 0, sizeof(unsigned), s)) != cudaSuccess)
    return cuda_fail(e, "clearing the device error word");
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  *bits = host;
  return ok();
}

}  // extern "C"
