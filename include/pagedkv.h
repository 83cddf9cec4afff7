/*
 * pagedkv.h -- C ABI of the paged KV-cache hot path on one GB300 (sm_103a).
 *
 * Two operations, after the pages on a mini vLLM inference engine:
 *
 *   kv_append               "从零实现一个 mini vLLM--开篇", section 2
 *                           ("LLM 推理到底在慢什么"): in decode only the new
 *                           token's K and V are computed and appended to the
 *                           cache.  The cache is cut into fixed 16-token
 *                           blocks ("跟着 Claude Code，我用 Python 实现了一个
 *                           轻量级的 vLLM", section "核心机制一：分页 KV Cache").
 *   paged_decode_attention  the same series, section 5 (phases 4 and 5): a
 *                           request owns a block table; its tokens are
 *                           logically contiguous and physically scattered, and
 *                           attention finds the real K and V through the block
 *                           table; every decode step attends over all cached
 *                           tokens (section 2).  The result is the plain
 *                           definition softmax(scale * q K^T) V per q head.
 *
 * Conventions (all tensors row-major and contiguous, caller-owned device
 * memory; the library allocates nothing and keeps no pointer after a call):
 *
 *   block size         16 tokens (PKV_BLOCK_SIZE); other values are rejected.
 *   k_cache, v_cache   bf16 [num_blocks][num_kv_heads][16][head_dim]: one
 *                      (block, kv head) tile is one contiguous 16 * head_dim
 *                      run.  Slot s is block s / 16, offset s % 16.
 *   head_dim           64 or 128.
 *   GQA                q head h reads kv head h / (num_q_heads / num_kv_heads);
 *                      num_q_heads / num_kv_heads must be 1, 2, 4 or 8.
 *   q, out             bf16 [num_seqs][num_q_heads][head_dim].
 *   block_tables       int32 [num_seqs][max_blocks_per_seq]; entries past
 *                      ceil(context_len / 16) are never read (may hold -1).
 *   context_lens       int32 [num_seqs]: number of cached tokens of each
 *                      sequence, including the token appended in this step
 *                      (append first, then attend; no mask).
 *   arithmetic         bf16 inputs widened exactly to fp32, fp32 accumulation
 *                      and online softmax, one round-to-nearest-even to bf16.
 *   alignment          every pointer argument 16-byte aligned.
 *   streams            every call only enqueues work on `stream` (a
 *                      cudaStream_t; NULL means the legacy default stream) and
 *                      never synchronises, except
 *                      pkv_get_and_clear_device_error.  The current CUDA
 *                      device must own every pointer.
 *
 * Errors.  A call returns PKV_OK or an error status; on error nothing was
 * enqueued and pkv_last_error_message() (per host thread) says why.
 * Conditions only the device can see (a slot past the pool, a block id
 * outside [0, num_blocks), a context length outside [0, 16 * max_blocks_per_seq],
 * a pipeline wait that ran out of time) never fault: the element is skipped
 * or clamped, its output is unspecified, and a bit is set in a sticky
 * per-device error word that pkv_get_and_clear_device_error() returns.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_BLOCK_SIZE 16

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARGUMENT = 1, /* null / misaligned pointer, bad size, workspace too small */
    PKV_ERR_UNSUPPORTED = 2,      /* head_dim, GQA group, block size or batch outside what is built */
    PKV_ERR_CUDA = 3,             /* a CUDA runtime call failed (message has the CUDA error) */
    PKV_ERR_NO_FREE_BLOCKS = 4    /* block manager: the pool cannot supply the blocks a call needs (nothing changed) */
} pkv_status;

/* Bits of the sticky device error word. */
#define PKV_DEVERR_SLOT_OUT_OF_RANGE 0x1u     /* kv_append: slot >= 16 * num_blocks (token skipped) */
#define PKV_DEVERR_BLOCK_ID_OUT_OF_RANGE 0x2u /* attention: table entry outside [0, num_blocks) (block 0 read instead) */
#define PKV_DEVERR_CONTEXT_LEN_NEGATIVE 0x4u  /* attention: context_len < 0 (treated as 0) */
#define PKV_DEVERR_CONTEXT_LEN_TOO_LONG 0x8u  /* attention: context_len > 16 * max_blocks_per_seq (clamped) */
#define PKV_DEVERR_PIPELINE_TIMEOUT 0x10u     /* attention: a shared-memory pipeline wait gave up (partition skipped) */
#define PKV_DEVERR_COPY_OUT_OF_RANGE 0x20u    /* copy_blocks: a source or destination block outside the pool (pair skipped) */
#define PKV_DEVERR_POSITION_OUT_OF_TABLE 0x40u /* decode_step: context_len - 1 >= max_position (last table row used) */
#define PKV_DEVERR_SMEM_ALIGNMENT 0x80u        /* prefill: dynamic shared memory not 1024-byte aligned (tile skipped) */

/* Most sequences one partition + merge launch pair handles.  A decode call with more runs as
   consecutive slices of at most PKV_MAX_SEQS sequences, in order on the same stream and workspace
   (the workspace query sizes it for the largest slice); only the split-phase entry point with a
   phase mask other than PKV_PHASE_ALL keeps the limit. */
#define PKV_MAX_SEQS 4096

/* Phases of one attention call (see pkv_paged_decode_attention_split). */
#define PKV_PHASE_PARTITION 0x1
#define PKV_PHASE_MERGE 0x2
#define PKV_PHASE_ALL 0x3

typedef struct CUstream_st* pkv_stream_t; /* the same type as cudaStream_t */

/*
 * Append this step's K and V into their paged slots.
 *
 * For every token i in [0, num_tokens) with s = slot_mapping[i] >= 0 and every
 * kv head h, copies the bits of k[i][h][:] into k_cache[s / 16][h][s % 16][:]
 * and v[i][h][:] into v_cache[s / 16][h][s % 16][:].  A negative slot is
 * padding and is skipped.  Slots must be distinct (duplicates give an
 * unspecified one of the writes).  Bit-exact: no arithmetic on the values.
 *
 *   k, v          device, bf16 [num_tokens][num_kv_heads][head_dim]
 *   slot_mapping  device, int64 [num_tokens]
 *   k_cache, v_cache  device, bf16 [num_blocks][num_kv_heads][16][head_dim], written in place
 *   block_size    must be 16
 *
 * num_tokens == 0 is a no-op.  Device-side: slot >= 16 * num_blocks sets
 * PKV_DEVERR_SLOT_OUT_OF_RANGE and the token is skipped.
 */
pkv_status pkv_kv_append(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                         int32_t num_kv_heads, int32_t head_dim, void* k_cache, void* v_cache,
                         int64_t num_blocks, int32_t block_size, pkv_stream_t stream);

/*
 * Bytes of device workspace one attention call needs.
 *
 * This replaces a query of the form size_t workspace_bytes(num_seqs,
 * num_q_heads, head_dim, max_blocks_per_seq, block_size): the workspace holds
 * two partial softmax states per piece, each G * head_dim + 4 * ceil(G / 2)
 * floats (G = num_q_heads / num_kv_heads), so it depends on num_kv_heads and
 * on num_partitions; the default num_partitions depends on the device, so the
 * query can fail and returns a status, the size through `bytes`.  block_size
 * is always 16 and is checked by the attention call.
 *
 * num_partitions is the number of contiguous, equal-length pieces the whole
 * batch's (sequence, kv head, block) stream is cut into (one warp each; a
 * piece that covers only part of a (sequence, kv head) pair leaves a partial
 * softmax state that the merge phase combines).  0 picks the default for the
 * current device: the number of warps the GPU keeps resident.  The same
 * num_partitions must be passed to the attention call.  Requires a CUDA device
 * when num_partitions == 0.  With num_seqs > PKV_MAX_SEQS the batch runs in
 * slices and the size is the largest slice's need (each slice's stream is cut
 * into num_partitions pieces, or its own default count).
 */
pkv_status pkv_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t max_blocks_per_seq, int32_t num_partitions,
                                     size_t* bytes);

/* The default num_partitions for these shapes on the current device (what 0 means; for
   num_seqs > PKV_MAX_SEQS, that of a full slice of PKV_MAX_SEQS sequences). */
pkv_status pkv_decode_default_partitions(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t max_blocks_per_seq,
                                         int32_t* num_partitions);

/*
 * Paged decode attention:
 *
 *   out[b][h][:] = sum_t softmax_t(scale * <q[b][h], K_t>) * V_t,   t < context_lens[b]
 *   K_t = k_cache[block_tables[b][t / 16]][h / G][t % 16][:]  (G = num_q_heads / num_kv_heads)
 *   V_t = v_cache[block_tables[b][t / 16]][h / G][t % 16][:]
 *
 * context_lens[b] == 0 writes zeros.  num_seqs == 0 is a no-op.
 *
 *   q             device, bf16 [num_seqs][num_q_heads][head_dim]
 *   k_cache, v_cache  device, bf16 [num_blocks][num_kv_heads][16][head_dim]
 *   block_tables  device, int32 [num_seqs][max_blocks_per_seq]
 *   context_lens  device, int32 [num_seqs]
 *   out           device, bf16 [num_seqs][num_q_heads][head_dim] (written)
 *   workspace     device scratch of at least pkv_decode_workspace_size(..., 0, ...)
 *                 bytes, 16-byte aligned, owned by the caller; its contents
 *                 are scratch and need no initialisation.  Two calls that
 *                 may run concurrently need two workspaces.
 *
 * Enqueues two kernels: the partition kernel (every warp streams one piece of
 * the batch's block stream through a TMA-fed shared-memory ring and writes a
 * finished output row or a partial softmax state) and the merge kernel.
 * Arithmetic: fp32 accumulation, one round-to-nearest-even to bf16 at the end.
 * With eight q heads per kv head the two products run on the tensor cores
 * (fp32 accumulation; each softmax weight enters P.V as two bf16 parts, about
 * 16 significant bits); with four or fewer the weights stay in fp32.
 *
 * If pkv_get_and_clear_device_error reports PKV_DEVERR_PIPELINE_TIMEOUT after
 * the call, the outputs of the call are undefined: a piece whose wait gave up
 * wrote no partial state, and the merge combined whatever the workspace held.
 */
pkv_status pkv_paged_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks,
                                      int32_t block_size, float scale, void* out, void* workspace,
                                      size_t workspace_bytes, pkv_stream_t stream);

/*
 * The same call with an explicit num_partitions (> 0, or 0 for the default)
 * and a phase mask.  PKV_PHASE_PARTITION enqueues only the partition kernel,
 * PKV_PHASE_MERGE only the merge kernel (which reads what the partition phase
 * left in the workspace, so it must follow a partition phase with identical
 * arguments on the same workspace), PKV_PHASE_ALL both.  The result does not
 * depend on num_partitions beyond fp32 rounding.  A phase mask other than
 * PKV_PHASE_ALL needs num_seqs <= PKV_MAX_SEQS (PKV_ERR_UNSUPPORTED otherwise:
 * the slices of a larger batch share the workspace).
 */
pkv_status pkv_paged_decode_attention_split(const void* q, const void* k_cache, const void* v_cache,
                                            const int32_t* block_tables, int32_t max_blocks_per_seq,
                                            const int32_t* context_lens, int32_t num_seqs,
                                            int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                            int64_t num_blocks, int32_t block_size, float scale, void* out,
                                            void* workspace, size_t workspace_bytes, int32_t num_partitions,
                                            int32_t phases, pkv_stream_t stream);

/* Bytes of the built-in scratch area behind pkv_paged_decode_attention_static (per device). */
#define PKV_STATIC_WORKSPACE_BYTES (16u * 1024u * 1024u)

/*
 * Decode attention without a caller workspace, for callers that cannot
 * allocate device memory: for example a plugin running inside a host process
 * that owns every device allocation, or a serving loop in which a cudaMalloc
 * would implicitly synchronise the device and stall its other streams.  The
 * source pages have no counterpart to this entry point.
 *
 * Same arguments, shapes and result as pkv_paged_decode_attention, minus the
 * workspace.  Scratch comes from one fixed array of PKV_STATIC_WORKSPACE_BYTES
 * inside the library, which every GPU that loads the library holds until the
 * process exits.  Shapes whose scratch need is larger return
 * PKV_ERR_UNSUPPORTED with a message (at the default partition count on a
 * 152-SM GB300 the built shapes need at most about 10.4 MB, eight q heads per
 * kv head at head_dim 128 with 4096 sequences of 8 kv heads; four heads about
 * 5.4 MB).  The
 * first call on a device,
 * with that device current, looks up the array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * Every call shares the array and it keeps the last call's contents (nothing
 * in it needs to start at zero), so calls that may overlap on the GPU race:
 * serialise them on one stream.  Calls no allocating routine.  As for
 * pkv_paged_decode_attention, a PKV_DEVERR_PIPELINE_TIMEOUT bit after the call
 * means its outputs are undefined (here the merge may combine an earlier
 * call's states left in the shared array).
 */
pkv_status pkv_paged_decode_attention_static(const void* q, const void* k_cache, const void* v_cache,
                                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                                             const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                                             int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks,
                                             int32_t block_size, float scale, void* out, pkv_stream_t stream);

/*
 * One fused decode step: RoPE, append and attention in the two attention
 * kernels, with no separate append launch.  "跟着 Claude Code，我用 Python 实现了
 * 一个轻量级的 vLLM", section "核心机制五": a full-attention layer runs QKV
 * projection + RoPE + KV cache + SDPA; "从零实现一个 mini vLLM--开篇",
 * section 2: decode appends the new token's K/V, then attends over all of it.
 *
 * For every sequence b with L = context_lens[b] >= 1 (L counts the new token,
 * at position L - 1):
 *   q'      = RoPE(q[b], L - 1)               rounded to bf16
 *   k'      = RoPE(k_new[b], L - 1)           rounded to bf16
 *   slot    = block_tables[b][(L-1) / 16] * 16 + (L-1) % 16
 *   k_cache / v_cache at slot := k', v_new[b]   (all kv heads)
 *   out[b]  = paged decode attention of q' over the L tokens (as
 *             pkv_paged_decode_attention)
 * RoPE is the rotate-half form: for i < D/2, with c = cos_sin[pos][i] and
 * s = cos_sin[pos][D/2 + i], x'[i] = x[i] c - x[i + D/2] s and
 * x'[i + D/2] = x[i + D/2] c + x[i] s, each product and sum one fp32 operation
 * rounded to nearest (no fused multiply-add).  cos_sin == NULL skips RoPE (the
 * step is then exactly pkv_kv_append + pkv_paged_decode_attention).
 *
 *   q             device, bf16 [num_seqs][num_q_heads][head_dim] (not modified)
 *   k_new, v_new  device, bf16 [num_seqs][num_kv_heads][head_dim]
 *   cos_sin       device, fp32 [max_position][head_dim], or NULL
 *   workspace     as for pkv_paged_decode_attention (same size)
 * The block holding position L - 1 must belong to sequence b alone (run the
 * block manager's copy-on-write first).  L == 0 writes zeros and appends
 * nothing.  Device-side: L - 1 >= max_position sets
 * PKV_DEVERR_POSITION_OUT_OF_TABLE and uses the last table row.
 */
pkv_status pkv_decode_step(const void* q, const void* k_new, const void* v_new, const float* cos_sin,
                           int64_t max_position, void* k_cache, void* v_cache, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                           int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks,
                           int32_t block_size, float scale, void* out, void* workspace, size_t workspace_bytes,
                           pkv_stream_t stream);

/*
 * Chunked paged prefill attention, on the tensor cores.  "从零实现一个 mini
 * vLLM--开篇", section 2: prefill runs the prompt at once and keeps every
 * layer's K and V; section 5 lists chunked prefill.  Sequence b appends C_b new
 * tokens, C_b = query_start[b+1] - query_start[b], after P_b cached ones;
 * context_lens[b] = P_b + C_b counts them all and the chunk's K/V must already
 * be in the cache (pkv_kv_append).  Query row t = query_start[b] + i attends
 * causally over the first P_b + i + 1 tokens:
 *
 *   out[t][h][:] = sum_{j <= P_b + i} softmax_j(scale * <q[t][h], K_j>) V_j
 *
 * with K_j / V_j found through block_tables as in paged decode (kv head h / G).
 * bf16 in and out; S = q K^T and O = P V run as tcgen05 MMAs with fp32
 * accumulation, P is rounded to bf16 for the second product (the softmax
 * denominator sums the fp32 weights, within 2^-9 relative of the rounded ones).
 *
 *   q, out        device, bf16 [T][num_q_heads][head_dim], T = query_start[num_seqs]
 *   query_start   device, int32 [num_seqs + 1], non-decreasing, query_start[0] = 0
 *   max_query_len host: at least every C_b (sizes the grid); at most 65535 CTAs
 *                 of 256 / G chunk tokens (G = num_q_heads / num_kv_heads), else
 *                 PKV_ERR_UNSUPPORTED
 * num_seqs at most 65535, else PKV_ERR_UNSUPPORTED.  No workspace.  num_seqs == 0 or max_query_len == 0 is a no-op.  Device-side:
 * C_b > max_query_len or C_b > context_lens[b] sets
 * PKV_DEVERR_CONTEXT_LEN_TOO_LONG (that sequence is skipped or cut); a bad
 * block id sets PKV_DEVERR_BLOCK_ID_OUT_OF_RANGE (block 0 is read instead).
 */
pkv_status pkv_paged_prefill_attention(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* context_lens, const int32_t* query_start,
                                       int32_t max_query_len, int32_t num_seqs, int32_t num_q_heads,
                                       int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks, int32_t block_size,
                                       float scale, void* out, pkv_stream_t stream);

/*
 * The same computation with each (tile pair, kv head, sequence) split over
 * num_splits CTAs, each taking a contiguous share of the key steps (keys 128 at
 * a time), and a merge pass that combines their fp32 partial states: for a row,
 * M = max m_s, out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s (the split-K
 * reduction of paged decode).  For calls whose CTAs do not fill the GPU (few
 * sequences, short chunks); a split with no key step only marks its rows empty.
 * The fp32 partial states are merged in another order than the unsplit call's
 * single accumulation, so results may differ from it by a bf16 step.
 *
 *   num_splits       host, 1..32; 1 is pkv_paged_prefill_attention (no workspace)
 *   workspace        device, 16-byte aligned, at least pkv_prefill_workspace_size
 *                    bytes; owned by the caller; the call writes the partial states
 *                    of the rows it covers and reads them back; not used after the
 *                    call's kernels finish (two launches on `stream`)
 * Errors as pkv_paged_prefill_attention, plus: num_splits out of range, a null or
 * short workspace (PKV_ERR_INVALID_ARGUMENT); num_seqs * num_splits above 65535
 * (PKV_ERR_UNSUPPORTED).  On a device-side timeout the outputs are undefined.
 */
pkv_status pkv_paged_prefill_attention_split(const void* q, const void* k_cache, const void* v_cache,
                                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                                             const int32_t* context_lens, const int32_t* query_start,
                                             int32_t max_query_len, int32_t num_seqs, int32_t num_q_heads,
                                             int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks,
                                             int32_t block_size, float scale, void* out, int32_t num_splits,
                                             void* workspace, size_t workspace_bytes, pkv_stream_t stream);

/*
 * A split count for pkv_paged_prefill_attention_split: the most splits that
 * keep the call's CTAs (num_seqs * num_kv_heads * ceil(max_query_len / (256 / G)))
 * within one CTA per SM of the current device, at most 32; 1 when the call already
 * fills the GPU.  A heuristic on host-known sizes only (the chunks and cached
 * lengths are on the device).  Queries the current device; writes *num_splits.
 */
pkv_status pkv_prefill_default_splits(int32_t num_seqs, int32_t max_query_len, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t* num_splits);

/*
 * Workspace bytes of pkv_paged_prefill_attention_split: num_splits * num_seqs *
 * R * num_q_heads * (head_dim + 2) * 4, R = max_query_len rounded up to the CTA's
 * 256 / G chunk tokens (0 for num_splits = 1).  Host only; writes *bytes.
 */
pkv_status pkv_prefill_workspace_size(int32_t num_seqs, int32_t max_query_len, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim, int32_t num_splits, size_t* bytes);

/*
 * Copy whole KV blocks inside the pool: the copy half of copy-on-write for
 * blocks shared between sequences.  The pages let requests share a prompt's
 * KV blocks ("v0版本介绍", section "为什么需要推理框架") and plan a prefix
 * cache ("从零实现一个 mini vLLM--开篇", section 4); a block shared by several
 * sequences must be copied before one of them appends into it.
 *
 * For every pair i: k_cache[dst_i][:][:][:] = k_cache[src_i][:][:][:] and the
 * same for v_cache (every kv head, all 16 slots), bit-exact.
 *
 *   src_dst     device, int64 [num_pairs][2] = (src, dst) block ids
 *   k_cache, v_cache  device, bf16 [num_blocks][num_kv_heads][16][head_dim]
 *
 * Destinations must be distinct and no destination may be a source of
 * another pair.  num_pairs == 0 is a no-op.  Device-side: a block id outside
 * [0, num_blocks) sets PKV_DEVERR_COPY_OUT_OF_RANGE and that pair is skipped.
 */
pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const int64_t* src_dst, int32_t num_pairs,
                           int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks, pkv_stream_t stream);

/*
 * Host block manager: the paged cache's allocator ("跟着 Claude Code，我用
 * Python 实现了一个轻量级的 vLLM", section "核心机制一：分页 KV Cache": fixed
 * 16-token blocks taken on demand and all returned when a sequence ends;
 * "从零实现一个 mini vLLM--开篇", section 5, phase 4: one block table per
 * request; "v0版本介绍", section "为什么需要推理框架": a new block is taken only
 * when the current one is full, and requests may share prompt blocks).
 *
 * Host memory only; every call on one manager is serialised by a lock inside
 * it.  Blocks carry a reference count: a fork shares all of the parent's
 * blocks, and appending into a shared, partly filled last block first moves
 * the sequence onto a fresh block (copy-on-write) and reports the (src, dst)
 * copy the caller must run with pkv_copy_blocks before the append.  The free
 * list is first-in first-out: blocks are taken from its front, and a
 * sequence's released blocks join its back in block-table order.  A call
 * that fails changes nothing.
 */
typedef struct pkv_block_manager pkv_block_manager;

/* Pool of num_blocks blocks.  initial_free_order (NULL = 0, 1, 2, ...) is a
   permutation of [0, num_blocks) giving the initial free list. */
pkv_status pkv_bm_create(int64_t num_blocks, const int64_t* initial_free_order, pkv_block_manager** out);
pkv_status pkv_bm_destroy(pkv_block_manager* bm);
/* Number of blocks on the free list. */
pkv_status pkv_bm_num_free(pkv_block_manager* bm, int64_t* num_free);
/* New sequence (an unused id >= 0) holding num_tokens tokens, ceil(num_tokens / 16)
   blocks.  slots (NULL or [num_tokens]) receives the slot of every position. */
pkv_status pkv_bm_add_sequence(pkv_block_manager* bm, int64_t seq_id, int64_t num_tokens, int64_t* slots);
/* Grow each listed sequence (ids distinct) by one token.  slots[i] receives
   its new token's slot.  Copy-on-write pairs go to copies[0 .. 2 * *num_copies)
   as (src, dst); there are at most num_seqs of them. */
pkv_status pkv_bm_append_slots(pkv_block_manager* bm, const int64_t* seq_ids, int32_t num_seqs, int64_t* slots,
                               int64_t* copies, int32_t* num_copies);
/* child_id (an unused id) shares every block of parent_id and has its length. */
pkv_status pkv_bm_fork(pkv_block_manager* bm, int64_t parent_id, int64_t child_id);
/* Release a sequence: each of its blocks loses one reference, and blocks left
   with none go back to the free list. */
pkv_status pkv_bm_free_sequence(pkv_block_manager* bm, int64_t seq_id);
/* Block tables and lengths of the listed sequences: tables is
   [num_seqs][width] int32 padded with -1; lengths is [num_seqs] int32. */
pkv_status pkv_bm_block_tables(pkv_block_manager* bm, const int64_t* seq_ids, int32_t num_seqs, int32_t width,
                               int32_t* tables, int32_t* lengths);
/* Reference count of one block (0 = free). */
pkv_status pkv_bm_ref_count(pkv_block_manager* bm, int64_t block, int32_t* count);

/*
 * Synchronises `stream`, then returns and clears the current device's sticky
 * error word (a mask of PKV_DEVERR_* bits; 0 = no device-side error since the
 * last clear).  The word is unsigned (uint32_t, not int32_t) because it is a
 * set of independent flags, each set by an atomic OR on the device.
 *
 * The word's device address is looked up once per device ordinal and kept for
 * the life of the process (as is the scratch address behind
 * pkv_paged_decode_attention_static); after a cudaDeviceReset, which destroys
 * the context those addresses belong to, this library must not be called
 * again on that device in the same process.
 */
pkv_status pkv_get_and_clear_device_error(uint32_t* bits, pkv_stream_t stream);

/*
 * Self-test of failure detection.  Every wait of the attention kernels on a
 * shared-memory barrier (a staged K/V copy landing) gives up after a time
 * limit, sets PKV_DEVERR_PIPELINE_TIMEOUT and leaves, so that a copy that never
 * lands ends in an error the host reads rather than in a hung GPU.  This call
 * launches one warp on `stream` that runs that same wait, with a limit of
 * limit_ns nanoseconds, on a barrier that nothing completes: the wait runs
 * out and the bit is set.  It faults nothing and the context stays usable.
 * limit_ns must lie in [1000, 1000000000] (1 us .. 1 s), else
 * PKV_ERR_INVALID_ARGUMENT before any launch.
 */
pkv_status pkv_selftest_wait_timeout(uint64_t limit_ns, pkv_stream_t stream);

/* Message of the last failed call on this host thread ("" if none).  Valid until the next call. */
const char* pkv_last_error_message(void);

/* Number of kernels this library has launched in this process (all devices). */
uint64_t pkv_kernel_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
