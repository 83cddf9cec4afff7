/*
 * pkv_oracle.c -- plain CPU reference for the paged KV-cache hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this library.  The product path
 * (the CUDA library and its Python binding) never calls it, links it or
 * falls back to it.  It shares no code, header, table or helper with the
 * CUDA path.
 *
 * Everything is computed in IEEE double from the exactly widened bf16 inputs,
 * in the order the definitions below state, with no blocking, fusion or
 * reordering.  Sources (web pages on a mini vLLM inference engine):
 *
 *  [P1] "跟着 Claude Code，我用 Python 实现了一个轻量级的 vLLM",
 *       section "核心机制一：分页 KV Cache": the KV cache is cut into
 *       fixed-size blocks of (for example) 16 tokens, allocated on demand.
 *  [P2] "从零实现一个 mini vLLM--开篇",
 *       section 2 "LLM 推理到底在慢什么": decode computes only the new
 *       token's K/V, appends it to the cache, and attends over all
 *       historical K/V;
 *       section 5 "这个系列会怎么展开" (phases 4 and 5): each request owns
 *       a block table; the sequence is logically contiguous, physically
 *       scattered over blocks, and attention finds the real K and V through
 *       the block table.
 *
 * Readings taken where the pages are silent (the same readings the CUDA
 * library documents in its header):
 *  - cache layout: k_cache and v_cache are each [num_blocks][num_kv_heads]
 *    [block_size][head_dim] bf16; slot s lives in block s / block_size at
 *    offset s % block_size;
 *  - a negative slot means "no slot" (padding) and is skipped;
 *  - q head h reads kv head h / (num_q_heads / num_kv_heads) (contiguous
 *    GQA groups);
 *  - context_lens[b] counts every cached token, including the one appended
 *    in this step; there is no mask; context_len 0 gives an all-zero output;
 *  - block-table entries past ceil(context_len / block_size) are never read.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Return codes (bit mask). */
#define ORACLE_OK 0
#define ORACLE_BAD_ARGUMENT 1
#define ORACLE_SLOT_OUT_OF_RANGE 2
#define ORACLE_DUPLICATE_SLOT 4
#define ORACLE_BLOCK_ID_OUT_OF_RANGE 8
#define ORACLE_CONTEXT_LEN_OUT_OF_RANGE 16

/* A bf16 value is the upper half of an IEEE binary32; widening is exact. */
static double bf16_to_double(uint16_t bits) {
    uint32_t word = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

static int cmp_i64(const void* a, const void* b) {
    int64_t x = *(const int64_t*)a, y = *(const int64_t*)b;
    return (x > y) - (x < y);
}

/*
 * Append [P2 section 2; P1 section 核心机制一]: for every token i whose slot
 * s = slot_mapping[i] is non-negative, copy the bits of k[i, h, :] into
 * k_cache[s / block_size, h, s % block_size, :] for every kv head h, and the
 * same for v.  An exact bit copy.  Slots past the pool are skipped and
 * flagged; duplicate non-negative slots are flagged (the operation is only
 * defined for distinct slots) and nothing is written then.
 */
int pkv_oracle_kv_append(const uint16_t* k, const uint16_t* v,
                         const int64_t* slot_mapping, int64_t num_tokens,
                         int32_t num_kv_heads, int32_t head_dim,
                         uint16_t* k_cache, uint16_t* v_cache,
                         int64_t num_blocks, int32_t block_size) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks < 0)
        return ORACLE_BAD_ARGUMENT;
    if (num_tokens == 0) return ORACLE_OK;

    /* Distinctness check on a sorted copy of the non-negative slots. */
    int64_t* sorted = (int64_t*)malloc(sizeof(int64_t) * (size_t)num_tokens);
    if (!sorted) return ORACLE_BAD_ARGUMENT;
    int64_t n_valid = 0;
    for (int64_t i = 0; i < num_tokens; ++i)
        if (slot_mapping[i] >= 0) sorted[n_valid++] = slot_mapping[i];
    qsort(sorted, (size_t)n_valid, sizeof(int64_t), cmp_i64);
    for (int64_t i = 1; i < n_valid; ++i) {
        if (sorted[i] == sorted[i - 1]) {
            free(sorted);
            return ORACLE_DUPLICATE_SLOT;
        }
    }
    free(sorted);

    int status = ORACLE_OK;
    const int64_t num_slots = num_blocks * (int64_t)block_size;
    for (int64_t i = 0; i < num_tokens; ++i) {
        const int64_t s = slot_mapping[i];
        if (s < 0) continue;
        if (s >= num_slots) {
            status |= ORACLE_SLOT_OUT_OF_RANGE;
            continue;
        }
        const int64_t block = s / block_size;
        const int64_t offset = s % block_size;
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            const int64_t src = (i * num_kv_heads + h) * (int64_t)head_dim;
            const int64_t dst = ((block * num_kv_heads + h) * block_size + offset) * (int64_t)head_dim;
            for (int32_t d = 0; d < head_dim; ++d) {
                k_cache[dst + d] = k[src + d];
                v_cache[dst + d] = v[src + d];
            }
        }
    }
    return status;
}

typedef struct {
    const uint16_t* q;
    const uint16_t* k_cache;
    const uint16_t* v_cache;
    const int32_t* block_tables;
    int32_t max_blocks_per_seq;
    const int32_t* context_lens;
    int32_t num_seqs;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int64_t num_blocks;
    int32_t block_size;
    double scale;
} problem_t;

/* GQA: q head h reads kv head h / (Hq / Hkv) (contiguous groups). */
static int32_t kv_head_of(const problem_t* P, int32_t h) {
    const int32_t group = P->num_q_heads / P->num_kv_heads;
    const int32_t kv = h / group;
    return kv;
}

/*
 * Attention of one query row over the first L cached tokens of sequence b,
 * kv head kv [P2 section 5, phases 4-5; P2 section 2]:
 *   K_t  = k_cache[block_tables[b, t / bs], kv, t % bs, :]   for t < L
 *   V_t  = v_cache[block_tables[b, t / bs], kv, t % bs, :]
 *   s_t  = scale * sum_d qrow[d] * K_t[d]
 *   p_t  = exp(s_t - max_t s_t) / sum_u exp(s_u - max_t s_t)
 *   out  = sum_t p_t * V_t
 * Writes head_dim doubles to out_row.  L == 0 writes zeros.
 */
static int attend_one(const problem_t* P, int32_t b, int32_t kv, const uint16_t* qrow, int32_t L, double* out_row) {
    const int32_t D = P->head_dim;
    for (int32_t d = 0; d < D; ++d) out_row[d] = 0.0;
    if (L == 0) return ORACLE_OK;

    double* scores = (double*)malloc(sizeof(double) * (size_t)L);
    const uint16_t** vrows = (const uint16_t**)malloc(sizeof(uint16_t*) * (size_t)L);
    if (!scores || !vrows) {
        free(scores);
        free((void*)vrows);
        return ORACLE_BAD_ARGUMENT;
    }

    /* Gather through the block table and form the scaled scores. */
    for (int32_t t = 0; t < L; ++t) {
        const int32_t logical_block = t / P->block_size;
        const int32_t offset = t % P->block_size;
        const int64_t phys = P->block_tables[(int64_t)b * P->max_blocks_per_seq + logical_block];
        if (phys < 0 || phys >= P->num_blocks) {
            free(scores);
            free((void*)vrows);
            for (int32_t d = 0; d < D; ++d) out_row[d] = 0.0;
            return ORACLE_BLOCK_ID_OUT_OF_RANGE;
        }
        const int64_t row = ((phys * P->num_kv_heads + kv) * P->block_size + offset) * (int64_t)D;
        const uint16_t* krow = P->k_cache + row;
        vrows[t] = P->v_cache + row;
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d) dot += bf16_to_double(qrow[d]) * bf16_to_double(krow[d]);
        scores[t] = P->scale * dot;
    }

    /* Softmax with the maximum subtracted. */
    double m = scores[0];
    for (int32_t t = 1; t < L; ++t)
        if (scores[t] > m) m = scores[t];
    double denom = 0.0;
    for (int32_t t = 0; t < L; ++t) {
        scores[t] = exp(scores[t] - m);
        denom += scores[t];
    }

    /* Probability-weighted sum of the value rows. */
    for (int32_t t = 0; t < L; ++t) {
        const double p = scores[t] / denom;
        for (int32_t d = 0; d < D; ++d) out_row[d] += p * bf16_to_double(vrows[t][d]);
    }
    free(scores);
    free((void*)vrows);
    return ORACLE_OK;
}

/* Decode: q row (b, h) attends over all context_lens[b] cached tokens. */
static int decode_one(const problem_t* P, int32_t b, int32_t h, double* out_row) {
    const int32_t D = P->head_dim;
    for (int32_t d = 0; d < D; ++d) out_row[d] = 0.0;
    if (b < 0 || b >= P->num_seqs || h < 0 || h >= P->num_q_heads) return ORACLE_BAD_ARGUMENT;
    const int32_t L = P->context_lens[b];
    if (L < 0 || (int64_t)L > (int64_t)P->max_blocks_per_seq * P->block_size)
        return ORACLE_CONTEXT_LEN_OUT_OF_RANGE;
    const uint16_t* qrow = P->q + ((int64_t)b * P->num_q_heads + h) * D;
    return attend_one(P, b, kv_head_of(P, h), qrow, L, out_row);
}

typedef struct {
    const problem_t* P;
    const int32_t* seq_idx;  /* NULL: item i is (i / Hq, i % Hq) */
    const int32_t* head_idx;
    int64_t begin, end;
    double* out;             /* item i writes out[i * head_dim ...] */
    int status;
} job_t;

static void* run_job(void* arg) {
    job_t* J = (job_t*)arg;
    const problem_t* P = J->P;
    for (int64_t i = J->begin; i < J->end; ++i) {
        int32_t b, h;
        if (J->seq_idx) {
            b = J->seq_idx[i];
            h = J->head_idx[i];
        } else {
            b = (int32_t)(i / P->num_q_heads);
            h = (int32_t)(i % P->num_q_heads);
        }
        J->status |= decode_one(P, b, h, J->out + i * P->head_dim);
    }
    return NULL;
}

static int run_items(const problem_t* P, const int32_t* seq_idx, const int32_t* head_idx,
                     int64_t n_items, double* out, int32_t num_threads) {
    if (P->num_kv_heads <= 0 || P->num_q_heads <= 0 || P->num_q_heads % P->num_kv_heads != 0 ||
        P->head_dim <= 0 || P->block_size <= 0 || P->num_seqs < 0 || P->max_blocks_per_seq < 0)
        return ORACLE_BAD_ARGUMENT;
    if (n_items <= 0) return ORACLE_OK;
    if (num_threads < 1) num_threads = 1;
    if (num_threads > 256) num_threads = 256;
    if ((int64_t)num_threads > n_items) num_threads = (int32_t)n_items;

    job_t jobs[256];
    pthread_t threads[256];
    int started[256];
    for (int32_t t = 0; t < num_threads; ++t) {
        jobs[t].P = P;
        jobs[t].seq_idx = seq_idx;
        jobs[t].head_idx = head_idx;
        jobs[t].begin = n_items * t / num_threads;
        jobs[t].end = n_items * (t + 1) / num_threads;
        jobs[t].out = out;
        jobs[t].status = 0;
        started[t] = 0;
    }
    for (int32_t t = 1; t < num_threads; ++t)
        started[t] = (pthread_create(&threads[t], NULL, run_job, &jobs[t]) == 0);
    run_job(&jobs[0]);
    int status = jobs[0].status;
    for (int32_t t = 1; t < num_threads; ++t) {
        if (started[t]) pthread_join(threads[t], NULL);
        else run_job(&jobs[t]);
        status |= jobs[t].status;
    }
    return status;
}

/*
 * Paged decode attention over every (sequence, q head): out is
 * [num_seqs][num_q_heads][head_dim] doubles.  num_threads only splits the
 * independent (b, h) items; each item is computed exactly as decode_one says.
 */
int pkv_oracle_paged_decode_attention(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks,
                                      int32_t block_size, double scale, double* out, int32_t num_threads) {
    problem_t P = {q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                   num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale};
    return run_items(&P, NULL, NULL, (int64_t)num_seqs * num_q_heads, out, num_threads);
}

/*
 * The same computation on a chosen sample of (sequence, q head) pairs: item i
 * is (seq_idx[i], head_idx[i]) and writes out[i][0..head_dim).
 */
int pkv_oracle_paged_decode_sampled(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                                    const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                                    int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks,
                                    int32_t block_size, double scale, const int32_t* seq_idx,
                                    const int32_t* head_idx, int64_t n_samples, double* out,
                                    int32_t num_threads) {
    problem_t P = {q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                   num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale};
    return run_items(&P, seq_idx, head_idx, n_samples, out, num_threads);
}

/*
 * Block copy for copy-on-write of shared blocks ("v0版本介绍", section
 * "为什么需要推理框架": requests may share a prompt's KV blocks; a shared block
 * is copied before one of its users appends into it): for every pair i,
 * k_cache[dst_i][:][:][:] = k_cache[src_i][:][:][:], the same for v_cache.
 * Pairs are applied in order.  Out-of-range ids are skipped and flagged.
 */
int pkv_oracle_copy_blocks(uint16_t* k_cache, uint16_t* v_cache, const int64_t* src_dst, int64_t num_pairs,
                           int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks, int32_t block_size) {
    if (num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks < 0)
        return ORACLE_BAD_ARGUMENT;
    const int64_t per_block = (int64_t)num_kv_heads * block_size * head_dim;
    int status = ORACLE_OK;
    for (int64_t i = 0; i < num_pairs; ++i) {
        const int64_t src = src_dst[2 * i], dst = src_dst[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            status |= ORACLE_BLOCK_ID_OUT_OF_RANGE;
            continue;
        }
        for (int64_t e = 0; e < per_block; ++e) {
            k_cache[dst * per_block + e] = k_cache[src * per_block + e];
            v_cache[dst * per_block + e] = v_cache[src * per_block + e];
        }
    }
    return status;
}

/*
 * fp32 -> bf16, round to nearest, ties to even (the definition: keep the top 16
 * bits of the binary32 after adding half of the dropped range, plus one more
 * when the kept part is odd).  NaN stays a quiet NaN.
 */
static uint16_t float_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
    const uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

int pkv_oracle_float_to_bf16(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = float_to_bf16_rne(in[i]);
    return ORACLE_OK;
}

/*
 * Rotary position embedding of the new token's q and k before they are used
 * ("跟着 Claude Code，我用 Python 实现了一个轻量级的 vLLM", section "核心机制五":
 * a full-attention layer is QKV projection + RoPE + KV cache + SDPA).  The
 * pages do not spell RoPE out; the reading is the rotate-half form of the
 * LLaMA / Qwen models they name: for i < D/2, with c = cos_sin[pos][i] and
 * s = cos_sin[pos][D/2 + i],
 *     x'[i]       = x[i] * c - x[i + D/2] * s
 *     x'[i + D/2] = x[i + D/2] * c + x[i] * s
 * Each product, difference and sum is one fp32 operation rounded to nearest
 * (this file is built without FMA contraction), and the result is rounded to
 * bf16, in place.  x is [n][heads][head_dim] bf16; positions is [n].
 */
int pkv_oracle_rope(uint16_t* x, int64_t n, int32_t heads, int32_t head_dim, const int64_t* positions,
                    const float* cos_sin, int64_t max_position) {
    if (n < 0 || heads <= 0 || head_dim <= 0 || (head_dim & 1)) return ORACLE_BAD_ARGUMENT;
    const int32_t half = head_dim / 2;
    for (int64_t r = 0; r < n; ++r) {
        const int64_t pos = positions[r];
        if (pos < 0 || pos >= max_position) return ORACLE_CONTEXT_LEN_OUT_OF_RANGE;
        const float* cs = cos_sin + pos * head_dim;
        for (int32_t h = 0; h < heads; ++h) {
            uint16_t* row = x + (r * heads + h) * (int64_t)head_dim;
            for (int32_t i = 0; i < half; ++i) {
                const float x1 = (float)bf16_to_double(row[i]);
                const float x2 = (float)bf16_to_double(row[i + half]);
                const float c = cs[i], s = cs[half + i];
                const float a = x1 * c;
                const float b = x2 * s;
                const float r1 = a - b;
                const float e = x2 * c;
                const float f = x1 * s;
                const float r2 = e + f;
                row[i] = float_to_bf16_rne(r1);
                row[i + half] = float_to_bf16_rne(r2);
            }
        }
    }
    return ORACLE_OK;
}

/*
 * Chunked prefill ("从零实现一个 mini vLLM--开篇", section 2: prefill runs the
 * whole prompt at once and stores every layer's K and V; section 5 lists
 * chunked prefill as a later topic).  Sequence b appends C_b new tokens,
 * C_b = query_start[b+1] - query_start[b], after P_b = context_lens[b] - C_b
 * cached ones (context_lens counts them all, the chunk's K/V already
 * appended).  Query row t = query_start[b] + i (i < C_b) sits at position
 * P_b + i and, causally, attends over the first P_b + i + 1 cached tokens.
 * q and out are [T][Hq][D] with T = query_start[num_seqs].
 */
typedef struct {
    const problem_t* P;
    const int32_t* query_start;
    int64_t begin, end;  /* items t * Hq + h */
    double* out;
    int status;
} prefill_job_t;

static int prefill_one(const problem_t* P, const int32_t* query_start, int64_t item, double* out_row) {
    const int32_t D = P->head_dim;
    const int64_t t = item / P->num_q_heads;
    const int32_t h = (int32_t)(item % P->num_q_heads);
    int32_t b = 0;
    while (b < P->num_seqs && (int64_t)query_start[b + 1] <= t) ++b;
    for (int32_t d = 0; d < D; ++d) out_row[d] = 0.0;
    if (b >= P->num_seqs) return ORACLE_BAD_ARGUMENT;
    const int32_t C = query_start[b + 1] - query_start[b];
    const int32_t Lb = P->context_lens[b];
    const int32_t i = (int32_t)(t - query_start[b]);
    if (C < 0 || Lb < C || (int64_t)Lb > (int64_t)P->max_blocks_per_seq * P->block_size)
        return ORACLE_CONTEXT_LEN_OUT_OF_RANGE;
    const int32_t prefix = Lb - C;
    const uint16_t* qrow = P->q + (t * P->num_q_heads + h) * D;
    return attend_one(P, b, kv_head_of(P, h), qrow, prefix + i + 1, out_row);
}

static void* run_prefill_job(void* arg) {
    prefill_job_t* J = (prefill_job_t*)arg;
    for (int64_t it = J->begin; it < J->end; ++it)
        J->status |= prefill_one(J->P, J->query_start, it, J->out + it * J->P->head_dim);
    return NULL;
}

int pkv_oracle_paged_prefill_attention(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* context_lens, const int32_t* query_start, int32_t num_seqs,
                                       int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                       int64_t num_blocks, int32_t block_size, double scale, double* out,
                                       int32_t num_threads) {
    problem_t P = {q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                   num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale};
    if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0 || num_seqs < 0)
        return ORACLE_BAD_ARGUMENT;
    for (int32_t b = 0; b < num_seqs; ++b)
        if (query_start[b + 1] < query_start[b]) return ORACLE_BAD_ARGUMENT;
    const int64_t items = (int64_t)query_start[num_seqs] * num_q_heads;
    if (items <= 0) return ORACLE_OK;
    if (num_threads < 1) num_threads = 1;
    if (num_threads > 256) num_threads = 256;
    if ((int64_t)num_threads > items) num_threads = (int32_t)items;
    prefill_job_t jobs[256];
    pthread_t threads[256];
    int started[256];
    for (int32_t k = 0; k < num_threads; ++k) {
        jobs[k].P = &P;
        jobs[k].query_start = query_start;
        jobs[k].begin = items * k / num_threads;
        jobs[k].end = items * (k + 1) / num_threads;
        jobs[k].out = out;
        jobs[k].status = 0;
        started[k] = 0;
    }
    for (int32_t k = 1; k < num_threads; ++k)
        started[k] = (pthread_create(&threads[k], NULL, run_prefill_job, &jobs[k]) == 0);
    run_prefill_job(&jobs[0]);
    int status = jobs[0].status;
    for (int32_t k = 1; k < num_threads; ++k) {
        if (started[k]) pthread_join(threads[k], NULL);
        else run_prefill_job(&jobs[k]);
        status |= jobs[k].status;
    }
    return status;
}
