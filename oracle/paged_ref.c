/*
 * paged_ref.c -- fp64 CPU oracle for paged decode attention, the KV cache write
 * and the copy-on-write block copy.
 *
 * TEST INFRASTRUCTURE ONLY. This file is loaded by the tests, by the package's
 * smoke check and by the CPU-baseline leg of the benchmark, and by nothing else.
 * It shares no header, helper or table with the CUDA library and never calls it.
 *
 * What it restates (sources are the four pages on PagedAttention):
 *  - "PagedAttention et RadixAttention : parlons de KV Cache" (aitalk.it),
 *    section "PagedAttention : la memoire comme un systeme d'exploitation":
 *    the cache of a sequence is cut into fixed logical blocks of 16 or 32
 *    tokens (step one); a per-sequence table maps each logical block to the
 *    physical block that holds it, and attention gathers the blocks through
 *    that table so that the model sees one continuous sequence (step two);
 *    blocks are shared between requests and copied only when one of them
 *    diverges (step four); and paging leaves the model's outputs unchanged.
 *  - "PagedAttention" (robocikowo.com), section "Jak dziala": physical blocks
 *    of typically 16 tokens per block per layer in HBM, a block table per
 *    sequence, an attention kernel that reads the blocks through that table,
 *    and a write into a shared block that triggers a copy.
 *
 * Because paging does not change what attention computes, the oracle is the
 * textbook definition: resolve the block table into a contiguous K and V for
 * the sequence, then out = softmax(scale * q K^T) V, all in fp64 with the
 * softmax taken as exp(s - max s) / sum.  Cache elements are fp32 or bf16
 * (raw bits) and are widened exactly to fp64; q is passed already in fp64.
 *
 * Layouts (row-major, chosen here because the pages fix none):
 *   cache          [num_blocks][num_kv_heads][block_size][head_dim]
 *   q, out         [num_seqs][num_q_heads][head_dim]
 *   block_tables   [num_seqs][max_blocks_per_seq]  int32
 *   context_lens   [num_seqs]                      int32
 * Query head h reads KV head h / (num_q_heads / num_kv_heads).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG -1
#define ORACLE_ERR_INDEX -4
#define ORACLE_ERR_NOMEM -9

#define ORACLE_F32 0
#define ORACLE_BF16 1

/* One cache element, widened exactly to fp64.  A bf16 value is the top half
 * of an IEEE fp32 bit pattern, so shifting its 16 bits up gives that fp32. */
static double widen(const void *base, int dtype, int64_t idx)
{
    if (dtype == ORACLE_F32)
        return (double)((const float *)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Textbook attention of one query row over n contiguous keys/values, fp64.
 * out[d] = sum_t p_t V[t][d] with p = softmax(scale * q.K[t]); n == 0 gives
 * an all-zero row (no token to attend to). */
static void attend_contiguous(double *out, const double *q, const double *K,
                              const double *V, int n, int hd, double scale,
                              double *s /* n scratch */)
{
    for (int d = 0; d < hd; ++d)
        out[d] = 0.0;
    if (n <= 0)
        return;
    double smax = -INFINITY;
    for (int t = 0; t < n; ++t) {
        double acc = 0.0;
        for (int d = 0; d < hd; ++d)
            acc += q[d] * K[(int64_t)t * hd + d];
        s[t] = scale * acc;
        if (s[t] > smax)
            smax = s[t];
    }
    double denom = 0.0;
    for (int t = 0; t < n; ++t) {
        s[t] = exp(s[t] - smax);
        denom += s[t];
    }
    for (int t = 0; t < n; ++t) {
        double p = s[t] / denom;
        for (int d = 0; d < hd; ++d)
            out[d] += p * V[(int64_t)t * hd + d];
    }
}

/* Resolve the block table of one sequence into contiguous K and V rows of one
 * KV head: token t lives in physical block table[t / bs] at slot t % bs. */
static int gather_sequence(double *K, double *V, const void *k_cache,
                           const void *v_cache, int dtype, const int32_t *table,
                           int n, int kv_head, int num_kv_heads, int hd, int bs,
                           int num_blocks)
{
    for (int t = 0; t < n; ++t) {
        int32_t phys = table[t / bs];
        if (phys < 0 || phys >= num_blocks)
            return ORACLE_ERR_INDEX;
        int64_t row = (((int64_t)phys * num_kv_heads + kv_head) * bs + (t % bs)) * hd;
        for (int d = 0; d < hd; ++d) {
            K[(int64_t)t * hd + d] = widen(k_cache, dtype, row + d);
            V[(int64_t)t * hd + d] = widen(v_cache, dtype, row + d);
        }
    }
    return ORACLE_OK;
}

typedef struct {
    double *out;
    const double *q;
    const void *k_cache, *v_cache;
    int dtype;
    const int32_t *block_tables;
    int max_blocks_per_seq;
    const int32_t *context_lens;
    int num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks;
    double scale;
    const int32_t *pairs; /* [num_pairs][2] = (seq, q head); NULL = all */
    int64_t num_pairs;
    int64_t first, last; /* this worker's slice of the pair list */
    int status;
} job_t;

static void *run_slice(void *arg)
{
    job_t *j = (job_t *)arg;
    int hd = j->head_dim, group = j->num_q_heads / j->num_kv_heads;
    int max_n = j->max_blocks_per_seq * j->block_size;
    double *K = (double *)malloc(sizeof(double) * (size_t)max_n * hd + 8);
    double *V = (double *)malloc(sizeof(double) * (size_t)max_n * hd + 8);
    double *s = (double *)malloc(sizeof(double) * (size_t)max_n + 8);
    if (!K || !V || !s) {
        j->status = ORACLE_ERR_NOMEM;
        free(K), free(V), free(s);
        return NULL;
    }
    int cached_seq = -1, cached_kv = -1;
    for (int64_t w = j->first; w < j->last; ++w) {
        int i, h;
        if (j->pairs) {
            i = j->pairs[2 * w];
            h = j->pairs[2 * w + 1];
        } else {
            i = (int)(w / j->num_q_heads);
            h = (int)(w % j->num_q_heads);
        }
        if (i < 0 || i >= j->num_seqs || h < 0 || h >= j->num_q_heads) {
            j->status = ORACLE_ERR_ARG;
            break;
        }
        int n = j->context_lens[i];
        if (n < 0 || n > max_n) {
            j->status = ORACLE_ERR_INDEX;
            break;
        }
        int kv = h / group;
        if (i != cached_seq || kv != cached_kv) {
            int rc = gather_sequence(K, V, j->k_cache, j->v_cache, j->dtype,
                                     j->block_tables + (int64_t)i * j->max_blocks_per_seq,
                                     n, kv, j->num_kv_heads, hd, j->block_size, j->num_blocks);
            if (rc != ORACLE_OK) {
                j->status = rc;
                break;
            }
            cached_seq = i, cached_kv = kv;
        }
        int64_t row = ((int64_t)i * j->num_q_heads + h) * hd;
        attend_contiguous(j->out + row, j->q + row, K, V, n, hd, j->scale, s);
    }
    free(K), free(V), free(s);
    return NULL;
}

/* Paged decode attention for every (sequence, query head), or for the listed
 * (sequence, query head) pairs only.  Rows not listed are left untouched.
 * Returns 0, ORACLE_ERR_ARG, ORACLE_ERR_INDEX (block id or length out of
 * range) or ORACLE_ERR_NOMEM. */
int oracle_paged_decode(double *out, const double *q, const void *k_cache,
                        const void *v_cache, int dtype, const int32_t *block_tables,
                        int max_blocks_per_seq, const int32_t *context_lens,
                        int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                        int block_size, int num_blocks, double scale,
                        const int32_t *pairs, int64_t num_pairs, int num_threads)
{
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return ORACLE_ERR_ARG;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16)
        return ORACLE_ERR_ARG;
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || num_blocks < 0 || max_blocks_per_seq < 0)
        return ORACLE_ERR_ARG;
    if (num_q_heads % num_kv_heads != 0)
        return ORACLE_ERR_ARG;
    int64_t total = pairs ? num_pairs : (int64_t)num_seqs * num_q_heads;
    if (total <= 0)
        return ORACLE_OK;
    if (num_threads < 1)
        num_threads = 1;
    if (num_threads > 256)
        num_threads = 256;
    if (num_threads > total)
        num_threads = (int)total;

    job_t jobs[256];
    pthread_t tids[256];
    for (int w = 0; w < num_threads; ++w) {
        job_t *j = &jobs[w];
        j->out = out, j->q = q, j->k_cache = k_cache, j->v_cache = v_cache;
        j->dtype = dtype, j->block_tables = block_tables;
        j->max_blocks_per_seq = max_blocks_per_seq, j->context_lens = context_lens;
        j->num_seqs = num_seqs, j->num_q_heads = num_q_heads;
        j->num_kv_heads = num_kv_heads, j->head_dim = head_dim;
        j->block_size = block_size, j->num_blocks = num_blocks, j->scale = scale;
        j->pairs = pairs, j->num_pairs = num_pairs;
        j->first = total * w / num_threads;
        j->last = total * (w + 1) / num_threads;
        j->status = ORACLE_OK;
    }
    if (num_threads == 1) {
        run_slice(&jobs[0]);
    } else {
        int started = 0;
        for (; started < num_threads; ++started)
            if (pthread_create(&tids[started], NULL, run_slice, &jobs[started]) != 0)
                break;
        for (int w = 0; w < started; ++w)
            pthread_join(tids[w], NULL);
        for (int w = started; w < num_threads; ++w)
            run_slice(&jobs[w]);
    }
    for (int w = 0; w < num_threads; ++w)
        if (jobs[w].status != ORACLE_OK)
            return jobs[w].status;
    return ORACLE_OK;
}

/* Cache write: token t's K and V rows (all KV heads) go to physical slot
 * slot_mapping[t] = block * block_size + offset; a negative slot is padding
 * and is skipped.  Plain byte copies of elem_bytes-wide elements.
 * ("PagedAttention", robocikowo.com, "Jak dziala": blocks grow on demand as
 * the sequence grows; aitalk.it page, third step: block-by-block growth.) */
int oracle_reshape_and_cache(const void *k, const void *v, void *k_cache, void *v_cache,
                             const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                             int head_dim, int block_size, int num_blocks, int elem_bytes)
{
    if (!k || !v || !k_cache || !v_cache || !slot_mapping || num_tokens < 0 ||
        num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks < 0 ||
        (elem_bytes != 2 && elem_bytes != 4))
        return ORACLE_ERR_ARG;
    int64_t num_slots = (int64_t)num_blocks * block_size;
    for (int t = 0; t < num_tokens; ++t)
        if (slot_mapping[t] >= num_slots)
            return ORACLE_ERR_INDEX;
    size_t row_bytes = (size_t)head_dim * elem_bytes;
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        int64_t blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            size_t src = ((size_t)t * num_kv_heads + h) * row_bytes;
            size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + off) * row_bytes;
            memcpy((char *)k_cache + dst, (const char *)k + src, row_bytes);
            memcpy((char *)v_cache + dst, (const char *)v + src, row_bytes);
        }
    }
    return ORACLE_OK;
}

/* Copy-on-write block copy: for each (src, dst) pair, the whole dst block
 * (every KV head and slot) of both caches becomes a copy of the src block.
 * Pairs are applied in list order.  ("PagedAttention", robocikowo.com,
 * "Komponenty": reference counting with lazy duplication on modification.) */
int oracle_copy_blocks(void *k_cache, void *v_cache, const int64_t *src_dst_pairs,
                       int num_pairs, int num_kv_heads, int head_dim, int block_size,
                       int num_blocks, int elem_bytes)
{
    if (!k_cache || !v_cache || (num_pairs > 0 && !src_dst_pairs) || num_pairs < 0 ||
        num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks < 0 ||
        (elem_bytes != 2 && elem_bytes != 4))
        return ORACLE_ERR_ARG;
    for (int p = 0; p < num_pairs; ++p) {
        int64_t s = src_dst_pairs[2 * p], d = src_dst_pairs[2 * p + 1];
        if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks)
            return ORACLE_ERR_INDEX;
    }
    size_t block_bytes = (size_t)num_kv_heads * block_size * head_dim * elem_bytes;
    for (int p = 0; p < num_pairs; ++p) {
        int64_t s = src_dst_pairs[2 * p], d = src_dst_pairs[2 * p + 1];
        memmove((char *)k_cache + d * block_bytes, (const char *)k_cache + s * block_bytes, block_bytes);
        memmove((char *)v_cache + d * block_bytes, (const char *)v_cache + s * block_bytes, block_bytes);
    }
    return ORACLE_OK;
}

/* Block copy between two pools of the same geometry (swap to or from host
 * memory): block dst of (dst_k, dst_v) becomes a copy of block src of
 * (src_k, src_v), pairs applied in list order.  ("PagedAttention" concept
 * sheet, analyticslegends.ai, "Points cles": cold pages go to CPU RAM and are
 * read back on demand.) */
int oracle_swap_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                       const int64_t *src_dst_pairs, int num_pairs, int src_num_blocks, int dst_num_blocks,
                       int num_kv_heads, int head_dim, int block_size, int elem_bytes)
{
    if (!src_k || !src_v || !dst_k || !dst_v || (num_pairs > 0 && !src_dst_pairs) || num_pairs < 0 ||
        num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || (elem_bytes != 2 && elem_bytes != 4))
        return ORACLE_ERR_ARG;
    for (int p = 0; p < num_pairs; ++p) {
        int64_t s = src_dst_pairs[2 * p], d = src_dst_pairs[2 * p + 1];
        if (s < 0 || s >= src_num_blocks || d < 0 || d >= dst_num_blocks)
            return ORACLE_ERR_INDEX;
    }
    size_t block_bytes = (size_t)num_kv_heads * block_size * head_dim * elem_bytes;
    for (int p = 0; p < num_pairs; ++p) {
        int64_t s = src_dst_pairs[2 * p], d = src_dst_pairs[2 * p + 1];
        memcpy((char *)dst_k + d * block_bytes, (const char *)src_k + s * block_bytes, block_bytes);
        memcpy((char *)dst_v + d * block_bytes, (const char *)src_v + s * block_bytes, block_bytes);
    }
    return ORACLE_OK;
}
