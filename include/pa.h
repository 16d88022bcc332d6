/*
 * pa.h -- C ABI of the GB300 (sm_103a) paged decode-attention library.
 *
 * The operations follow four pages on PagedAttention:
 *  [P1] "PagedAttention", ayinedjimi-consultants.fr glossary, "Definition";
 *  [P2] "PagedAttention — Gestion memoire pour LLM a long contexte",
 *       analyticslegends.ai, "Pourquoi c'est important", "Points cles",
 *       "Termes employes sur cette page";
 *  [P3] "PagedAttention", robocikowo.com, "Jak dziala", "Komponenty",
 *       "Pulapki implementacyjne", "Zlozonosc obliczeniowa";
 *  [P4] "PagedAttention et RadixAttention : parlons de KV Cache", aitalk.it,
 *       "PagedAttention : la memoire comme un systeme d'exploitation".
 *
 * Conventions for every call:
 *  - Pointers named *_cache, q, out, k, v, block_tables, context_lens,
 *    slot_mapping, src_dst_pairs, workspace and dev_status are DEVICE pointers
 *    owned by the caller.  The library never allocates device memory.
 *  - `stream` is a cudaStream_t passed as void*; NULL means the legacy default
 *    stream.  Device calls only enqueue work and return before it runs.  They
 *    launch on the calling thread's current CUDA device: every device pointer
 *    (and the stream) must belong to it.
 *  - Every call returns PA_OK (0) or a negative PA_ERR_* code; nothing is
 *    thrown across the ABI.  pa_last_error_string() describes the last failure
 *    of the calling thread.
 *  - Argument errors are reported before anything is enqueued.  Errors that
 *    depend on device data (a block id outside the pool, a context length
 *    beyond the table, a slot outside the pool, a bad copy pair) cannot be
 *    seen on the host: kernels skip the offending access, OR a PA_STATUS_* bit
 *    into *dev_status (when not NULL) and carry on, so no input can make a
 *    kernel read or write outside the buffers described here.
 *
 * Layouts (row-major, element type = `dtype` unless stated):
 *   k_cache, v_cache  [num_blocks][num_kv_heads][block_size][head_dim]
 *   q, out            [num_seqs][num_q_heads][head_dim]
 *   block_tables      [num_seqs][max_blocks_per_seq] int32 (physical ids)
 *   context_lens      [num_seqs] int32
 *   k, v (new tokens) [num_tokens][num_kv_heads][head_dim]
 *   slot_mapping      [num_tokens] int64, slot = block * block_size + offset
 *   src_dst_pairs     [num_pairs][2] int64 (src block, dst block)
 * Query head h attends with KV head h / (num_q_heads / num_kv_heads).
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ---------------------------------------------------- */
#define PA_OK 0
#define PA_ERR_INVALID_ARG -1 /* null pointer, bad size, inconsistent shape */
#define PA_ERR_UNSUPPORTED -2 /* valid request the library has no kernel for */
#define PA_ERR_CUDA -3        /* a CUDA runtime/driver call failed */
#define PA_ERR_BAD_INDEX -4   /* host-visible id out of range */
#define PA_ERR_NO_BLOCKS -5   /* block manager: free pool exhausted */
#define PA_ERR_REFCOUNT -6    /* block manager: unknown sequence or id misuse */
#define PA_ERR_WORKSPACE -7   /* workspace missing or too small */

/* ---- element types ---------------------------------------------------- */
#define PA_F32 0  /* IEEE fp32 */
#define PA_BF16 1 /* bfloat16 (fp32 accumulation inside the kernels) */

/* ---- device status bits (OR-ed into *dev_status by the kernels) -------- */
#define PA_STATUS_BAD_BLOCK_ID 1    /* block table entry outside [0, num_blocks) */
#define PA_STATUS_BAD_CONTEXT_LEN 2 /* context_lens[i] < 0 or beyond the table or max_context_len */
#define PA_STATUS_BAD_SLOT 4        /* slot_mapping entry >= num_blocks * block_size, or (fused
                                       write) not the slot of the sequence's last position */
#define PA_STATUS_BAD_PAIR 8        /* copy pair out of range, or its dst is another pair's src/dst */
#define PA_STATUS_WAIT_TIMEOUT 16   /* a bounded wait for staged data gave up */

/* ---- decode attention --------------------------------------------------
 * [P3] "Jak dziala" / "Komponenty": the attention kernel reads the K/V cache
 * of each sequence through its block table of fixed-size physical blocks;
 * [P4] step two: the table makes the scattered blocks look like one
 * continuous sequence, and paging leaves attention's result unchanged.
 *
 * For every sequence i and query head h, with n = context_lens[i] and KV head
 * kv = h / (num_q_heads / num_kv_heads):
 *   out[i][h] = sum_t softmax_t(scale * q[i][h] . K_i[t]) V_i[t],  t < n,
 *   K_i[t] = k_cache[block_tables[i][t / block_size]][kv][t % block_size].
 * n == 0 gives a zero row.  Cache slots at or past n in the last block are
 * never used, whatever they hold (NaN included).
 *
 * Long contexts are cut into partitions of `partition_size` tokens that are
 * processed independently and merged by a second pass (split-K), which needs
 * `workspace`.  With a workspace, the bf16 pass also hands out its work items
 * through a counter held there, so CTAs that finish early take more.
 * Arithmetic: fp32 accumulation; for PA_BF16 the products q.K and p.V run on
 * bf16 tensor-core MMAs, p entering as the sum of two bf16 parts (about 16
 * significant bits); for PA_F32 on fp32 FMAs.  Results are deterministic for
 * a given input and partition size (which CTA runs an item does not change
 * its arithmetic).
 */
typedef struct pa_decode_args {
    int num_seqs;           /* S >= 0 */
    int max_blocks_per_seq; /* row stride (in entries) of block_tables, >= 1 */
    int num_blocks;         /* physical blocks in each cache tensor, >= 1 */
    int dtype;              /* PA_F32 or PA_BF16: q, k_cache, v_cache and out */
    int partition_size;     /* tokens per split-K partition, multiple of 16 in
                               [16, 4096]; 0 picks 512 */
    int max_context_len;    /* host upper bound of context_lens[i]; longer
                               entries are clamped and flagged */
    void *workspace;        /* device scratch, 256-byte aligned is best: the
                               partition pass's work counter in its first 8
                               bytes, then the split-K partials; may be NULL
                               when max_context_len <= partition_size.  No
                               part needs to start at zero (see
                               skip_counter_reset).  One workspace serves one
                               call at a time: two calls that may run at the
                               same time on the GPU (different streams with no
                               ordering between them) must not share it, since
                               they would race on its work counter and
                               partials.  Calls ordered on one stream may
                               share it. */
    size_t workspace_bytes; /* >= pa_decode_workspace_size(...) */
    int32_t *dev_status;    /* optional device word for PA_STATUS_* bits */
    void *stream;           /* cudaStream_t */
    int phase;              /* PA_PHASE_ALL (0): both passes.  PA_PHASE_PARTITIONS
                               (1): only the per-partition pass (final rows of
                               single-partition sequences, partials of the
                               others).  PA_PHASE_REDUCE (2): only the merge of
                               the partials; it must follow phase 1 on the same
                               stream with identical arguments.  Splitting lets a
                               caller time or overlap the two passes. */
    /* Optional fused cache write (all three NULL to disable).  Sequence i's new
     * token is its last one, position context_lens[i] - 1: the call writes
     * k_new[i] / v_new[i] ([num_seqs][num_kv_heads][head_dim], dtype) into
     * k_cache / v_cache at slot_mapping[i] and attends with those values, the
     * same result as pa_reshape_and_cache followed by pa_decode, in one launch
     * fewer.  slot_mapping[i] < 0 skips sequence i's write.  A slot that is not
     * the slot of position context_lens[i] - 1 is not written and sets
     * PA_STATUS_BAD_SLOT.  When enabled, k_cache and v_cache are written.
     * (Pages: [P3] "Jak dziala", [P4] step three.) */
    const void *k_new;
    const void *v_new;
    const int64_t *slot_mapping;
    int simt;               /* PA_BF16 only: nonzero computes q.K and p.V with
                               plain fp32 FMAs (p kept in fp32, 8 query heads
                               per work item) instead of tensor-core MMAs;
                               0, the default, uses the MMAs.  Same results
                               within the tolerance; for comparison and for
                               callers who want fp32 products throughout. */
    int skip_counter_reset; /* The bf16 pass hands out work items through a
                               counter at the start of the workspace.  Each
                               call leaves that counter zero when it completes,
                               and by default also zeroes it first with a
                               cudaMemsetAsync on `stream` (8 bytes).  Nonzero
                               skips that memset (one operation, a few
                               microseconds, fewer per call): valid once the
                               counter is zero, i.e. after any completed call
                               on this workspace, or when the caller zeroed its
                               first 8 bytes. */
} pa_decode_args;

#define PA_PHASE_ALL 0
#define PA_PHASE_PARTITIONS 1
#define PA_PHASE_REDUCE 2

/* Supported: head_dim in {64, 128}; block_size in {16, 32}; num_q_heads a
 * multiple of num_kv_heads.  Returns PA_ERR_UNSUPPORTED otherwise. */
int pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
              const int32_t *block_tables, const int32_t *context_lens,
              int num_q_heads, int num_kv_heads, int head_dim, int block_size,
              float scale, const pa_decode_args *args);

/* Bytes of workspace pa_decode needs for these sizes (0 when no sequence can
 * span more than one partition).  partition_size 0 means the default.  A
 * helper of this library's split-K design: the pages describe no kernel-level
 * split of long contexts, so this call has no counterpart there. */
size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int head_dim,
                                int max_context_len, int partition_size);

/* ---- decode attention without a caller workspace ----------------------
 * The paper has no counterpart to this call; it is a convenience of this
 * library.
 *
 * For callers that cannot allocate device memory -- a plugin or framework
 * that owns every allocation and passes the library only its inputs and
 * outputs, or a hot path where a cudaMalloc, which may synchronise the
 * device, is not allowed.  Same computation, arguments and results as
 * pa_decode; args->workspace and args->workspace_bytes are ignored.  The
 * split-K scratch is a fixed array of PA_NOALLOC_WORKSPACE_BYTES (64 MiB)
 * inside the library, which every GPU that loads the library keeps until the
 * process exits.  The call allocates and frees nothing.
 *  - Sizes whose pa_decode_workspace_size() exceeds PA_NOALLOC_WORKSPACE_BYTES
 *    are rejected with PA_ERR_WORKSPACE before anything is enqueued.
 *  - The first call on a device that needs the scratch looks up its device
 *    address (cudaGetSymbolAddress) with that device current; make that first
 *    call before any stream capture on the device.  The address is kept for
 *    the life of the process: after cudaDeviceReset (or anything else that
 *    destroys the device's primary context) it is stale, and this call must
 *    not be used on that device again.
 *  - Arguments are checked as pa_decode checks them, before the scratch is
 *    sized; a bad partition_size, block_size or head_dim gives the same code
 *    as there.
 *  - Every call on a device shares the one array, which keeps the last call's
 *    contents; no part of it needs to start at zero (each call writes every
 *    partial it reads, and the work counter is reset before each pass unless
 *    skip_counter_reset is set; the array starts at zero and each completed
 *    call leaves the counter zero, so setting it is valid here).
 *  - Calls that overlap on the GPU -- on different streams without ordering
 *    between them -- race on the array. */
#define PA_NOALLOC_WORKSPACE_BYTES (64u * 1024u * 1024u)

int pa_decode_noalloc(void *out, const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_tables, const int32_t *context_lens,
                      int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                      float scale, const pa_decode_args *args);

/* ---- cache write ------------------------------------------------------
 * [P3] "Jak dziala" and [P4] step three: blocks are filled as the sequence
 * grows.  For each token t with slot s = slot_mapping[t] >= 0:
 *   k_cache[s / block_size][h][s % block_size][:] = k[t][h][:]  (all h), same
 *   for v.  Negative slots are padding and are skipped.  Bit-exact copy.
 * Slots must be distinct; two tokens naming one slot race. */
int pa_reshape_and_cache(const void *k, const void *v, void *k_cache, void *v_cache,
                         const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int num_blocks, int dtype,
                         int32_t *dev_status, void *stream);

/* ---- block copy (copy-on-write) ----------------------------------------
 * [P3] "Komponenty": shared prefix blocks carry reference counts and are
 * duplicated only when one sharer modifies them; [P4] step four.
 * For each pair p: block dst_p of both caches (every KV head and slot)
 * becomes a bit-exact copy of block src_p.  A dst that appears twice, or that
 * is also another pair's src, is rejected on the device: that pair is not
 * copied and PA_STATUS_BAD_PAIR is set.  src == dst is a no-op. */
int pa_copy_blocks(void *k_cache, void *v_cache, const int64_t *src_dst_pairs, int num_pairs,
                   int num_kv_heads, int head_dim, int block_size, int num_blocks, int dtype,
                   int32_t *dev_status, void *stream);

/* ---- block swap between two pools (device cache <-> host memory) --------
 * [P2] "Points cles" / "Termes employes sur cette page" (page eviction): when
 * GPU memory runs out, cold pages are written to CPU RAM and read back when
 * needed.  For each pair p, block dst_p of (dst_k, dst_v) becomes a bit-exact
 * copy of block src_p of (src_k, src_v): every KV head and slot.  The two
 * pools share the block geometry (num_kv_heads, block_size, head_dim, dtype)
 * and must be different allocations; each may be device memory or pinned host
 * memory the device can address (cudaHostAlloc / cudaHostRegister; checked
 * with cudaPointerGetAttributes, anything else is PA_ERR_INVALID_ARG).
 * src_dst_pairs must be device-accessible as well.  A pair out of range, or a
 * dst named twice, is skipped and sets PA_STATUS_BAD_PAIR. */
int pa_swap_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                   const int64_t *src_dst_pairs, int num_pairs, int src_num_blocks, int dst_num_blocks,
                   int num_kv_heads, int head_dim, int block_size, int dtype, int32_t *dev_status,
                   void *stream);

/* ---- host block manager -----------------------------------------------
 * [P3] "Komponenty": a block manager hands out and takes back physical
 * blocks from a free pool and keeps per-block reference counts for shared
 * prefixes; [P2] "Pourquoi c'est important": blocks are allocated on demand
 * and released one by one when a request ends; [P1] "Definition": freed
 * blocks are reused at once, and parallel samples share the prompt's blocks
 * until they diverge.
 *
 * Host memory only; not thread-safe (one manager per thread, or external
 * locking).  Allocation order: block 0 first, then 1, 2, ...; a freed block
 * is the next handed out (a LIFO pool); a sequence releases its blocks from
 * the last logical block to the first.  Failed calls leave the state as it
 * was.  Sequence ids are any non-negative int. */
typedef struct pa_bm pa_bm;

pa_bm *pa_bm_create(int num_blocks, int block_size); /* NULL on bad sizes */
void pa_bm_destroy(pa_bm *bm);

/* New sequence holding num_tokens tokens in ceil(num_tokens / block_size)
 * fresh blocks.  PA_ERR_NO_BLOCKS if the pool is short. */
int pa_bm_add_seq(pa_bm *bm, int seq_id, int num_tokens);

/* child shares every block of parent (refcount + 1 each). */
int pa_bm_fork(pa_bm *bm, int parent_id, int child_id);

/* Reserve the slot for the sequence's next token.  If the last block is full
 * a fresh block is appended.  If it is partial and shared (refcount > 1) it
 * is replaced by a fresh block, its refcount drops by one, and
 * (*cow_src, *cow_dst) name the copy the caller must run before writing
 * (pa_copy_blocks); otherwise both are -1.  *slot = block * block_size +
 * offset. */
int pa_bm_append_slot(pa_bm *bm, int seq_id, int64_t *slot, int32_t *cow_src, int32_t *cow_dst);

/* Drop the sequence; each of its blocks loses one reference and returns to
 * the pool at zero. */
int pa_bm_free_seq(pa_bm *bm, int seq_id);

/* Copy the sequence's physical block ids into out[0..cap).  Returns the
 * number of blocks (>= 0), or PA_ERR_INVALID_ARG if cap is too small. */
int pa_bm_block_table(const pa_bm *bm, int seq_id, int32_t *out, int cap);

/* Tokens the sequence holds, or a negative error code. */
int pa_bm_num_tokens(const pa_bm *bm, int seq_id);
int pa_bm_num_free(const pa_bm *bm);   /* free plus cached (both can be handed out) */
int pa_bm_refcount(const pa_bm *bm, int block); /* negative if out of range */

/* ---- automatic prefix caching (chained block hash, tenant salt) --------
 * [P4] "Deux couches, pas deux rivaux": every full block is keyed by a hash of
 * its parent block's key, its own tokens and optional extra data, so equal
 * token prefixes give equal key chains and find blocks already computed;
 * [P4] "Au-dela": a per-tenant salt mixed into the key keeps tenants apart.
 *
 * key_0 = H(0, salt, tokens[0..bs)), key_i = H(key_{i-1}, salt, tokens of block i),
 * H = 64-bit FNV-1a over the little-endian bytes of (parent key u64, salt u64,
 * each token as int32).  A key hit also compares the stored tokens, so hash
 * collisions cannot alias blocks.  Only full blocks are keyed.  A keyed block
 * whose refcount drops to zero stays cached (its K/V intact) and can be reused
 * by a later request until the pool runs short: allocation takes a free block
 * first, then evicts the least recently released cached block. */

/* New sequence of n tokens: leading full blocks whose keys are cached are
 * shared (refcount + 1); the rest are fresh, and the fresh full blocks are
 * keyed.  *num_cached_tokens = tokens whose K/V are already present (the
 * caller must compute and write the others before any other request can use
 * the newly keyed blocks).  PA_ERR_NO_BLOCKS leaves the state unchanged. */
int pa_bm_add_seq_cached(pa_bm *bm, int seq_id, const int32_t *tokens, int n, uint64_t salt,
                         int *num_cached_tokens);

/* Key the sequence's full blocks that are not keyed yet (for example after
 * decoding filled a block); tokens[0..n) are the sequence's tokens, n equal
 * to its length.  A block whose key already names another cached block stays
 * private.  Returns the number of blocks newly keyed, or an error code. */
int pa_bm_register_blocks(pa_bm *bm, int seq_id, const int32_t *tokens, int n, uint64_t salt);

/* Blocks held only by the cache (refcount 0, reusable on a hit). */
int pa_bm_num_cached(const pa_bm *bm);

/* Move a sequence from one manager to another (a device pool and a host pool
 * of the same block size): every block gets a fresh block in `to`, the pairs
 * (from block, to block) are written to pairs[2 * k], pairs[2 * k + 1] for the
 * caller's pa_swap_blocks, and the blocks in `from` are released.  All of the
 * sequence's blocks must be unshared (refcount 1): PA_ERR_REFCOUNT otherwise.
 * PA_ERR_NO_BLOCKS if `to` is short; *num_pairs = blocks moved; cap is the
 * room of pairs in pairs.  On failure nothing changes. */
int pa_bm_move_seq(pa_bm *from, pa_bm *to, int seq_id, int64_t *pairs, int cap, int *num_pairs);

/* Batched decode-step helper: append one slot to each of n sequences in order.
 * slots[k] receives the slot of seq_ids[k]; copy pairs are appended to
 * cow_pairs (int64 [n][2], host) and their count stored in *num_pairs.
 * Stops at the first failure and returns its code; *num_done tells how many
 * sequences were served (their effects stay). */
int pa_bm_append_slots(pa_bm *bm, const int32_t *seq_ids, int n, int64_t *slots,
                       int64_t *cow_pairs, int *num_pairs, int *num_done);

/* Padded block tables and lengths for a batch, ready for pa_decode:
 * tables [n][max_blocks_per_seq] (unused entries = -1), context_lens [n]. */
int pa_bm_build_tables(const pa_bm *bm, const int32_t *seq_ids, int n, int32_t *tables,
                       int max_blocks_per_seq, int32_t *context_lens);

/* ---- self-test of the bounded wait ----------------------------------------
 * Every wait of the decode kernels for staged data gives up after about two
 * seconds, sets PA_STATUS_WAIT_TIMEOUT and lets the kernel finish, so a copy
 * that never lands cannot hang the GPU.  This call runs that same wait in a
 * one-thread kernel on a barrier that nothing completes, with a limit of
 * limit_us microseconds (1..1000000), and ORs PA_STATUS_WAIT_TIMEOUT into
 * *dev_status when it gives up (it always does).  For tests of that path. */
int pa_selftest_wait_timeout(int32_t *dev_status, int limit_us, void *stream);

/* ---- misc --------------------------------------------------------------- */
const char *pa_last_error_string(void); /* thread-local, never NULL */
int pa_version(void);                   /* (major << 16) | minor */

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
