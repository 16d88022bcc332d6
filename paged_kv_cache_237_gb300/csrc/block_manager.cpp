// Host block manager: free pool, per-block reference counts, copy-on-write
// trigger.  Pure host code; it never touches the device.
//
// "PagedAttention" (robocikowo.com), "Komponenty": the block manager allocates
// and releases physical blocks and keeps the free pool; shared prefix blocks are
// reference-counted and duplicated lazily on modification.  "Jak dziala": blocks
// are allocated on demand as a sequence grows; a write into a shared block
// triggers the copy.  The policy details (LIFO pool starting at block 0,
// last-to-first release) are this library's choice and are declared in pa.h.
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"
#include "pa_internal.h"

struct PaSeq {
    std::vector<int32_t> blocks;
    int64_t num_tokens = 0;
};

struct pa_bm {
    int num_blocks = 0;
    int block_size = 0;
    std::vector<int32_t> free_stack;  // back() is handed out next
    std::vector<int32_t> refcount;
    std::unordered_map<int, PaSeq> seqs;

    int32_t pop_free() {
        int32_t b = free_stack.back();
        free_stack.pop_back();
        refcount[b] = 1;
        return b;
    }
};

extern "C" pa_bm *pa_bm_create(int num_blocks, int block_size) {
    if (num_blocks < 0 || block_size <= 0) {
        pa_set_error("pa_bm_create: num_blocks must be >= 0 and block_size > 0");
        return nullptr;
    }
    pa_bm *bm = new (std::nothrow) pa_bm;
    if (!bm) {
        pa_set_error("pa_bm_create: out of host memory");
        return nullptr;
    }
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->free_stack.resize(num_blocks);
    for (int i = 0; i < num_blocks; ++i) bm->free_stack[i] = num_blocks - 1 - i;
    bm->refcount.assign(num_blocks, 0);
    return bm;
}

extern "C" void pa_bm_destroy(pa_bm *bm) { delete bm; }

extern "C" int pa_bm_add_seq(pa_bm *bm, int seq_id, int num_tokens) {
    if (!bm || seq_id < 0 || num_tokens < 0)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_add_seq: bad manager, id or length");
    if (bm->seqs.count(seq_id))
        return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_add_seq: sequence id already live");
    int64_t need = (static_cast<int64_t>(num_tokens) + bm->block_size - 1) / bm->block_size;
    if (need > static_cast<int64_t>(bm->free_stack.size()))
        return pa_fail(PA_ERR_NO_BLOCKS, "pa_bm_add_seq: free pool exhausted");
    PaSeq s;
    s.blocks.reserve(need);
    for (int64_t k = 0; k < need; ++k) s.blocks.push_back(bm->pop_free());
    s.num_tokens = num_tokens;
    bm->seqs.emplace(seq_id, std::move(s));
    return PA_OK;
}

extern "C" int pa_bm_fork(pa_bm *bm, int parent_id, int child_id) {
    if (!bm || child_id < 0) return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_fork: bad arguments");
    auto it = bm->seqs.find(parent_id);
    if (it == bm->seqs.end()) return pa_fail(PA_ERR_REFCOUNT, "pa_bm_fork: unknown parent");
    if (bm->seqs.count(child_id))
        return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_fork: child id already live");
    PaSeq child = it->second;
    for (int32_t b : child.blocks) bm->refcount[b] += 1;
    bm->seqs.emplace(child_id, std::move(child));
    return PA_OK;
}

extern "C" int pa_bm_append_slot(pa_bm *bm, int seq_id, int64_t *slot, int32_t *cow_src,
                                 int32_t *cow_dst) {
    if (!bm || !slot || !cow_src || !cow_dst)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_append_slot: null argument");
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return pa_fail(PA_ERR_REFCOUNT, "pa_bm_append_slot: unknown sequence");
    PaSeq &s = it->second;
    const int64_t off = s.num_tokens % bm->block_size;
    int32_t src = -1, dst = -1;
    if (off == 0) {
        if (bm->free_stack.empty())
            return pa_fail(PA_ERR_NO_BLOCKS, "pa_bm_append_slot: free pool exhausted");
        s.blocks.push_back(bm->pop_free());
    } else {
        int32_t last = s.blocks.back();
        if (bm->refcount[last] > 1) {
            if (bm->free_stack.empty())
                return pa_fail(PA_ERR_NO_BLOCKS, "pa_bm_append_slot: free pool exhausted");
            int32_t fresh = bm->pop_free();
            bm->refcount[last] -= 1;
            s.blocks.back() = fresh;
            src = last;
            dst = fresh;
        }
    }
    s.num_tokens += 1;
    *slot = static_cast<int64_t>(s.blocks.back()) * bm->block_size + off;
    *cow_src = src;
    *cow_dst = dst;
    return PA_OK;
}

extern "C" int pa_bm_free_seq(pa_bm *bm, int seq_id) {
    if (!bm) return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_free_seq: null manager");
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return pa_fail(PA_ERR_REFCOUNT, "pa_bm_free_seq: unknown sequence");
    const std::vector<int32_t> &blocks = it->second.blocks;
    for (auto b = blocks.rbegin(); b != blocks.rend(); ++b) {
        if (--bm->refcount[*b] == 0) bm->free_stack.push_back(*b);
    }
    bm->seqs.erase(it);
    return PA_OK;
}

extern "C" int pa_bm_block_table(const pa_bm *bm, int seq_id, int32_t *out, int cap) {
    if (!bm || (cap > 0 && !out) || cap < 0)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_block_table: bad arguments");
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return pa_fail(PA_ERR_REFCOUNT, "pa_bm_block_table: unknown sequence");
    const auto &blocks = it->second.blocks;
    if (static_cast<int64_t>(blocks.size()) > cap)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_block_table: output too small");
    for (size_t k = 0; k < blocks.size(); ++k) out[k] = blocks[k];
    return static_cast<int>(blocks.size());
}

extern "C" int pa_bm_num_tokens(const pa_bm *bm, int seq_id) {
    if (!bm) return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_num_tokens: null manager");
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return pa_fail(PA_ERR_REFCOUNT, "pa_bm_num_tokens: unknown sequence");
    return static_cast<int>(it->second.num_tokens);
}

extern "C" int pa_bm_num_free(const pa_bm *bm) {
    if (!bm) return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_num_free: null manager");
    return static_cast<int>(bm->free_stack.size());
}

extern "C" int pa_bm_refcount(const pa_bm *bm, int block) {
    if (!bm || block < 0 || block >= bm->num_blocks)
        return pa_fail(PA_ERR_BAD_INDEX, "pa_bm_refcount: block out of range");
    return bm->refcount[block];
}

extern "C" int pa_bm_append_slots(pa_bm *bm, const int32_t *seq_ids, int n, int64_t *slots,
                                  int64_t *cow_pairs, int *num_pairs, int *num_done) {
    if (!bm || n < 0 || (n > 0 && (!seq_ids || !slots || !cow_pairs)) || !num_pairs || !num_done)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_append_slots: bad arguments");
    *num_pairs = 0;
    *num_done = 0;
    for (int k = 0; k < n; ++k) {
        int32_t src, dst;
        int rc = pa_bm_append_slot(bm, seq_ids[k], &slots[k], &src, &dst);
        if (rc != PA_OK) return rc;
        if (src >= 0) {
            cow_pairs[2 * *num_pairs] = src;
            cow_pairs[2 * *num_pairs + 1] = dst;
            *num_pairs += 1;
        }
        *num_done = k + 1;
    }
    return PA_OK;
}

extern "C" int pa_bm_build_tables(const pa_bm *bm, const int32_t *seq_ids, int n, int32_t *tables,
                                  int max_blocks_per_seq, int32_t *context_lens) {
    if (!bm || n < 0 || max_blocks_per_seq < 1 || (n > 0 && (!seq_ids || !tables || !context_lens)))
        return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_build_tables: bad arguments");
    for (int k = 0; k < n; ++k) {
        auto it = bm->seqs.find(seq_ids[k]);
        if (it == bm->seqs.end())
            return pa_fail(PA_ERR_REFCOUNT, "pa_bm_build_tables: unknown sequence");
        const auto &blocks = it->second.blocks;
        if (static_cast<int64_t>(blocks.size()) > max_blocks_per_seq)
            return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_build_tables: table row too short");
        int32_t *row = tables + static_cast<int64_t>(k) * max_blocks_per_seq;
        for (int j = 0; j < max_blocks_per_seq; ++j)
            row[j] = j < static_cast<int>(blocks.size()) ? blocks[j] : -1;
        context_lens[k] = static_cast<int32_t>(it->second.num_tokens);
    }
    return PA_OK;
}
