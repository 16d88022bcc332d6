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
#include <iterator>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"
#include "pa_internal.h"

struct PaSeq {
    std::vector<int32_t> blocks;
    int64_t num_tokens = 0;
};

// Identity of a keyed (prefix-cached) block: its chain key and what it was
// computed from, compared on every hit so that a hash collision never aliases.
struct PaKey {
    uint64_t key = 0, parent = 0, salt = 0;
    std::vector<int32_t> tokens;
};

struct pa_bm {
    int num_blocks = 0;
    int block_size = 0;
    std::vector<int32_t> free_stack;  // back() is handed out next
    std::vector<int32_t> refcount;
    std::unordered_map<int, PaSeq> seqs;
    // prefix cache
    std::vector<char> keyed;
    std::vector<PaKey> keys;
    std::unordered_map<uint64_t, int32_t> index;       // key -> keyed block
    std::list<int32_t> lru;                            // keyed blocks at refcount 0; front = evicted first
    std::vector<std::list<int32_t>::iterator> lru_pos;
    std::vector<char> in_lru;

    int available() const { return static_cast<int>(free_stack.size() + lru.size()); }

    void unkey(int32_t b) {
        auto it = index.find(keys[b].key);
        if (it != index.end() && it->second == b) index.erase(it);
        keyed[b] = 0;
        keys[b] = PaKey();
    }

    void lru_remove(int32_t b) {
        if (in_lru[b]) {
            lru.erase(lru_pos[b]);
            in_lru[b] = 0;
        }
    }

    // Hand out a block: a free one first, else evict the least recently
    // released cached block.  The caller has checked available() > 0.
    int32_t pop_free() {
        int32_t b;
        if (!free_stack.empty()) {
            b = free_stack.back();
            free_stack.pop_back();
        } else {
            b = lru.front();
            lru_remove(b);
            unkey(b);
        }
        refcount[b] = 1;
        return b;
    }

    // A block's last reference is gone: keyed blocks stay cached.
    void release(int32_t b) {
        if (keyed[b]) {
            lru.push_back(b);
            lru_pos[b] = std::prev(lru.end());
            in_lru[b] = 1;
        } else {
            free_stack.push_back(b);
        }
    }
};

namespace {

// 64-bit FNV-1a over little-endian bytes.
struct Fnv1a64 {
    uint64_t h = 14695981039346656037ull;
    void byte(uint8_t b) {
        h ^= b;
        h *= 1099511628211ull;
    }
    void u64(uint64_t v) {
        for (int i = 0; i < 8; ++i) byte(static_cast<uint8_t>(v >> (8 * i)));
    }
    void i32(int32_t v) {
        const uint32_t u = static_cast<uint32_t>(v);
        for (int i = 0; i < 4; ++i) byte(static_cast<uint8_t>(u >> (8 * i)));
    }
};

uint64_t block_key(uint64_t parent, uint64_t salt, const int32_t *tokens, int bs) {
    Fnv1a64 f;
    f.u64(parent);
    f.u64(salt);
    for (int i = 0; i < bs; ++i) f.i32(tokens[i]);
    return f.h;
}

// The cached block for (key, parent, salt, tokens), or -1.
int32_t lookup(const pa_bm *bm, uint64_t key, uint64_t parent, uint64_t salt, const int32_t *tokens) {
    auto it = bm->index.find(key);
    if (it == bm->index.end()) return -1;
    const PaKey &k = bm->keys[it->second];
    if (k.parent != parent || k.salt != salt) return -1;
    for (int i = 0; i < bm->block_size; ++i)
        if (k.tokens[i] != tokens[i]) return -1;
    return it->second;
}

void set_key(pa_bm *bm, int32_t b, uint64_t key, uint64_t parent, uint64_t salt, const int32_t *tokens) {
    bm->keyed[b] = 1;
    bm->keys[b].key = key;
    bm->keys[b].parent = parent;
    bm->keys[b].salt = salt;
    bm->keys[b].tokens.assign(tokens, tokens + bm->block_size);
    bm->index[key] = b;
}

}  // namespace

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
    bm->keyed.assign(num_blocks, 0);
    bm->keys.resize(num_blocks);
    bm->lru_pos.resize(num_blocks);
    bm->in_lru.assign(num_blocks, 0);
    return bm;
}

extern "C" void pa_bm_destroy(pa_bm *bm) { delete bm; }

extern "C" int pa_bm_add_seq(pa_bm *bm, int seq_id, int num_tokens) {
    if (!bm || seq_id < 0 || num_tokens < 0)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_add_seq: bad manager, id or length");
    if (bm->seqs.count(seq_id))
        return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_add_seq: sequence id already live");
    int64_t need = (static_cast<int64_t>(num_tokens) + bm->block_size - 1) / bm->block_size;
    if (need > bm->available()) return pa_fail(PA_ERR_NO_BLOCKS, "pa_bm_add_seq: free pool exhausted");
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
        if (bm->available() == 0) return pa_fail(PA_ERR_NO_BLOCKS, "pa_bm_append_slot: free pool exhausted");
        s.blocks.push_back(bm->pop_free());
    } else {
        int32_t last = s.blocks.back();
        if (bm->refcount[last] > 1) {
            if (bm->available() == 0)
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
        if (--bm->refcount[*b] == 0) bm->release(*b);
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
    return bm->available();
}

extern "C" int pa_bm_num_cached(const pa_bm *bm) {
    if (!bm) return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_num_cached: null manager");
    return static_cast<int>(bm->lru.size());
}

extern "C" int pa_bm_add_seq_cached(pa_bm *bm, int seq_id, const int32_t *tokens, int n, uint64_t salt,
                                    int *num_cached_tokens) {
    if (!bm || seq_id < 0 || n < 0 || (n > 0 && !tokens) || !num_cached_tokens)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_add_seq_cached: bad arguments");
    if (bm->seqs.count(seq_id)) return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_add_seq_cached: sequence id already live");
    const int bs = bm->block_size;
    const int nfull = n / bs, nblocks = (n + bs - 1) / bs;
    // Plan without touching the state: the leading run of cache hits.
    std::vector<uint64_t> keyv(nfull);
    std::vector<int32_t> hits;
    uint64_t parent = 0;
    bool hitting = true;
    int lru_hits = 0;
    for (int i = 0; i < nfull; ++i) {
        keyv[i] = block_key(parent, salt, tokens + static_cast<int64_t>(i) * bs, bs);
        if (hitting) {
            const int32_t b = lookup(bm, keyv[i], parent, salt, tokens + static_cast<int64_t>(i) * bs);
            if (b >= 0) {
                hits.push_back(b);
                lru_hits += bm->in_lru[b] ? 1 : 0;
            } else {
                hitting = false;
            }
        }
        parent = keyv[i];
    }
    const int fresh = nblocks - static_cast<int>(hits.size());
    if (fresh > bm->available() - lru_hits) return pa_fail(PA_ERR_NO_BLOCKS, "pa_bm_add_seq_cached: free pool exhausted");
    PaSeq s;
    s.blocks.reserve(nblocks);
    for (int32_t b : hits) {
        bm->lru_remove(b);
        bm->refcount[b] += 1;
        s.blocks.push_back(b);
    }
    for (int i = static_cast<int>(hits.size()); i < nblocks; ++i) {
        const int32_t b = bm->pop_free();
        s.blocks.push_back(b);
        if (i < nfull && !bm->index.count(keyv[i]))
            set_key(bm, b, keyv[i], i ? keyv[i - 1] : 0, salt, tokens + static_cast<int64_t>(i) * bs);
    }
    s.num_tokens = n;
    bm->seqs.emplace(seq_id, std::move(s));
    *num_cached_tokens = static_cast<int>(hits.size()) * bs;
    return PA_OK;
}

extern "C" int pa_bm_register_blocks(pa_bm *bm, int seq_id, const int32_t *tokens, int n, uint64_t salt) {
    if (!bm || n < 0 || (n > 0 && !tokens)) return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_register_blocks: bad arguments");
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return pa_fail(PA_ERR_REFCOUNT, "pa_bm_register_blocks: unknown sequence");
    if (it->second.num_tokens != n)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_register_blocks: n must equal the sequence's length");
    const int bs = bm->block_size;
    uint64_t parent = 0;
    int added = 0;
    for (int i = 0; i < n / bs; ++i) {
        const int32_t *tk = tokens + static_cast<int64_t>(i) * bs;
        const uint64_t key = block_key(parent, salt, tk, bs);
        const int32_t b = it->second.blocks[i];
        if (!bm->keyed[b] && !bm->index.count(key)) {
            set_key(bm, b, key, parent, salt, tk);
            ++added;
        }
        parent = key;
    }
    return added;
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

extern "C" int pa_bm_move_seq(pa_bm *from, pa_bm *to, int seq_id, int64_t *pairs, int cap, int *num_pairs) {
    if (!from || !to || !num_pairs || cap < 0 || (cap > 0 && !pairs) || from == to)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_move_seq: bad arguments");
    if (from->block_size != to->block_size)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_move_seq: block sizes differ");
    auto it = from->seqs.find(seq_id);
    if (it == from->seqs.end()) return pa_fail(PA_ERR_REFCOUNT, "pa_bm_move_seq: unknown sequence");
    if (to->seqs.count(seq_id)) return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_move_seq: id already live in the target");
    const std::vector<int32_t> &blocks = it->second.blocks;
    for (int32_t b : blocks)
        if (from->refcount[b] != 1) return pa_fail(PA_ERR_REFCOUNT, "pa_bm_move_seq: a block is shared");
    if (static_cast<int64_t>(blocks.size()) > cap) return pa_fail(PA_ERR_INVALID_ARG, "pa_bm_move_seq: pairs too small");
    if (static_cast<int64_t>(blocks.size()) > to->available())
        return pa_fail(PA_ERR_NO_BLOCKS, "pa_bm_move_seq: target pool exhausted");
    PaSeq moved;
    moved.num_tokens = it->second.num_tokens;
    for (size_t k = 0; k < blocks.size(); ++k) {
        const int32_t nb = to->pop_free();
        moved.blocks.push_back(nb);
        pairs[2 * k] = blocks[k];
        pairs[2 * k + 1] = nb;
    }
    for (auto b = blocks.rbegin(); b != blocks.rend(); ++b) {
        from->refcount[*b] = 0;
        from->release(*b);
    }
    *num_pairs = static_cast<int>(blocks.size());
    from->seqs.erase(it);
    to->seqs.emplace(seq_id, std::move(moved));
    return PA_OK;
}
