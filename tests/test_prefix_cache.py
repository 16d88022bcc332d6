"""Automatic prefix caching by chained block keys with a tenant salt.

Pins: the model's FNV-1a against the hash's published test vectors; hand-
worked reuse, salting, partial-prefix and eviction cases on the model; the
library's block manager against the model id for id on random multi-tenant
request streams ("PagedAttention et RadixAttention : parlons de KV Cache",
aitalk.it, "Deux couches, pas deux rivaux" and "Au-dela")."""
import numpy as np
import pytest

from oracle.block_manager_ref import BlockManagerModel, NoBlocks, block_key, fnv1a64
from paged_kv_cache_237_gb300 import build as pa_build


@pytest.fixture(scope="module")
def binding():
    pa_build.build()
    from paged_kv_cache_237_gb300 import binding
    return binding


def test_fnv1a64_published_vectors():
    assert fnv1a64(b"") == 0xCBF29CE484222325
    assert fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert fnv1a64(b"foobar") == 0x85944171F73967E8


def test_key_chain_depends_on_parent_salt_and_tokens():
    t = list(range(16))
    k0 = block_key(0, 7, t)
    assert block_key(0, 7, t) == k0
    assert block_key(0, 8, t) != k0                      # other tenant
    assert block_key(1, 7, t) != k0                      # other parent
    assert block_key(0, 7, t[:-1] + [99]) != k0          # other tokens


def test_model_same_prompt_reuses_full_blocks_only():
    m = BlockManagerModel(32, 16)
    prompt = list(range(100, 150))                       # 50 tokens: 3 full blocks + 2
    assert m.add_seq_cached(0, prompt, salt=1) == 0
    assert m.add_seq_cached(1, prompt, salt=1) == 48
    t0, t1 = m.block_table(0), m.block_table(1)
    assert t0[:3] == t1[:3] and t0[3] != t1[3]           # partial last block stays private
    assert [m.refcount(b) for b in t0[:3]] == [2, 2, 2]


def test_model_salt_isolates_tenants():
    m = BlockManagerModel(32, 16)
    prompt = list(range(64))
    m.add_seq_cached(0, prompt, salt=1)
    assert m.add_seq_cached(1, prompt, salt=2) == 0
    assert set(m.block_table(0)).isdisjoint(m.block_table(1))


def test_model_partial_prefix_and_divergence():
    m = BlockManagerModel(32, 16)
    a = list(range(64))
    b = list(range(40)) + [999] * 24                     # diverges inside block 2
    m.add_seq_cached(0, a)
    assert m.add_seq_cached(1, b) == 32
    assert m.block_table(1)[:2] == m.block_table(0)[:2]
    assert m.block_table(1)[2] != m.block_table(0)[2]


def test_model_freed_blocks_stay_cached_then_evict_lru():
    m = BlockManagerModel(6, 16)
    m.add_seq_cached(0, list(range(48)))                  # blocks 0,1,2 keyed
    m.free_seq(0)                                         # released 2, 1, 0 -> cached
    assert m.num_cached() == 3 and m.num_free() == 6
    assert m.add_seq_cached(1, list(range(48))) == 48     # full hit from the cache
    assert m.num_cached() == 0
    m.free_seq(1)                                         # cached again, release order 2, 1, 0
    m.add_seq(2, 16 * 4)                                  # 3 free blocks + evicts the LRU one (block 2)
    assert list(m.lru) == [1, 0]
    m.free_seq(2)                                         # unkeyed blocks go back to the free pool
    assert m.add_seq_cached(3, list(range(48))) == 32     # blocks 0 and 1 hit; block 2 was evicted
    assert m.block_table(3)[:2] == [0, 1]
    with pytest.raises(NoBlocks):
        m.add_seq(4, 16 * 10)


def _random_stream(rng, n_ops, tenants=3, prompts_per_tenant=3):
    bank = {(t, p): rng.integers(0, 50000, size=int(rng.integers(16, 200))).tolist()
            for t in range(tenants) for p in range(prompts_per_tenant)}
    ops = []
    for _ in range(n_ops):
        r = rng.random()
        if r < 0.45:
            t, p = int(rng.integers(0, tenants)), int(rng.integers(0, prompts_per_tenant))
            suffix = rng.integers(0, 50000, size=int(rng.integers(0, 40))).tolist()
            cut = int(rng.integers(1, len(bank[(t, p)]) + 1))
            ops.append(("add", bank[(t, p)][:cut] + suffix, 1000 + t))
        elif r < 0.6:
            ops.append(("append",))
        elif r < 0.7:
            ops.append(("register",))
        else:
            ops.append(("free",))
    return ops


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_library_prefix_cache_matches_model(binding, seed):
    rng = np.random.default_rng(seed)
    nb, bs = 64, 16
    bm = binding.BlockManager(nb, bs)
    m = BlockManagerModel(nb, bs)
    live, tokens, salts, nxt = [], {}, {}, 0
    for op in _random_stream(rng, 1500):
        if op[0] == "add":
            _, toks, salt = op
            try:
                exp = m.add_seq_cached(nxt, toks, salt)
            except NoBlocks:
                with pytest.raises(binding.PAError) as e:
                    bm.add_seq_cached(nxt, toks, salt)
                assert e.value.code == binding.PA_ERR_NO_BLOCKS
            else:
                assert bm.add_seq_cached(nxt, toks, salt) == exp
                live.append(nxt)
                tokens[nxt], salts[nxt] = list(toks), salt
            nxt += 1
        elif not live:
            continue
        elif op[0] == "append":
            sid = int(rng.choice(live))
            try:
                exp = m.append_slot(sid)
            except NoBlocks:
                with pytest.raises(binding.PAError):
                    bm.append_slot(sid)
            else:
                assert bm.append_slot(sid) == exp
                tokens[sid].append(int(rng.integers(0, 50000)))
        elif op[0] == "register":
            sid = int(rng.choice(live))
            assert bm.register_blocks(sid, tokens[sid], salts[sid]) == m.register_blocks(sid, tokens[sid], salts[sid])
        else:
            sid = int(rng.choice(live))
            m.free_seq(sid)
            bm.free_seq(sid)
            live.remove(sid)
        assert bm.num_free() == m.num_free() and bm.num_cached() == m.num_cached()
    for sid in live:
        assert bm.block_table(sid) == m.block_table(sid)
    for b in range(nb):
        assert bm.refcount(b) == m.refcount(b)


def test_library_tenant_isolation_and_reuse(binding):
    bm = binding.BlockManager(512, 16)
    system = list(range(2048))
    assert bm.add_seq_cached(0, system + [1, 2, 3], salt=11) == 0
    assert bm.add_seq_cached(1, system + [4, 5], salt=11) == 2048
    assert bm.add_seq_cached(2, system + [4, 5], salt=12) == 0
    assert bm.block_table(0)[:128] == bm.block_table(1)[:128]
    assert set(bm.block_table(2)).isdisjoint(bm.block_table(0))
