"""The library's host block manager against the model in oracle/ (same
documented allocation policy, so ids must match exactly), plus error paths."""
import numpy as np
import pytest

from oracle.block_manager_ref import BlockManagerModel, NoBlocks
from paged_kv_cache_237_gb300 import build as pa_build


@pytest.fixture(scope="module")
def binding():
    pa_build.build()
    from paged_kv_cache_237_gb300 import binding
    return binding


def same_state(bm, model, nb):
    assert bm.num_free() == model.num_free()
    for b in range(nb):
        assert bm.refcount(b) == model.refcount(b)
    for sid in model.seqs:
        assert bm.block_table(sid) == model.block_table(sid)
        assert bm.num_tokens(sid) == model.num_tokens(sid)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_operations_match_the_model_id_for_id(binding, seed):
    rng = np.random.default_rng(seed)
    nb, bs = 48, 16
    bm = binding.BlockManager(nb, bs)
    model = BlockManagerModel(nb, bs)
    live, nxt = [], 0
    for step in range(2500):
        op = int(rng.integers(0, 4))
        if op == 0 or not live:
            n = int(rng.integers(0, 60))
            try:
                model.add_seq(nxt, n)
                bm.add_seq(nxt, n)
                live.append(nxt)
            except NoBlocks:
                with pytest.raises(binding.PAError) as e:
                    bm.add_seq(nxt, n)
                assert e.value.code == binding.PA_ERR_NO_BLOCKS
            nxt += 1
        elif op == 1:
            p = int(rng.choice(live))
            model.fork(p, nxt)
            bm.fork(p, nxt)
            live.append(nxt)
            nxt += 1
        elif op == 2:
            sid = int(rng.choice(live))
            try:
                expect = model.append_slot(sid)
            except NoBlocks:
                with pytest.raises(binding.PAError) as e:
                    bm.append_slot(sid)
                assert e.value.code == binding.PA_ERR_NO_BLOCKS
            else:
                assert bm.append_slot(sid) == expect
        else:
            sid = int(rng.choice(live))
            model.free_seq(sid)
            bm.free_seq(sid)
            live.remove(sid)
        if step % 50 == 0:
            same_state(bm, model, nb)
    same_state(bm, model, nb)


def test_batched_append_and_tables(binding):
    bm = binding.BlockManager(64, 16)
    bm.add_seq(0, 37)
    bm.fork(0, 1)
    bm.add_seq(2, 16)
    slots, pairs = bm.append_slots([0, 1, 2])
    assert pairs.tolist() == [[2, 4]]             # seq 0 copies the shared partial block 2
    assert slots.tolist() == [4 * 16 + 5, 2 * 16 + 5, 5 * 16]
    tables, lens = bm.build_tables([0, 1, 2], 4)
    assert tables.tolist() == [[0, 1, 4, -1], [0, 1, 2, -1], [3, 5, -1, -1]]
    assert lens.tolist() == [38, 38, 17]


def test_error_codes(binding):
    bm = binding.BlockManager(4, 16)
    with pytest.raises(binding.PAError) as e:
        bm.free_seq(3)
    assert e.value.code == binding.PA_ERR_REFCOUNT
    bm.add_seq(1, 10)
    with pytest.raises(binding.PAError) as e:
        bm.add_seq(1, 10)
    assert e.value.code == binding.PA_ERR_INVALID_ARG
    with pytest.raises(binding.PAError) as e:
        bm.refcount(4)
    assert e.value.code == binding.PA_ERR_BAD_INDEX
    with pytest.raises(binding.PAError):
        bm.build_tables([1], 0)
    with pytest.raises(binding.PAError):
        binding.BlockManager(-1, 16)


def test_prefix_sharing_stores_the_prompt_once(binding):
    """50 requests over one 2048-token prompt (128 blocks of 16) hold 128
    prompt blocks, each with refcount 50."""
    bm = binding.BlockManager(2048, 16)
    bm.add_seq(1000, 2048)
    for r in range(50):
        bm.fork(1000, r)
    bm.free_seq(1000)
    assert bm.num_free() == 2048 - 128
    assert all(bm.refcount(b) == 50 for b in range(128))
