"""Invariants of the block-manager model in oracle/block_manager_ref.py.

The model restates the pages' block manager (free pool, per-block refcount,
copy-on-write on a write into a shared block); these tests pin it by brute
force: refcounts recomputed from every live table, conservation of blocks,
and the copy-on-write cases spelled out by hand.
"""
import numpy as np
import pytest

from oracle.block_manager_ref import BlockManagerModel, NoBlocks


def recount(m: BlockManagerModel, num_blocks: int):
    ref = [0] * num_blocks
    for sid in m.seqs:
        for b in m.block_table(sid):
            ref[b] += 1
    return ref


def check(m, num_blocks):
    ref = recount(m, num_blocks)
    assert ref == m.ref
    used = sum(1 for r in ref if r > 0)
    assert used + m.num_free() == num_blocks
    assert len(set(m.free)) == len(m.free)
    assert all(ref[b] == 0 for b in m.free)
    for sid in m.seqs:
        n = m.num_tokens(sid)
        assert len(m.block_table(sid)) == -(-n // m.block_size)


def test_allocation_order_and_recycling():
    m = BlockManagerModel(8, 16)
    m.add_seq(0, 40)                  # 3 blocks: 0, 1, 2
    assert m.block_table(0) == [0, 1, 2]
    m.add_seq(1, 1)                   # block 3
    m.free_seq(0)                     # released 2, 1, 0 -> next handed out is 0
    m.add_seq(2, 17)
    assert m.block_table(2) == [0, 1]
    check(m, 8)


def test_fork_then_write_copies_only_the_partial_shared_block():
    m = BlockManagerModel(16, 16)
    m.add_seq(0, 37)                  # blocks 0,1,2; last holds 5 tokens
    m.fork(0, 1)
    assert [m.refcount(b) for b in (0, 1, 2)] == [2, 2, 2]
    slot, src, dst = m.append_slot(0)
    assert (src, dst) == (2, 3) and slot == 3 * 16 + 5
    assert m.block_table(0) == [0, 1, 3] and m.block_table(1) == [0, 1, 2]
    assert m.refcount(2) == 1 and m.refcount(3) == 1
    slot, src, dst = m.append_slot(1)  # now sole owner: write in place
    assert (src, dst) == (-1, -1) and slot == 2 * 16 + 5
    check(m, 16)


def test_write_after_full_shared_block_allocates_fresh_block():
    m = BlockManagerModel(8, 16)
    m.add_seq(0, 32)
    m.fork(0, 1)
    slot, src, dst = m.append_slot(1)
    assert (src, dst) == (-1, -1) and slot == 2 * 16
    assert m.refcount(0) == 2 and m.refcount(1) == 2
    check(m, 8)


def test_exhaustion_leaves_state_unchanged():
    m = BlockManagerModel(4, 16)
    m.add_seq(0, 48)
    with pytest.raises(NoBlocks):
        m.add_seq(1, 40)
    assert 1 not in m.seqs and m.num_free() == 1
    check(m, 4)


def test_random_operation_sequences_keep_invariants():
    rng = np.random.default_rng(0)
    nb = 64
    m = BlockManagerModel(nb, 16)
    live, next_id = [], 0
    for _ in range(3000):
        op = rng.integers(0, 4)
        try:
            if op == 0 or not live:
                m.add_seq(next_id, int(rng.integers(0, 70)))
                live.append(next_id)
                next_id += 1
            elif op == 1:
                m.fork(int(rng.choice(live)), next_id)
                live.append(next_id)
                next_id += 1
            elif op == 2:
                m.append_slot(int(rng.choice(live)))
            else:
                sid = int(rng.choice(live))
                m.free_seq(sid)
                live.remove(sid)
        except NoBlocks:
            pass
        check(m, nb)
