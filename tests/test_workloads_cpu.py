"""The seeded input recipes: lengths, placement and cache-write slots of the
synthetic workloads, checked on the host (no cache values are drawn)."""
import math

import numpy as np
import pytest

from paged_kv_cache_237_gb300.workloads import (WORKLOADS, context_lengths, new_token_slots, place_blocks,
                                                pool_blocks)


def lengths(name, **kw):
    w = WORKLOADS[name]
    return w, context_lengths(w, np.random.default_rng(w.seed), **kw)


def test_length_recipes():
    _, n = lengths("tiny_f32")
    assert n.tolist() == [7, 16, 33, 50]
    w, n = lengths("mha_llama2_7b")
    assert len(n) == w.num_seqs == 64 and n.min() >= 128 and n.max() <= 2048
    w, n = lengths("long_context")
    assert len(n) == 256 and int((n == 131072).sum()) == 8
    rest = n[n != 131072]
    assert rest.min() >= 16 and rest.max() <= 32768
    assert int(n.sum()) == 5_074_911                    # the figure the benchmark reports


def test_gqa_lognormal_and_its_sensitivity_case():
    w, a = lengths("gqa_llama3_70b")
    _, b = lengths("gqa_llama3_70b", gqa_sigma=0.5)
    assert len(a) == len(b) == 32
    assert a.min() >= 256 and a.max() <= 32768 and b.min() >= 256 and b.max() <= 32768
    # same normal draws, scaled: where neither is clipped, log(n / 4096) halves
    z = np.random.default_rng(w.seed).standard_normal(32)
    free = (np.abs(z) < math.log(8)) & (a > 256) & (a < 32768)
    assert np.allclose(np.log(b[free] / 4096.0), 0.5 * np.log(a[free] / 4096.0), atol=2e-3)
    assert np.std(np.log(b)) < np.std(np.log(a))
    assert int(a.sum()) == 219_876


@pytest.mark.parametrize("name", ["tiny_f32", "mha_llama2_7b", "gqa_llama3_70b", "long_context"])
def test_placement_is_a_valid_paging(name):
    w, n = lengths(name)
    per = [-(-int(x) // w.block_size) for x in n]
    nb = pool_blocks(w, sum(per))
    tables, need = place_blocks(n, w.block_size, nb, np.random.default_rng(1))
    assert need == sum(per) <= nb
    used = []
    for i, k in enumerate(per):
        row = tables[i]
        assert (row[:k] >= 0).all() and (row[:k] < nb).all() and (row[k:] == -1).all()
        used.extend(row[:k].tolist())
    assert len(set(used)) == len(used)                  # no block is shared: private pages
    if name == "long_context":
        assert 0.955 <= need / nb <= 0.961
    ident, _ = place_blocks(n, w.block_size, nb, np.random.default_rng(1), shuffle=False)
    assert ident[0, :per[0]].tolist() == list(range(per[0]))


def test_new_token_slot_is_the_last_position():
    w, n = lengths("gqa_llama3_70b")
    per = [-(-int(x) // w.block_size) for x in n]
    tables, _ = place_blocks(n, w.block_size, pool_blocks(w, sum(per)), np.random.default_rng(2))
    slots = new_token_slots(n, tables, w.block_size)
    for i, x in enumerate(n):
        blk, off = divmod(int(slots[i]), w.block_size)
        assert blk == tables[i, (int(x) - 1) // w.block_size] and off == (int(x) - 1) % w.block_size


def test_generators_are_deterministic():
    """Same seed, same inputs, bit for bit (both sides of every parity test
    are fed from these generators); another seed gives other values."""
    import torch
    from paged_kv_cache_237_gb300.workloads import decode_inputs, randn
    a, b = decode_inputs("tiny_f32"), decode_inputs("tiny_f32")
    for key in ("q", "k_cache", "v_cache", "block_tables", "context_lens", "k_new", "v_new", "slot_mapping"):
        assert torch.equal(a[key], b[key]), key
    x = randn((3, 1000), torch.bfloat16, 5, "cpu")
    assert torch.equal(x.view(torch.int16), randn((3, 1000), torch.bfloat16, 5, "cpu").view(torch.int16))
    assert not torch.equal(x, randn((3, 1000), torch.bfloat16, 6, "cpu"))
    # chunked drawing equals one draw of the same stream
    assert torch.equal(randn((4, 100), torch.float32, 9, "cpu", chunk_elems=64),
                       randn((4, 100), torch.float32, 9, "cpu"))


def test_a_slice_keeps_the_first_sequences_of_the_drawn_batch():
    """num_seqs keeps the first sequences of the same draw (lengths in their
    seeded order), with the pool sized by the workload's own rule."""
    from paged_kv_cache_237_gb300.workloads import decode_inputs
    w, full = lengths("gqa_llama3_70b")
    d = decode_inputs("gqa_llama3_70b", device="cpu", num_seqs=3)
    assert d["lens"].tolist() == full[:3].tolist()
    need = sum(-(-int(n) // w.block_size) for n in full[:3])
    assert d["num_blocks"] == pool_blocks(w, need) and d["k_cache"].shape[0] == d["num_blocks"]
    assert d["q"].shape == (3, w.num_q_heads, w.head_dim) and d["block_tables"].shape[0] == 3


@pytest.mark.parametrize("name", ["mha_llama2_7b", "gqa_llama3_70b"])
def test_fp32_twins_share_lengths_placement_and_values(name):
    """The fp32 batches draw the same lengths, placement and N(0, 1) values as
    their bf16 counterparts; the bf16 values are the fp32 ones rounded."""
    import torch
    from paged_kv_cache_237_gb300.workloads import decode_inputs
    a = decode_inputs(name, device="cpu", num_seqs=2)
    b = decode_inputs(name + "_f32", device="cpu", num_seqs=2)
    assert b["workload"].dtype == torch.float32 and a["workload"].dtype == torch.bfloat16
    assert a["lens"].tolist() == b["lens"].tolist()
    assert np.array_equal(a["tables"], b["tables"]) and a["num_blocks"] == b["num_blocks"]
    for key in ("q", "k_cache", "v_cache", "k_new", "v_new"):
        assert torch.equal(b[key].to(torch.bfloat16), a[key]), key
    assert torch.equal(a["slot_mapping"], b["slot_mapping"])
