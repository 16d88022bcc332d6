"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test ties the oracle to a library routine on contiguous data, a closed
form, an invariant the pages state, or brute force on tiny inputs.  The pages
("PagedAttention et RadixAttention : parlons de KV Cache", section
"PagedAttention : la memoire comme un systeme d'exploitation") say that paging
only changes where K/V live, never what attention returns; that is the
contiguous-equivalence pin.  Sharing and copy-on-write pins follow the same
section's fourth step and "PagedAttention" (robocikowo.com), "Jak dziala".
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


# ---------------------------------------------------------------- helpers ---
def place_contiguous(K_list, V_list, block_size, num_blocks, perm, dtype):
    """Test-side scatter of contiguous per-sequence K/V [n, Hkv, hd] into a
    paged cache, using numpy indexing (independent of the oracle's gather).
    Logical blocks take pool ids perm[0], perm[1], ... in sequence order."""
    Hkv, hd = K_list[0].shape[1], K_list[0].shape[2]
    kc = torch.full((num_blocks, Hkv, block_size, hd), float("nan"), dtype=torch.float64)
    vc = kc.clone()
    per = [max(1, -(-k.shape[0] // block_size)) for k in K_list]
    tables = -np.ones((len(K_list), max(per)), dtype=np.int32)
    pos = 0
    for i, (K, V) in enumerate(zip(K_list, V_list)):
        n = K.shape[0]
        ids = np.asarray(perm[pos:pos + per[i]])
        pos += per[i]
        tables[i, :per[i]] = ids
        t = np.arange(n)
        blk = torch.from_numpy(ids[t // block_size].astype(np.int64))
        off = torch.from_numpy(t % block_size)
        # cache[blk, h, off, :] = K[t, h, :]
        kc[blk, :, off, :] = K.to(torch.float64)
        vc[blk, :, off, :] = V.to(torch.float64)
    return kc.to(dtype), vc.to(dtype), torch.from_numpy(tables)


def sdpa_reference(q, K, V, scale):
    """torch SDPA in fp64 on contiguous data.  q [Hq, hd]; K, V [n, Hkv, hd]."""
    qq = q.to(torch.float64)[None, :, None, :]              # [1, Hq, 1, hd]
    kk = K.to(torch.float64).permute(1, 0, 2)[None]           # [1, Hkv, n, hd]
    vv = V.to(torch.float64).permute(1, 0, 2)[None]
    o = F.scaled_dot_product_attention(qq, kk, vv, scale=scale,
                                       enable_gqa=q.shape[0] != K.shape[1])
    return o[0, :, 0, :]                                      # [Hq, hd]


def rand_case(seed, lens, Hq, Hkv, hd, dtype):
    g = torch.Generator().manual_seed(seed)
    K = [torch.randn(n, Hkv, hd, generator=g).to(dtype) for n in lens]
    V = [torch.randn(n, Hkv, hd, generator=g).to(dtype) for n in lens]
    q = torch.randn(len(lens), Hq, hd, generator=g).to(dtype)
    return q, K, V


def run_oracle(q, kc, vc, tables, lens, scale, lib=None):
    return oracle.paged_decode(q, kc, vc, tables, torch.tensor(lens, dtype=torch.int32), scale,
                               threads=2, lib=lib)


# ------------------------------------------------ contiguous equivalence ---
@pytest.mark.parametrize("cache_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("bs,hd,Hq,Hkv", [(16, 64, 4, 4), (32, 128, 8, 2), (16, 128, 8, 1),
                                          (32, 64, 6, 3)])
def test_oracle_equals_sdpa_on_contiguous_data(cache_dtype, bs, hd, Hq, Hkv):
    lens = [1, 15, 16, 17, 33, 64, 95]
    q, K, V = rand_case(7 + bs + hd, lens, Hq, Hkv, hd, cache_dtype)
    need = sum(-(-n // bs) for n in lens)
    perm = np.random.default_rng(11).permutation(need + 9)
    kc, vc, tables = place_contiguous(K, V, bs, need + 9, perm, cache_dtype)
    scale = 1.0 / math.sqrt(hd)
    out = run_oracle(q, kc, vc, tables, lens, scale)
    for i in range(len(lens)):
        ref = sdpa_reference(q[i], K[i], V[i], scale)
        assert torch.allclose(out[i], ref, rtol=0, atol=1e-12), (i, (out[i] - ref).abs().max())


def test_block_permutation_invariance_is_bitwise():
    lens = [5, 16, 40, 77]
    q, K, V = rand_case(3, lens, 4, 2, 64, torch.bfloat16)
    need = sum(-(-n // 16) for n in lens)
    outs = []
    for s in range(4):
        perm = np.random.default_rng(100 + s).permutation(need + 20)
        kc, vc, tables = place_contiguous(K, V, 16, need + 20, perm, torch.bfloat16)
        outs.append(run_oracle(q, kc, vc, tables, lens, 0.125))
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_shared_prefix_blocks_equal_private_copies():
    """Two sequences whose first 3 blocks hold the same prefix: pointing both
    tables at one physical copy gives the same outputs as private copies."""
    bs, hd, H = 16, 64, 2
    g = torch.Generator().manual_seed(5)
    prefix_k = torch.randn(48, H, hd, generator=g)
    prefix_v = torch.randn(48, H, hd, generator=g)
    suf = [(torch.randn(n, H, hd, generator=g), torch.randn(n, H, hd, generator=g)) for n in (9, 21)]
    K = [torch.cat([prefix_k, s[0]]) for s in suf]
    V = [torch.cat([prefix_v, s[1]]) for s in suf]
    q = torch.randn(2, H, hd, generator=g)
    lens = [57, 69]
    # private: 4 + 5 blocks
    kc, vc, tables = place_contiguous(K, V, bs, 12, np.arange(12)[::-1].copy(), torch.float32)
    private = run_oracle(q, kc, vc, tables, lens, 0.1)
    # shared: sequence 1's first 3 table entries point at sequence 0's prefix blocks
    shared_tables = tables.clone()
    shared_tables[1, :3] = tables[0, :3]
    kc2, vc2 = kc.clone(), vc.clone()
    kc2[tables[1, :3].long()] = float("nan")   # the now-unused private prefix copy
    vc2[tables[1, :3].long()] = float("nan")
    shared = run_oracle(q, kc2, vc2, shared_tables, lens, 0.1)
    assert torch.equal(private, shared)


def test_copy_on_write_leaves_the_other_sharer_unchanged():
    """Two samples share every block, the last one partial.  The first writes
    its next token: copy the shared last block, repoint its table, write the
    token.  The other sample's blocks and output are untouched; the writer's
    output equals contiguous attention over its extended sequence."""
    bs, hd, H = 16, 64, 2
    g = torch.Generator().manual_seed(9)
    n = 37
    K0 = torch.randn(n, H, hd, generator=g)
    V0 = torch.randn(n, H, hd, generator=g)
    kc, vc, tables = place_contiguous([K0], [V0], bs, 8, np.arange(8), torch.float32)
    tables = torch.cat([tables, tables])            # both samples: blocks 0, 1, 2
    q = torch.randn(2, H, hd, generator=g)
    before = run_oracle(q, kc, vc, tables, [n, n], 0.125)
    other_blocks = kc[tables[1].long()].clone()
    # sample 0 writes token n into a copy of the shared partial block 2 -> block 5
    oracle.copy_blocks(kc, vc, torch.tensor([[2, 5]], dtype=torch.int64))
    tables[0, 2] = 5
    k_new = torch.randn(1, H, hd, generator=g)
    v_new = torch.randn(1, H, hd, generator=g)
    oracle.reshape_and_cache(k_new, v_new, kc, vc, torch.tensor([5 * bs + n % bs]))
    after = run_oracle(q, kc, vc, tables, [n + 1, n], 0.125)
    assert torch.equal(after[1], before[1])
    assert torch.equal(kc[tables[1].long()].view(torch.int32), other_blocks.view(torch.int32))
    ref = sdpa_reference(q[0], torch.cat([K0, k_new]), torch.cat([V0, v_new]), 0.125)
    assert torch.allclose(after[0], ref, rtol=0, atol=1e-12)


# ------------------------------------------------------- closed forms ------
def test_single_token_returns_its_value_exactly():
    q, K, V = rand_case(1, [1, 1], 4, 4, 64, torch.float32)
    kc, vc, tables = place_contiguous(K, V, 16, 4, np.array([3, 1]), torch.float32)
    out = run_oracle(q, kc, vc, tables, [1, 1], 0.125)
    for i in range(2):
        assert torch.equal(out[i], V[i][0].to(torch.float64))


def test_zero_scale_gives_mean_of_values():
    lens = [3, 40]
    q, K, V = rand_case(2, lens, 2, 2, 64, torch.float32)
    kc, vc, tables = place_contiguous(K, V, 16, 6, np.array([5, 0, 4, 2]), torch.float32)
    out = run_oracle(q, kc, vc, tables, lens, 0.0)
    for i, n in enumerate(lens):
        mean = V[i].to(torch.float64).numpy().mean(axis=0)  # [Hkv, hd]
        assert np.allclose(out[i].numpy(), mean, rtol=0, atol=1e-13)


def test_identical_keys_give_mean_of_values():
    n, H, hd = 29, 2, 64
    g = torch.Generator().manual_seed(4)
    key = torch.randn(1, H, hd, generator=g)
    K = key.expand(n, H, hd).clone()
    V = torch.randn(n, H, hd, generator=g)
    q = torch.randn(1, H, hd, generator=g)
    kc, vc, tables = place_contiguous([K], [V], 16, 2, np.array([1, 0]), torch.float32)
    out = run_oracle(q, kc, vc, tables, [n], 0.7)
    assert np.allclose(out[0].numpy(), V.double().numpy().mean(axis=0), rtol=0, atol=1e-13)


def test_two_tokens_follow_the_logistic_closed_form():
    """softmax over two logits is the logistic function of their difference."""
    H, hd, scale = 3, 64, 0.125
    q, K, V = rand_case(6, [2], H, H, hd, torch.float32)
    kc, vc, tables = place_contiguous(K, V, 16, 1, np.array([0]), torch.float32)
    out = run_oracle(q, kc, vc, tables, [2], scale)
    qd, kd, vd = q[0].double(), K[0].double(), V[0].double()
    for h in range(H):
        delta = scale * float(qd[h] @ (kd[0, h] - kd[1, h]))
        w0 = 1.0 / (1.0 + math.exp(-delta))
        ref = w0 * vd[0, h] + (1.0 - w0) * vd[1, h]
        assert torch.allclose(out[0, h], ref, rtol=0, atol=1e-13)


def test_dominant_key_selects_its_value():
    """With orthogonal keys and q aligned with key j, a large scale puts all
    the weight on token j."""
    n, hd = 16, 64
    K = torch.zeros(n, 1, hd)
    for t in range(n):
        K[t, 0, t] = 1.0
    g = torch.Generator().manual_seed(8)
    V = torch.randn(n, 1, hd, generator=g)
    j = 11
    q = torch.zeros(1, 1, hd)
    q[0, 0, j] = 1.0
    kc, vc, tables = place_contiguous([K], [V], 16, 3, np.array([2]), torch.float32)
    out = run_oracle(q, kc, vc, tables, [n], 200.0)
    assert torch.allclose(out[0, 0], V[j, 0].double(), rtol=0, atol=1e-12)


def test_gqa_equals_mha_with_repeated_kv_heads():
    """Query head h reads KV head h // (Hq / Hkv): the same as MHA after
    repeating every KV head Hq / Hkv times in place."""
    lens = [19, 50]
    Hq, Hkv, hd = 8, 2, 64
    q, K, V = rand_case(12, lens, Hq, Hkv, hd, torch.float32)
    perm = np.random.default_rng(1).permutation(10)
    kc, vc, tables = place_contiguous(K, V, 16, 10, perm, torch.float32)
    gqa = run_oracle(q, kc, vc, tables, lens, 0.125)
    Kr = [k.repeat_interleave(Hq // Hkv, dim=1) for k in K]
    Vr = [v.repeat_interleave(Hq // Hkv, dim=1) for v in V]
    kc2, vc2, tables2 = place_contiguous(Kr, Vr, 16, 10, perm, torch.float32)
    mha = run_oracle(q, kc2, vc2, tables2, lens, 0.125)
    assert torch.equal(gqa, mha)


def test_empty_context_gives_zero_output():
    q, K, V = rand_case(13, [1], 2, 2, 64, torch.float32)
    kc, vc, tables = place_contiguous(K, V, 16, 1, np.array([0]), torch.float32)
    out = run_oracle(q, kc, vc, tables, [0], 0.125)
    assert torch.equal(out, torch.zeros_like(out))


def test_bf16_cache_is_widened_exactly():
    lens = [21, 48]
    q, K, V = rand_case(14, lens, 4, 2, 128, torch.bfloat16)
    perm = np.arange(4)
    kc, vc, tables = place_contiguous(K, V, 32, 4, perm, torch.bfloat16)
    a = run_oracle(q, kc, vc, tables, lens, 0.09)
    b = run_oracle(q, kc.float(), vc.float(), tables, lens, 0.09)
    assert torch.equal(a, b)


def test_pair_selection_matches_full_run():
    lens = [10, 33, 70]
    q, K, V = rand_case(15, lens, 4, 2, 64, torch.float32)
    kc, vc, tables = place_contiguous(K, V, 16, 9, np.random.default_rng(2).permutation(9),
                                      torch.float32)
    full = run_oracle(q, kc, vc, tables, lens, 0.125)
    pairs = torch.tensor([[2, 3], [0, 1], [1, 0]], dtype=torch.int32)
    part = oracle.paged_decode(q, kc, vc, tables, torch.tensor(lens, dtype=torch.int32), 0.125,
                               pairs=pairs, threads=1)
    for i, h in pairs.tolist():
        assert torch.equal(part[i, h], full[i, h])
    assert torch.isnan(part[2, 0]).all()


def test_out_of_range_block_id_is_an_error():
    q, K, V = rand_case(16, [20], 2, 2, 64, torch.float32)
    kc, vc, tables = place_contiguous(K, V, 16, 2, np.array([0, 1]), torch.float32)
    tables[0, 1] = 7
    with pytest.raises(ValueError):
        run_oracle(q, kc, vc, tables, [20], 0.125)


# ------------------------------------------------- cache write / copy -------
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_reshape_and_cache_matches_index_assignment(dtype):
    nb, H, bs, hd, T = 6, 3, 16, 64, 9
    g = torch.Generator().manual_seed(21)
    kc = torch.randn(nb, H, bs, hd, generator=g).to(dtype)
    vc = torch.randn(nb, H, bs, hd, generator=g).to(dtype)
    k = torch.randn(T, H, hd, generator=g).to(dtype)
    v = torch.randn(T, H, hd, generator=g).to(dtype)
    slots = np.random.default_rng(3).choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[4] = -1   # padding token
    ek, ev = kc.clone(), vc.clone()
    for t, s in enumerate(slots):
        if s >= 0:
            ek[s // bs, :, s % bs, :] = k[t]
            ev[s // bs, :, s % bs, :] = v[t]
    oracle.reshape_and_cache(k, v, kc, vc, torch.from_numpy(slots))
    assert torch.equal(kc.view(torch.int16 if dtype == torch.bfloat16 else torch.int32),
                       ek.view(torch.int16 if dtype == torch.bfloat16 else torch.int32))
    assert torch.equal(vc, ev)


def test_reshape_and_cache_rejects_slot_past_pool():
    kc = torch.zeros(2, 1, 16, 64)
    with pytest.raises(ValueError):
        oracle.reshape_and_cache(torch.ones(1, 1, 64), torch.ones(1, 1, 64), kc, kc.clone(),
                                 torch.tensor([32]))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_copy_blocks_matches_block_assignment(dtype):
    nb, H, bs, hd = 10, 2, 32, 64
    g = torch.Generator().manual_seed(22)
    kc = torch.randn(nb, H, bs, hd, generator=g).to(dtype)
    vc = torch.randn(nb, H, bs, hd, generator=g).to(dtype)
    pairs = torch.tensor([[1, 7], [3, 2], [1, 9]], dtype=torch.int64)
    ek, ev = kc.clone(), vc.clone()
    for s, d in pairs.tolist():
        ek[d] = kc[s]
        ev[d] = vc[s]
    oracle.copy_blocks(kc, vc, pairs)
    assert torch.equal(kc, ek) and torch.equal(vc, ev)


def test_copy_blocks_rejects_out_of_range_pair():
    kc = torch.zeros(2, 1, 16, 64)
    with pytest.raises(ValueError):
        oracle.copy_blocks(kc, kc.clone(), torch.tensor([[0, 2]], dtype=torch.int64))
