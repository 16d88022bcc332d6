"""Swapping sequences between a device pool and a host pool: the library's
pa_bm_move_seq against the model (id for id), the oracle's pool-to-pool copy
against numpy, and (GPU) pa_swap_blocks between device memory and pinned host
memory, bit-exact against the oracle ("PagedAttention" concept sheet,
analyticslegends.ai, "Points cles" and "Termes employes sur cette page": cold
pages are written to CPU RAM and read back on demand)."""
import numpy as np
import pytest
import torch

import oracle
from oracle.block_manager_ref import BlockManagerModel, NoBlocks
from paged_kv_cache_237_gb300 import build as pa_build


@pytest.fixture(scope="module")
def binding():
    pa_build.build()
    from paged_kv_cache_237_gb300 import binding
    return binding


def test_oracle_swap_matches_numpy():
    g = torch.Generator().manual_seed(1)
    src_k = torch.randn(6, 2, 16, 64, generator=g)
    src_v = torch.randn(6, 2, 16, 64, generator=g)
    dst_k = torch.zeros(9, 2, 16, 64)
    dst_v = torch.zeros(9, 2, 16, 64)
    pairs = torch.tensor([[0, 8], [5, 1], [2, 2]])
    ek, ev = dst_k.clone(), dst_v.clone()
    for s, d in pairs.tolist():
        ek[d], ev[d] = src_k[s], src_v[s]
    oracle.swap_blocks(src_k, src_v, dst_k, dst_v, pairs)
    assert torch.equal(dst_k, ek) and torch.equal(dst_v, ev)
    with pytest.raises(ValueError):
        oracle.swap_blocks(src_k, src_v, dst_k, dst_v, torch.tensor([[6, 0]]))


@pytest.mark.parametrize("seed", [0, 1])
def test_move_seq_matches_model(binding, seed):
    rng = np.random.default_rng(seed)
    dev, host = binding.BlockManager(40, 16), binding.BlockManager(60, 16)
    mdev, mhost = BlockManagerModel(40, 16), BlockManagerModel(60, 16)
    where = {}
    for sid in range(12):
        n = int(rng.integers(1, 90))
        try:
            mdev.add_seq(sid, n)
        except NoBlocks:
            continue
        dev.add_seq(sid, n)
        where[sid] = "dev"
    for _ in range(60):
        sid = int(rng.choice(list(where)))
        src, dst, msrc, mdst = (dev, host, mdev, mhost) if where[sid] == "dev" else (host, dev, mhost, mdev)
        try:
            expect = msrc.move_seq(mdst, sid)
        except NoBlocks:
            with pytest.raises(binding.PAError) as e:
                src.move_seq(dst, sid)
            assert e.value.code == binding.PA_ERR_NO_BLOCKS
            continue
        got = src.move_seq(dst, sid)
        assert got.tolist() == [list(p) for p in expect]
        where[sid] = "host" if where[sid] == "dev" else "dev"
        assert dev.num_free() == mdev.num_free() and host.num_free() == mhost.num_free()
        for s, w in where.items():
            assert (dev if w == "dev" else host).block_table(s) == (mdev if w == "dev" else mhost).block_table(s)


def test_move_seq_refuses_shared_blocks(binding):
    dev, host = binding.BlockManager(10, 16), binding.BlockManager(10, 16)
    dev.add_seq(0, 40)
    dev.fork(0, 1)
    with pytest.raises(binding.PAError) as e:
        dev.move_seq(host, 0)
    assert e.value.code == binding.PA_ERR_REFCOUNT
    assert host.num_free() == 10 and dev.block_table(0) == [0, 1, 2]


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_swap_out_and_in_through_pinned_host_memory(binding, dtype):
    nb_dev, nb_host, Hkv, bs, hd = 48, 64, 8, 32, 128
    g = torch.Generator().manual_seed(4)
    dk = torch.randn(nb_dev, Hkv, bs, hd, generator=g).to(dtype).cuda()
    dv = torch.randn(nb_dev, Hkv, bs, hd, generator=g).to(dtype).cuda()
    hk = torch.zeros(nb_host, Hkv, bs, hd, dtype=dtype).pin_memory()
    hv = torch.zeros(nb_host, Hkv, bs, hd, dtype=dtype).pin_memory()
    out_pairs = torch.tensor([[3, 60], [17, 0], [47, 31], [0, 5]], dtype=torch.int64)
    ref_hk, ref_hv = hk.clone(), hv.clone()
    oracle.swap_blocks(dk.cpu(), dv.cpu(), ref_hk, ref_hv, out_pairs)
    status = binding.DeviceStatus()
    binding.pa_swap_blocks(dk, dv, hk, hv, out_pairs.cuda(), status=status)       # device -> host
    torch.cuda.synchronize()
    assert status.read() == 0
    assert torch.equal(hk.view(torch.uint8), ref_hk.view(torch.uint8))
    assert torch.equal(hv.view(torch.uint8), ref_hv.view(torch.uint8))
    # back in to other device blocks, pairs in pinned host memory
    in_pairs = torch.tensor([[60, 10], [0, 11], [31, 12], [5, 13]], dtype=torch.int64).pin_memory()
    ref_dk, ref_dv = dk.cpu(), dv.cpu()
    oracle.swap_blocks(hk, hv, ref_dk, ref_dv, in_pairs)
    binding.pa_swap_blocks(hk, hv, dk, dv, in_pairs, status=status)              # host -> device
    torch.cuda.synchronize()
    assert status.read() == 0
    assert torch.equal(dk.cpu().view(torch.uint8), ref_dk.view(torch.uint8))
    assert torch.equal(dv.cpu().view(torch.uint8), ref_dv.view(torch.uint8))


@pytest.mark.gpu
def test_swap_rejects_pageable_memory_and_flags_bad_pairs(binding):
    dk = torch.zeros(4, 1, 16, 64, device="cuda")
    hk = torch.zeros(4, 1, 16, 64)            # pageable
    with pytest.raises(ValueError):
        binding.pa_swap_blocks(dk, dk.clone(), hk, hk.clone(), torch.tensor([[0, 0]]).cuda())
    # the C ABI refuses it too (checked with cudaPointerGetAttributes)
    import ctypes
    rc = binding._lib.pa_swap_blocks(dk.data_ptr(), dk.data_ptr() + 4096 * 4, hk.data_ptr(),
                                     hk.data_ptr() + 4096 * 4, torch.tensor([[0, 0]]).cuda().data_ptr(), 1, 4, 4,
                                     1, 64, 16, binding.PA_F32, None, None)
    assert rc == binding.PA_ERR_INVALID_ARG
    pk = torch.zeros(4, 1, 16, 64).pin_memory()
    pv = torch.zeros(4, 1, 16, 64).pin_memory()
    status = binding.DeviceStatus()
    binding.pa_swap_blocks(dk, dk.clone(), pk, pv, torch.tensor([[0, 9], [1, 2], [3, 2]]).cuda(), status=status)
    torch.cuda.synchronize()
    assert status.read() & binding.STATUS_BAD_PAIR
