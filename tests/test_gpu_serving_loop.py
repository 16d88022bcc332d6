"""Several decode steps driven by the host block manager, the way a serving
loop would: prefix-cached admission (two tenants), a fork mid-way (parallel
sampling, so the next step copies a shared partial block), frees, and a late
admission.  Each step: append a slot per live sequence, copy-on-write copies,
then one fused decode launch that writes every new token and attends.  The
oracle runs on a host copy of the caches, updated step by step with its own
cache write and block copy; every step's outputs must match, and the caches
must match bit for bit at the end."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_decode_close

pytestmark = pytest.mark.gpu


def bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_multi_step_serving_loop_matches_the_oracle(dtype):
    from paged_kv_cache_237_gb300 import binding
    from paged_kv_cache_237_gb300.engine import DecodeStep
    rng = np.random.default_rng(17)
    nb, bs, Hq, Hkv, hd, scale = 400, 16, 16, 2, 128, 0.09
    g = torch.Generator().manual_seed(17)
    kc_h = torch.randn(nb, Hkv, bs, hd, generator=g).to(dtype)     # arbitrary prompt K/V
    vc_h = torch.randn(nb, Hkv, bs, hd, generator=g).to(dtype)
    kc, vc = kc_h.cuda(), vc_h.cuda()
    bm = binding.BlockManager(nb, bs)
    prompts = {t: rng.integers(0, 30000, size=int(rng.integers(300, 700))).tolist() for t in range(2)}
    live, nxt = [], 0

    def admit(t):
        nonlocal nxt
        toks = prompts[t] + rng.integers(0, 30000, size=int(rng.integers(1, 80))).tolist()
        bm.add_seq_cached(nxt, toks, salt=t)
        live.append(nxt)
        nxt += 1

    for i in range(6):
        admit(i % 2)
    status = binding.DeviceStatus()
    for step in range(6):
        if step == 2:                                   # parallel sampling: two forks share partial blocks
            for par in live[:2]:
                bm.fork(par, nxt)
                live.append(nxt)
                nxt += 1
        if step == 4:                                   # one request ends, another arrives
            bm.free_seq(live.pop(1))
            admit(1)
        seqs = list(live)
        slots, pairs = bm.append_slots(seqs)
        tables, lens = bm.build_tables(seqs, max(len(bm.block_table(s)) for s in seqs))
        q = torch.randn(len(seqs), Hq, hd, generator=g).to(dtype)
        kn = torch.randn(len(seqs), Hkv, hd, generator=g).to(dtype)
        vn = torch.randn(len(seqs), Hkv, hd, generator=g).to(dtype)
        dstep = DecodeStep(q.cuda(), kc, vc, tables.cuda(), lens.cuda(), scale, int(lens.max()), 64,
                           status=status)
        out = dstep.run_fused(kn.cuda(), vn.cuda(), slots.cuda(), pairs.cuda() if pairs.numel() else None)
        torch.cuda.synchronize()
        assert status.read() == 0, f"step {step}"
        if step == 2:
            assert pairs.numel() > 0, "the forks should have triggered copy-on-write"
        if pairs.numel():
            oracle.copy_blocks(kc_h, vc_h, pairs)
        oracle.reshape_and_cache(kn, vn, kc_h, vc_h, slots)
        ref = oracle.paged_decode(q, kc_h, vc_h, tables, lens, scale)
        assert_decode_close(out, ref, dtype, what=f"serving step {step} {dtype}")
    assert torch.equal(bits(kc.cpu()), bits(kc_h)) and torch.equal(bits(vc.cpu()), bits(vc_h))


def test_serving_loop_with_a_sequence_swapped_out_and_back_in():
    """A sequence leaves the device mid-loop (its blocks moved to a pinned host
    pool with pa_swap_blocks), sits out two steps while its device blocks are
    reused, comes back into fresh device blocks, and decodes on: every step
    matches the oracle, and both pools match their host truth bit for bit."""
    from paged_kv_cache_237_gb300 import binding
    from paged_kv_cache_237_gb300.engine import DecodeStep
    rng = np.random.default_rng(23)
    nb, nb_host, bs, Hq, Hkv, hd, scale = 160, 64, 16, 16, 2, 128, 0.09
    g = torch.Generator().manual_seed(23)
    kc_h = torch.randn(nb, Hkv, bs, hd, generator=g).to(torch.bfloat16)
    vc_h = torch.randn(nb, Hkv, bs, hd, generator=g).to(torch.bfloat16)
    kc, vc = kc_h.cuda(), vc_h.cuda()
    hk = torch.zeros(nb_host, Hkv, bs, hd, dtype=torch.bfloat16).pin_memory()
    hv = torch.zeros(nb_host, Hkv, bs, hd, dtype=torch.bfloat16).pin_memory()
    hk_h, hv_h = hk.clone(), hv.clone()
    dev, host = binding.BlockManager(nb, bs), binding.BlockManager(nb_host, bs)
    prompt = rng.integers(0, 30000, size=400).tolist()
    live = []
    for sid in range(3):                               # prefix-cached: their prompt blocks are shared
        dev.add_seq_cached(sid, prompt + rng.integers(0, 30000, size=int(rng.integers(1, 40))).tolist(), salt=0)
        live.append(sid)
    for sid in (3, 4):                                 # private sequences: movable
        dev.add_seq(sid, int(rng.integers(100, 300)))
        live.append(sid)
    status = binding.DeviceStatus()
    moved = 4
    for step in range(7):
        if step == 2:                                  # swap out: device -> pinned host
            pairs = dev.move_seq(host, moved)
            binding.pa_swap_blocks(kc, vc, hk, hv, pairs.cuda(), status=status)
            oracle.swap_blocks(kc_h, vc_h, hk_h, hv_h, pairs)
            live.remove(moved)
        if step == 5:                                  # swap back in, to whatever device blocks are free
            pairs = host.move_seq(dev, moved)
            binding.pa_swap_blocks(hk, hv, kc, vc, pairs.cuda(), status=status)
            oracle.swap_blocks(hk_h, hv_h, kc_h, vc_h, pairs)
            live.append(moved)
        seqs = list(live)
        slots, cow = dev.append_slots(seqs)
        tables, lens = dev.build_tables(seqs, max(len(dev.block_table(s)) for s in seqs))
        q = torch.randn(len(seqs), Hq, hd, generator=g).to(torch.bfloat16)
        kn = torch.randn(len(seqs), Hkv, hd, generator=g).to(torch.bfloat16)
        vn = torch.randn(len(seqs), Hkv, hd, generator=g).to(torch.bfloat16)
        dstep = DecodeStep(q.cuda(), kc, vc, tables.cuda(), lens.cuda(), scale, int(lens.max()), 128,
                           status=status)
        out = dstep.run_fused(kn.cuda(), vn.cuda(), slots.cuda(), cow.cuda() if cow.numel() else None)
        torch.cuda.synchronize()
        assert status.read() == 0, f"step {step}"
        if cow.numel():
            oracle.copy_blocks(kc_h, vc_h, cow)
        oracle.reshape_and_cache(kn, vn, kc_h, vc_h, slots)
        ref = oracle.paged_decode(q, kc_h, vc_h, tables, lens, scale)
        assert_decode_close(out, ref, torch.bfloat16, what=f"swap loop step {step}")
    assert torch.equal(bits(kc.cpu()), bits(kc_h)) and torch.equal(bits(vc.cpu()), bits(vc_h))
    assert torch.equal(bits(hk), bits(hk_h)) and torch.equal(bits(hv), bits(hv_h))
