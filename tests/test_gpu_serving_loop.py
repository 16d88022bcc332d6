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
    return t.view(torch.int16)


def test_multi_step_serving_loop_matches_the_oracle():
    from paged_kv_cache_237_gb300 import binding
    from paged_kv_cache_237_gb300.engine import DecodeStep
    rng = np.random.default_rng(17)
    nb, bs, Hq, Hkv, hd, scale = 400, 16, 16, 2, 128, 0.09
    g = torch.Generator().manual_seed(17)
    kc_h = torch.randn(nb, Hkv, bs, hd, generator=g).to(torch.bfloat16)     # arbitrary prompt K/V
    vc_h = torch.randn(nb, Hkv, bs, hd, generator=g).to(torch.bfloat16)
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
        q = torch.randn(len(seqs), Hq, hd, generator=g).to(torch.bfloat16)
        kn = torch.randn(len(seqs), Hkv, hd, generator=g).to(torch.bfloat16)
        vn = torch.randn(len(seqs), Hkv, hd, generator=g).to(torch.bfloat16)
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
        assert_decode_close(out, ref, torch.bfloat16, what=f"serving step {step}")
    assert torch.equal(bits(kc.cpu()), bits(kc_h)) and torch.equal(bits(vc.cpu()), bits(vc_h))
