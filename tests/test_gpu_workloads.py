"""The five synthetic workloads, run as one decode step on the GPU and
compared with the fp64 oracle: whole outputs for the four that the oracle
finishes in seconds, sampled sequences (all heads) at full size for the
long-context batch, in the same launch configuration the benchmark times."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_decode_close, compact_for_oracle, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    from paged_kv_cache_237_gb300 import binding, engine, workloads
    return binding, engine, workloads


def bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def step_and_check(pa, name, full=True, **kw):
    binding, engine, workloads = pa
    d = workloads.decode_inputs(name, device="cuda", **kw)
    w = d["workload"]
    step = engine.DecodeStep(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                             d["scale"], d["max_context_len"], w.partition_size)
    kc_before = d["k_cache"].cpu() if full else None
    vc_before = d["v_cache"].cpu() if full else None
    out = step.run(d["k_new"], d["v_new"], d["slot_mapping"])
    torch.cuda.synchronize()
    assert step.status.read() == 0
    return d, step, out, kc_before, vc_before


def test_tiny_f32_step(pa):
    d, step, out, kc0, vc0 = step_and_check(pa, "tiny_f32")
    # cache writes: bit-exact against the oracle's host write
    oracle.reshape_and_cache(d["k_new"].cpu(), d["v_new"].cpu(), kc0, vc0, d["slot_mapping"].cpu())
    assert torch.equal(bits(d["k_cache"].cpu()), bits(kc0))
    assert torch.equal(bits(d["v_cache"].cpu()), bits(vc0))
    ref = oracle_decode(d["q"], kc0, vc0, d["block_tables"], d["context_lens"], d["scale"])
    assert_decode_close(out, ref, torch.float32, what="tiny_f32")


@pytest.mark.parametrize("name,kw", [("mha_llama2_7b", {}), ("gqa_llama3_70b", {}),
                                     ("gqa_llama3_70b", {"gqa_sigma": 0.5})])
def test_bf16_workload_step_full_parity(pa, name, kw):
    d, step, out, kc0, vc0 = step_and_check(pa, name, **kw)
    oracle.reshape_and_cache(d["k_new"].cpu(), d["v_new"].cpu(), kc0, vc0, d["slot_mapping"].cpu())
    assert torch.equal(bits(d["k_cache"].cpu()), bits(kc0))
    ref = oracle_decode(d["q"], kc0, vc0, d["block_tables"], d["context_lens"], d["scale"])
    assert_decode_close(out, ref, torch.bfloat16, what=name)


@pytest.mark.parametrize("name", ["mha_llama2_7b_f32", "gqa_llama3_70b_f32"])
def test_f32_workload_step_full_parity(pa, name):
    """The MHA and GQA batches in fp32 (the fp32-FMA pass): every output within
    1e-5 of the oracle, the cache write bit-exact, and the fused write (the
    launch the benchmark times) bit-identical to write-then-decode."""
    binding, engine, workloads = pa
    d, step, out, kc0, vc0 = step_and_check(pa, name)
    oracle.reshape_and_cache(d["k_new"].cpu(), d["v_new"].cpu(), kc0, vc0, d["slot_mapping"].cpu())
    assert torch.equal(bits(d["k_cache"].cpu()), bits(kc0))
    assert torch.equal(bits(d["v_cache"].cpu()), bits(vc0))
    ref = oracle_decode(d["q"], kc0, vc0, d["block_tables"], d["context_lens"], d["scale"])
    assert_decode_close(out, ref, torch.float32, what=name)
    first = out.clone()
    d2 = workloads.decode_inputs(name, device="cuda")
    w = d2["workload"]
    step2 = engine.DecodeStep(d2["q"], d2["k_cache"], d2["v_cache"], d2["block_tables"], d2["context_lens"],
                              d2["scale"], d2["max_context_len"], w.partition_size)
    fused = step2.run_fused(d2["k_new"], d2["v_new"], d2["slot_mapping"])
    torch.cuda.synchronize()
    assert step2.status.read() == 0
    assert torch.equal(bits(fused), bits(first))
    assert torch.equal(bits(d2["k_cache"]), bits(d["k_cache"]))


def test_prefix_share_step_with_copy_on_write(pa):
    binding, engine, _ = pa
    st = engine.prefix_share_state("cuda")
    bm = st["block_manager"]
    assert all(bm.refcount(b) == 50 for b in st["prompt_blocks"])
    pairs = st["pairs"]
    suffix = st["lens"].numpy()[0::2] - 2049      # pair suffix length u
    assert len(pairs) == int(np.count_nonzero(suffix % 16)), "one copy per pair with a partial last block"
    kc0, vc0 = st["k_cache"].cpu(), st["v_cache"].cpu()
    tables = st["tables"].cuda()
    lens = st["lens"].cuda()
    step = engine.DecodeStep(st["q"], st["k_cache"], st["v_cache"], tables, lens, st["scale"],
                             st["max_context_len"])
    out = step.run(st["k_new"], st["v_new"], st["slots"].cuda(), st["pairs"].cuda())
    torch.cuda.synchronize()
    assert step.status.read() == 0
    oracle.copy_blocks(kc0, vc0, pairs)
    oracle.reshape_and_cache(st["k_new"].cpu(), st["v_new"].cpu(), kc0, vc0, st["slots"])
    assert torch.equal(bits(st["k_cache"].cpu()), bits(kc0))
    assert torch.equal(bits(st["v_cache"].cpu()), bits(vc0))
    ref = oracle_decode(st["q"], kc0, vc0, st["tables"], st["lens"], st["scale"])
    assert_decode_close(out, ref, torch.bfloat16, what="prefix_share")


def test_long_context_full_size_sampled(pa):
    """Full 256-sequence batch (8 x 131072 + 248 mixed), bs 32, partitions of
    512; the oracle checks every head of 10 sampled sequences, including two
    of the 131072-token ones and the shortest one."""
    binding, engine, workloads = pa
    d = workloads.decode_inputs("long_context", device="cuda")
    w = d["workload"]
    step = engine.DecodeStep(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                             d["scale"], d["max_context_len"], w.partition_size)
    out_sep = step.run(d["k_new"], d["v_new"], d["slot_mapping"]).clone()
    torch.cuda.synchronize()
    assert step.status.read() == 0
    # the benchmark's step: one decode launch that also writes the new tokens
    out = step.run_fused(d["k_new"], d["v_new"], d["slot_mapping"])
    torch.cuda.synchronize()
    assert step.status.read() == 0
    assert torch.equal(bits(out), bits(out_sep))
    lens = d["lens"]
    longs = [int(i) for i in np.flatnonzero(lens == 131072)[:2]]
    rng = np.random.default_rng(0)
    others = [int(i) for i in rng.choice(np.flatnonzero(lens < 131072), size=7, replace=False)]
    seqs = sorted(set(longs + others + [int(np.argmin(lens))]))
    kc, vc, tab, ln = compact_for_oracle(d["k_cache"], d["v_cache"], d["block_tables"],
                                         d["context_lens"], seqs)
    ref = oracle.paged_decode(d["q"][seqs].cpu(), kc, vc, tab, ln, d["scale"])
    assert_decode_close(out[seqs], ref, torch.bfloat16, what="long_context sample")
    # the step's cache writes landed: each sampled sequence's last token row equals k_new
    for s in seqs:
        slot = int(d["slot_mapping"][s])
        row = d["k_cache"][slot // w.block_size, :, slot % w.block_size, :]
        assert torch.equal(bits(row.cpu()), bits(d["k_new"][s].cpu()))
    del d, step, out
    torch.cuda.empty_cache()


def test_prefix_cached_batch_decodes_like_private_copies(pa):
    """Requests admitted through the chained-key prefix cache (two tenants, one
    system prompt each, salted) share their prompt blocks; one fused decode
    step over the shared tables matches the oracle."""
    binding, engine, workloads = pa
    rng = np.random.default_rng(5)
    bs, Hq, Hkv, hd = 16, 16, 2, 128
    systems = [rng.integers(0, 1000, size=600).tolist() for _ in range(2)]
    bm = binding.BlockManager(400, bs)
    reqs = []
    for sid in range(12):
        t = sid % 2
        toks = systems[t] + rng.integers(0, 1000, size=int(rng.integers(1, 60))).tolist()
        hit = bm.add_seq_cached(sid, toks, salt=t)
        assert hit == (0 if sid < 2 else 592)        # 37 full blocks of the 600-token prompt
        reqs.append(toks)
    seqs = list(range(12))
    slots, pairs = bm.append_slots(seqs)
    assert pairs.numel() == 0
    tables, lens = bm.build_tables(seqs, max(len(bm.block_table(s)) for s in seqs))
    g = torch.Generator().manual_seed(3)
    kc = torch.randn(400, Hkv, bs, hd, generator=g).to(torch.bfloat16)
    vc = torch.randn(400, Hkv, bs, hd, generator=g).to(torch.bfloat16)
    q = torch.randn(12, Hq, hd, generator=g).to(torch.bfloat16)
    kn = torch.randn(12, Hkv, hd, generator=g).to(torch.bfloat16)
    vn = torch.randn(12, Hkv, hd, generator=g).to(torch.bfloat16)
    step = engine.DecodeStep(q.cuda(), kc.cuda(), vc.cuda(), tables.cuda(), lens.cuda(), 0.09, int(lens.max()))
    out = step.run_fused(kn.cuda(), vn.cuda(), slots.cuda())
    torch.cuda.synchronize()
    assert step.status.read() == 0
    oracle.reshape_and_cache(kn, vn, kc, vc, slots)
    ref = oracle_decode(q, kc, vc, tables, lens, 0.09)
    assert_decode_close(out, ref, torch.bfloat16, what="prefix-cached batch")


def test_f32_longest_contexts_stay_within_1e5(pa):
    """fp32 at the long-context mix's longest length: two sequences of 131072
    tokens and one of 16, GQA 16/2, head_dim 128, block_size 32, partitions
    of 512 (256 partials per row merged), fused cache write; every output
    within 1e-5 of the oracle."""
    from helpers import make_case
    binding, engine, _ = pa
    lens = [131072, 16, 131072]
    Hq, Hkv, hd, bs = 16, 2, 128, 32
    q, kc, vc, tables, lens_t = make_case(lens, Hq, Hkv, hd, bs, torch.float32, seed=97, slack=4, nan_tails=False)
    tab = tables.cpu()
    slots = torch.tensor([int(tab[i, (n - 1) // bs]) * bs + (n - 1) % bs for i, n in enumerate(lens)],
                         dtype=torch.int64)
    g = torch.Generator().manual_seed(98)
    kn = torch.randn(3, Hkv, hd, generator=g)
    vn = torch.randn(3, Hkv, hd, generator=g)
    step = engine.DecodeStep(q, kc, vc, tables, lens_t, 1 / 128 ** 0.5, max(lens), 512)
    out = step.run_fused(kn.cuda(), vn.cuda(), slots.cuda())
    torch.cuda.synchronize()
    assert step.status.read() == 0
    ref = oracle_decode(q, kc, vc, tables, lens_t, 1 / 128 ** 0.5)    # caches already hold the new rows
    assert_decode_close(out, ref, torch.float32, what="fp32 131072-token sequences")
