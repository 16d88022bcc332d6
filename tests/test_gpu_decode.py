"""pa_decode on the GPU against the fp64 oracle: edge cases, group sizes,
head dims, block sizes, split-K partitioning, NaN tails, status flags,
determinism and placement invariance."""
import math

import numpy as np
import pytest
import torch

from helpers import assert_decode_close, make_case, oracle_decode

pytestmark = pytest.mark.gpu

EDGE_LENS = [1, 15, 16, 17, 31, 32, 33, 100, 511, 512, 513, 1000, 2049]


@pytest.fixture(scope="module")
def pa():
    from paged_kv_cache_237_gb300 import binding
    return binding


def run(pa, q, kc, vc, tables, lens, scale, partition_size=0, status=None, max_ctx=None):
    out = torch.empty_like(q)
    max_ctx = int(lens.max().item()) if max_ctx is None else max_ctx
    pa.pa_decode(out, q, kc, vc, tables, lens, scale, max_context_len=max_ctx,
                 partition_size=partition_size, status=status)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("dtype,simt", [(torch.bfloat16, False), (torch.bfloat16, True), (torch.float32, False)])
@pytest.mark.parametrize("hd", [64, 128])
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (6, 3), (8, 2), (16, 2), (16, 1), (12, 4), (40, 2)])
def test_edge_lengths_match_oracle(pa, dtype, simt, hd, bs, Hq, Hkv):
    q, kc, vc, tables, lens = make_case(EDGE_LENS, Hq, Hkv, hd, bs, dtype, seed=hd + bs + Hq)
    scale = 1.0 / math.sqrt(hd)
    status = pa.DeviceStatus()
    out = torch.empty_like(q)
    pa.pa_decode(out, q, kc, vc, tables, lens, scale, max_context_len=int(lens.max().item()), status=status,
                 simt=simt)
    torch.cuda.synchronize()
    assert status.read() == 0
    ref = oracle_decode(q, kc, vc, tables, lens, scale)
    assert_decode_close(out, ref, dtype, what=f"{dtype} hd{hd} bs{bs} {Hq}/{Hkv}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("P", [16, 64, 512, 4096])
def test_partition_sizes_match_oracle(pa, dtype, P):
    lens = [1, 16, 17, 64, 65, 700, 4096, 5000]
    q, kc, vc, tables, lens_t = make_case(lens, 8, 1, 128, 16, dtype, seed=P)
    out = run(pa, q, kc, vc, tables, lens_t, 0.088, partition_size=P)
    ref = oracle_decode(q, kc, vc, tables, lens_t, 0.088)
    assert_decode_close(out, ref, dtype, what=f"P={P}")


def test_split_and_unsplit_agree(pa):
    lens = [3000, 4096, 77]
    q, kc, vc, tables, lens_t = make_case(lens, 8, 2, 128, 32, torch.bfloat16, seed=3)
    a = run(pa, q, kc, vc, tables, lens_t, 0.1, partition_size=128).double()
    b = run(pa, q, kc, vc, tables, lens_t, 0.1, partition_size=4096).double()
    assert_decode_close(a, b, torch.bfloat16, what="split vs unsplit")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_empty_context_and_zero_scale(pa, dtype):
    lens = [0, 5, 40, 0]
    q, kc, vc, tables, lens_t = make_case(lens, 4, 2, 64, 16, dtype, seed=9)
    out = run(pa, q, kc, vc, tables, lens_t, 0.125, max_ctx=64)
    assert torch.equal(out[0].float().cpu(), torch.zeros(4, 64))
    assert torch.equal(out[3].float().cpu(), torch.zeros(4, 64))
    out0 = run(pa, q, kc, vc, tables, lens_t, 0.0)
    ref0 = oracle_decode(q, kc, vc, tables, lens_t, 0.0)
    assert_decode_close(out0, ref0, dtype, what="scale 0")


def test_single_token_returns_value_row(pa):
    q, kc, vc, tables, lens = make_case([1, 1, 1], 8, 8, 128, 16, torch.float32, seed=2)
    out = run(pa, q, kc, vc, tables, lens, 0.3)
    for s in range(3):
        v0 = vc[tables[s, 0].long(), :, 0, :]
        assert torch.allclose(out[s], v0, rtol=0, atol=1e-6)


def test_outputs_are_deterministic_and_placement_invariant(pa):
    lens = [700, 1500, 33, 2048]
    q, kc, vc, tables, lens_t = make_case(lens, 16, 2, 128, 16, torch.bfloat16, seed=4, nan_tails=False)
    a = run(pa, q, kc, vc, tables, lens_t, 0.1)
    b = run(pa, q, kc, vc, tables, lens_t, 0.1)
    assert torch.equal(a, b)
    # move every block to a new physical id and rewrite the tables
    nb = kc.shape[0]
    perm = torch.from_numpy(np.random.default_rng(8).permutation(nb)).cuda()
    kc2 = torch.empty_like(kc)
    vc2 = torch.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    t2 = torch.where(tables >= 0, perm[tables.clamp(min=0).long()].int(), tables)
    c = run(pa, q, kc2, vc2, t2, lens_t, 0.1)
    assert torch.equal(a, c)


def test_bad_block_id_and_length_are_flagged_not_faulted(pa):
    lens = [40, 40, 40]
    q, kc, vc, tables, lens_t = make_case(lens, 8, 2, 128, 16, torch.bfloat16, seed=5)
    good = run(pa, q, kc, vc, tables, lens_t, 0.1)
    bad = tables.clone()
    bad[1, 1] = kc.shape[0] + 1000          # outside the pool
    bad[2, 0] = -5
    status = pa.DeviceStatus()
    out = run(pa, q, kc, vc, bad, lens_t, 0.1, status=status)
    assert status.read() & pa.STATUS_BAD_BLOCK_ID
    assert torch.equal(out[0], good[0])
    long_lens = lens_t.clone()
    long_lens[0] = 10_000                   # beyond the 3-entry table row
    out = run(pa, q, kc, vc, tables, long_lens, 0.1, status=status, max_ctx=10_000)
    assert status.read() & pa.STATUS_BAD_CONTEXT_LEN
    assert torch.equal(out[1], good[1])


def test_bad_block_id_fp32_path_is_flagged(pa):
    q, kc, vc, tables, lens_t = make_case([20, 20], 4, 4, 64, 16, torch.float32, seed=6)
    bad = tables.clone()
    bad[0, 1] = 1 << 20
    status = pa.DeviceStatus()
    out = run(pa, q, kc, vc, bad, lens_t, 0.1, status=status)
    assert status.read() & pa.STATUS_BAD_BLOCK_ID
    ref = oracle_decode(q, kc, vc, tables, lens_t, 0.1)
    assert_decode_close(out[1:], ref[1:], torch.float32)


def test_large_batch_many_items(pa):
    """More work items than one persistent wave, mixed lengths, GQA 8."""
    rng = np.random.default_rng(12)
    lens = rng.integers(1, 3000, size=96).tolist()
    q, kc, vc, tables, lens_t = make_case(lens, 32, 4, 128, 16, torch.bfloat16, seed=12)
    out = run(pa, q, kc, vc, tables, lens_t, 1 / math.sqrt(128), partition_size=256)
    ref = oracle_decode(q, kc, vc, tables, lens_t, 1 / math.sqrt(128))
    assert_decode_close(out, ref, torch.bfloat16, what="96 seqs")


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


@pytest.mark.parametrize("dtype,simt", [(torch.bfloat16, False), (torch.bfloat16, True), (torch.float32, False)])
@pytest.mark.parametrize("hd,bs,Hq,Hkv", [(128, 16, 8, 1), (64, 32, 40, 2), (128, 32, 32, 8)])
def test_fused_cache_write_matches_write_then_decode(pa, dtype, simt, hd, bs, Hq, Hkv):
    """One launch that writes each sequence's new token and attends with it gives
    bit-identical outputs and caches to pa_reshape_and_cache then pa_decode.
    Sequence 2 is padding (slot -1): neither path writes it."""
    lens = [1, 16, 17, 40, 513, 1025, 2000]
    q, kc, vc, tables, lens_t = make_case(lens, Hq, Hkv, hd, bs, dtype, seed=31 + hd + Hq)
    S = len(lens)
    g = torch.Generator().manual_seed(5)
    k_new = torch.randn(S, Hkv, hd, generator=g).to(dtype).cuda()
    v_new = torch.randn(S, Hkv, hd, generator=g).to(dtype).cuda()
    tab = tables.cpu()
    slots = torch.tensor([int(tab[i, (n - 1) // bs]) * bs + (n - 1) % bs for i, n in enumerate(lens)],
                         dtype=torch.int64)
    slots[2] = -1
    slots = slots.cuda()
    kc_a, vc_a = kc.clone(), vc.clone()
    pa.pa_reshape_and_cache(k_new, v_new, kc_a, vc_a, slots)
    out_a = torch.empty_like(q)
    pa.pa_decode(out_a, q, kc_a, vc_a, tables, lens_t, 0.1, max_context_len=max(lens), partition_size=256,
                 simt=simt)
    status = pa.DeviceStatus()
    out_b = torch.empty_like(q)
    pa.pa_decode(out_b, q, kc, vc, tables, lens_t, 0.1, max_context_len=max(lens), partition_size=256,
                 status=status, k_new=k_new, v_new=v_new, slot_mapping=slots, simt=simt)
    torch.cuda.synchronize()
    assert status.read() == 0
    assert torch.equal(_bits(out_a), _bits(out_b))
    assert torch.equal(_bits(kc_a), _bits(kc)) and torch.equal(_bits(vc_a), _bits(vc))
    ref = oracle_decode(q, kc_a, vc_a, tables, lens_t, 0.1)
    assert_decode_close(out_b, ref, dtype, what="fused")


def test_fused_cache_write_rejects_a_slot_that_is_not_the_last_position(pa):
    lens = [40, 40]
    q, kc, vc, tables, lens_t = make_case(lens, 8, 2, 128, 16, torch.bfloat16, seed=3, nan_tails=False)
    k_new = torch.ones(2, 2, 128, dtype=torch.bfloat16, device="cuda")
    tab = tables.cpu()
    good = int(tab[0, 39 // 16]) * 16 + 39 % 16
    slots = torch.tensor([good, int(tab[1, 0]) * 16 + 3], dtype=torch.int64, device="cuda")  # seq 1: wrong slot
    before = kc.clone()
    status = pa.DeviceStatus()
    out = torch.empty_like(q)
    pa.pa_decode(out, q, kc, vc, tables, lens_t, 0.1, max_context_len=40, status=status,
                 k_new=k_new, v_new=k_new, slot_mapping=slots)
    torch.cuda.synchronize()
    assert status.read() & pa.STATUS_BAD_SLOT
    blk1 = tables[1].long()
    assert torch.equal(_bits(kc[blk1]), _bits(before[blk1]))        # nothing written for sequence 1
    assert kc[good // 16, :, good % 16].eq(1).all()                 # sequence 0 written
    plain = run(pa, q, kc, vc, tables, lens_t, 0.1)
    assert torch.equal(_bits(out[1]), _bits(plain[1]))


def test_thousands_of_short_sequences(pa):
    """3000 sequences of 0..300 tokens (many single-partition, some split with
    P = 128): the warp-parallel walk from work items to sequences stays exact
    far past one warp's 32 sequences per step."""
    rng = np.random.default_rng(77)
    lens = rng.integers(0, 301, size=3000).tolist()
    q, kc, vc, tables, lens_t = make_case(lens, 16, 2, 128, 16, torch.bfloat16, seed=77, slack=3)
    status = pa.DeviceStatus()
    out = run(pa, q, kc, vc, tables, lens_t, 0.1, partition_size=128, status=status)
    assert status.read() == 0
    sample = torch.from_numpy(np.stack([np.repeat(np.arange(0, 3000, 7), 2),
                                        np.tile([0, 15], len(range(0, 3000, 7)))], 1).astype(np.int32))
    import oracle
    ref = oracle.paged_decode(q.cpu(), kc.cpu(), vc.cpu(), tables.cpu(), lens_t.cpu(), 0.1, pairs=sample)
    mask = torch.zeros(q.shape[:2], dtype=torch.bool)
    mask[sample[:, 0].long(), sample[:, 1].long()] = True
    assert_decode_close(out, ref, torch.bfloat16, mask=mask, what="3000 sequences")


def test_step_captured_in_a_cuda_graph_replays_bit_identically(pa):
    """The decode step (fused cache write + both passes) captured once in a
    CUDA graph and replayed gives the same bits as launching it eagerly."""
    from paged_kv_cache_237_gb300.engine import DecodeStep
    lens = [40, 700, 1500, 5]
    q, kc, vc, tables, lens_t = make_case(lens, 16, 2, 128, 16, torch.bfloat16, seed=41, nan_tails=False)
    g = torch.Generator().manual_seed(41)
    kn = torch.randn(4, 2, 128, generator=g).to(torch.bfloat16).cuda()
    vn = torch.randn(4, 2, 128, generator=g).to(torch.bfloat16).cuda()
    tab = tables.cpu()
    slots = torch.tensor([int(tab[i, (n - 1) // 16]) * 16 + (n - 1) % 16 for i, n in enumerate(lens)],
                         dtype=torch.int64).cuda()
    step = DecodeStep(q, kc, vc, tables, lens_t, 0.1, max(lens), 256)
    eager = step.run_fused(kn, vn, slots).clone()
    torch.cuda.synchronize()
    step.out.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="relaxed"):
        step.run_fused(kn, vn, slots)
    for _ in range(3):
        step.out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(_bits(step.out), _bits(eager))
    assert step.status.read() == 0


def test_concurrent_first_calls_from_host_threads(pa):
    """Several host threads calling pa_decode at once, each on its own stream
    (the library's per-kernel launch settings are set up under a lock)."""
    import threading
    cases = [make_case([300 + 97 * i, 33, 1200], 8, 1, 64 if i % 2 else 128, 16 if i < 2 else 32,
                       torch.bfloat16, seed=50 + i) for i in range(4)]
    outs, errors = [None] * 4, []

    def work(i):
        try:
            q, kc, vc, tables, lens_t = cases[i]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                out = torch.empty_like(q)
                pa.pa_decode(out, q, kc, vc, tables, lens_t, 0.1, max_context_len=int(lens_t.max()),
                             partition_size=128, stream=s)
            s.synchronize()
            outs[i] = out
        except Exception as e:  # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i, (q, kc, vc, tables, lens_t) in enumerate(cases):
        ref = oracle_decode(q, kc, vc, tables, lens_t, 0.1)
        assert_decode_close(outs[i], ref, torch.bfloat16, what=f"thread {i}")


def test_workspace_contents_do_not_matter(pa):
    """The workspace may hold anything before a call: every partial is written
    before it is read, and the work counter of the partition pass is reset on
    the stream before the pass.  A workspace filled with 0xff bytes (NaN
    partials, a huge counter) gives the same bits as a zeroed one, and both
    match the oracle; so do later calls on it, with or without the reset.
    Every call leaves the counter (the workspace's first 8 bytes) at zero."""
    lens = [5000, 17, 2049, 4096, 600, 1]
    q, kc, vc, tables, lens_t = make_case(lens, 16, 2, 128, 16, torch.bfloat16, seed=21)
    max_ctx = int(lens_t.max().item())
    need = pa.pa_decode_workspace_size(len(lens), 16, 128, max_ctx, 256)
    assert need > 0
    zeroed = torch.zeros(need, dtype=torch.uint8, device="cuda")
    dirty = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    outs = []
    # the third call finds the second's contents; the fourth also skips the
    # counter reset, valid because every completed call leaves the counter zero
    for ws, skip in ((zeroed, False), (dirty, False), (dirty, False), (dirty, True)):
        out = torch.empty_like(q)
        status = pa.DeviceStatus()
        pa.pa_decode(out, q, kc, vc, tables, lens_t, 0.09, max_context_len=max_ctx, partition_size=256,
                     workspace=ws, status=status, skip_counter_reset=skip)
        torch.cuda.synchronize()
        assert status.read() == 0
        assert int(ws[:8].view(torch.int64).item()) == 0, "the work counter must be left at zero"
        outs.append(out)
    ref = oracle_decode(q, kc, vc, tables, lens_t, 0.09)
    assert_decode_close(outs[0], ref, torch.bfloat16, what="zeroed workspace")
    for out in outs[1:]:
        assert torch.equal(out.view(torch.int16), outs[0].view(torch.int16))


def test_work_counter_survives_phases_graphs_and_size_changes(pa):
    """The self-resetting work counter across the ways a workspace is reused:
    split phases, CUDA-graph replays, and calls of other sizes on the same
    buffer, all with the reset skipped after the first call."""
    lens = [3000, 700, 4096, 1, 513]
    q, kc, vc, tables, lens_t = make_case(lens, 8, 1, 128, 32, torch.bfloat16, seed=33)
    max_ctx = int(lens_t.max().item())
    ws = torch.zeros(pa.pa_decode_workspace_size(64, 64, 128, 8192, 128), dtype=torch.uint8, device="cuda")
    status = pa.DeviceStatus()
    ref = oracle_decode(q, kc, vc, tables, lens_t, 0.1)

    def call(out, phase=0, P=128, **kw):
        pa.pa_decode(out, q, kc, vc, tables, lens_t, 0.1, max_context_len=max_ctx, partition_size=P,
                     workspace=ws, status=status, phase=phase, skip_counter_reset=True, **kw)

    a = torch.empty_like(q)
    call(a)
    b = torch.empty_like(q)
    call(b, phase=pa.PA_PHASE_PARTITIONS)
    call(b, phase=pa.PA_PHASE_REDUCE)
    torch.cuda.synchronize()
    assert status.read() == 0 and int(ws[:8].view(torch.int64).item()) == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert_decode_close(a, ref, torch.bfloat16, what="skip reset")
    c = torch.empty_like(q)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(c)
    for _ in range(3):
        c.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(c.view(torch.int16), a.view(torch.int16))
    for P in (512, 16, 128):                       # other layouts of the partials, same counter word
        d = torch.empty_like(q)
        call(d, P=P)
        torch.cuda.synchronize()
        assert status.read() == 0 and int(ws[:8].view(torch.int64).item()) == 0
        assert_decode_close(d, ref, torch.bfloat16, what=f"P={P} after other sizes")


def test_loose_max_context_len_leaves_most_ctas_without_work(pa):
    """max_context_len far above the real lengths: the host's bound on work
    items (and so the grid) is much larger than the items that exist, so most
    CTAs find no item at all.  They must still report finishing, so the work
    counter is back at zero, and every row matches the oracle, call after
    call."""
    lens = [5, 700, 33, 1]
    width = 4096                                   # table room for 65,536 tokens at bs 16
    q, kc, vc, tables, lens_t = make_case(lens, 16, 2, 128, 16, torch.bfloat16, seed=41)
    wide = torch.full((len(lens), width), -1, dtype=torch.int32, device="cuda")
    wide[:, :tables.shape[1]] = tables
    max_ctx = 65536
    need = pa.pa_decode_workspace_size(len(lens), 16, 128, max_ctx, 512)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    ref = oracle_decode(q, kc, vc, tables, lens_t, 0.1)
    for skip in (False, True, True):
        out = torch.empty_like(q)
        status = pa.DeviceStatus()
        pa.pa_decode(out, q, kc, vc, wide, lens_t, 0.1, max_context_len=max_ctx, partition_size=512,
                     workspace=ws, status=status, skip_counter_reset=skip)
        torch.cuda.synchronize()
        assert status.read() == 0
        assert int(ws[:8].view(torch.int64).item()) == 0
        assert_decode_close(out, ref, torch.bfloat16, what=f"loose max_context_len, skip={skip}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_inputs_written_by_the_preceding_kernel_are_seen(pa, dtype):
    """The partition pass is a programmatic dependent launch: it may be
    scheduled while the kernel before it still runs, and must read nothing
    before its grid-dependency wait.  Ordinary device kernels rewrite q, the
    tables, the lengths and the caches right before each call (eagerly, then
    inside a CUDA graph); every output must be the oracle's on the new inputs."""
    from paged_kv_cache_237_gb300.engine import DecodeStep
    Hq, Hkv, hd, bs = 16, 2, 128, 16
    cases = [make_case(lens, Hq, Hkv, hd, bs, dtype, seed=60 + i, slack=3, nan_tails=False)
             for i, lens in enumerate(([900, 33, 2100], [1500, 640, 17], [5, 2047, 1200]))]
    nb = max(c[1].shape[0] for c in cases)
    width = max(c[3].shape[1] for c in cases)
    # one set of device buffers, large enough for every case
    q = torch.zeros_like(cases[0][0])
    kc = torch.zeros(nb, Hkv, bs, hd, dtype=dtype, device="cuda")
    vc = torch.zeros_like(kc)
    tables = torch.full((3, width), -1, dtype=torch.int32, device="cuda")
    lens_t = torch.zeros(3, dtype=torch.int32, device="cuda")
    step = DecodeStep(q, kc, vc, tables, lens_t, 1 / math.sqrt(hd), 2100, 256)

    def load(case):
        cq, ckc, cvc, ct, cl = case
        q.copy_(cq)                      # device-to-device copy kernels, enqueued just before the call
        kc[: ckc.shape[0]].copy_(ckc)
        vc[: cvc.shape[0]].copy_(cvc)
        tables.fill_(-1)
        tables[:, : ct.shape[1]].copy_(ct)
        lens_t.copy_(cl)

    def check(case, out, what):
        cq, ckc, cvc, ct, cl = case
        assert_decode_close(out, oracle_decode(cq, ckc, cvc, ct, cl, 1 / math.sqrt(hd)), dtype, what=what)

    for i, case in enumerate(cases):          # eager: each call right after the copies
        load(case)
        out = step.decode().clone()
        check(case, out, f"eager case {i}")
    graphs = []
    for case in cases:                        # the copies and the call captured together
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            load(case)
            step.decode()
        graphs.append(g)
    for rep in range(2):
        for i, (case, g) in enumerate(zip(cases, graphs)):
            g.replay()
            check(case, step.out.clone(), f"graph case {i}, replay {rep}")
    torch.cuda.synchronize()
    assert step.status.read() == 0
