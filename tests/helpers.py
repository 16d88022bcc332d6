"""Shared helpers for the GPU parity tests: oracle calls on CPU copies and the
comparison rules.

Tolerances: fp32 inputs, max |out - ref| <= 1e-5; bf16 inputs (fp32
accumulation), every element |out - ref| <= 2e-3 + 1e-2 |ref|.  Cache writes
and block copies are compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

F32_ATOL = 1e-5
BF16_ATOL, BF16_RTOL = 2e-3, 1e-2


def assert_decode_close(out: torch.Tensor, ref: torch.Tensor, dtype: torch.dtype, mask=None, what=""):
    o = out.detach().double().cpu()
    r = ref.double().cpu()
    if mask is not None:
        o, r = o[mask], r[mask]
    assert torch.isfinite(o).all(), f"{what}: non-finite output"
    err = (o - r).abs()
    if dtype == torch.float32:
        worst = err.max().item() if err.numel() else 0.0
        assert worst <= F32_ATOL, f"{what}: max abs err {worst:.3e} > {F32_ATOL}"
    else:
        tol = BF16_ATOL + BF16_RTOL * r.abs()
        bad = err > tol
        if bad.any():
            i = torch.nonzero(bad)[0].tolist()
            raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance, first at {i}: "
                                 f"out {o[tuple(i)].item():.6f} ref {r[tuple(i)].item():.6f}; "
                                 f"max abs {err.max().item():.3e}")


def oracle_decode(q, k_cache, v_cache, tables, lens, scale, pairs=None):
    """Run the oracle on CPU copies of (possibly CUDA) tensors."""
    return oracle.paged_decode(q.detach().cpu(), k_cache.detach().cpu(), v_cache.detach().cpu(),
                               tables.detach().cpu().to(torch.int32), lens.detach().cpu().to(torch.int32),
                               scale, pairs=pairs)


def compact_for_oracle(k_cache, v_cache, tables, lens, seqs):
    """Copy only the blocks that the listed sequences use to the host.

    Returns (k_cpu, v_cpu, tables_cpu, lens_cpu) for a batch made of `seqs`,
    with the block ids renumbered into the compact pool.  The gather happens
    with torch indexing on the device (test plumbing, not the product path).
    """
    bs = k_cache.shape[2]
    lens_h = lens.detach().cpu().numpy()
    tab_h = tables.detach().cpu().numpy()
    ids, rows = [], []
    for s in seqs:
        nb = -(-int(lens_h[s]) // bs)
        rows.append(tab_h[s, :nb])
        ids.extend(tab_h[s, :nb].tolist())
    uniq = np.unique(np.array(ids, dtype=np.int64)) if ids else np.zeros(0, np.int64)
    remap = {int(b): i for i, b in enumerate(uniq)}
    idx = torch.from_numpy(uniq).to(k_cache.device)
    kc = k_cache.index_select(0, idx).cpu() if len(uniq) else k_cache[:1].cpu()
    vc = v_cache.index_select(0, idx).cpu() if len(uniq) else v_cache[:1].cpu()
    width = max(1, max(len(r) for r in rows))
    t = np.full((len(seqs), width), -1, dtype=np.int32)
    for i, r in enumerate(rows):
        t[i, :len(r)] = [remap[int(b)] for b in r]
    return kc, vc, torch.from_numpy(t), torch.from_numpy(lens_h[list(seqs)].astype(np.int32))


def fill_tails_with_nan(k_cache, v_cache, tables, lens):
    """Write NaN into every slot at or past each sequence's length in its last
    block, so any read of a masked slot would poison the output."""
    bs = k_cache.shape[2]
    tab = tables.cpu().numpy()
    for s, n in enumerate(lens.cpu().numpy().tolist()):
        if n % bs == 0:
            continue
        blk = int(tab[s, n // bs])
        k_cache[blk, :, n % bs:, :] = float("nan")
        v_cache[blk, :, n % bs:, :] = float("nan")


def make_case(lens, Hq, Hkv, hd, bs, dtype, seed, device="cuda", slack=7, nan_tails=True):
    """Random paged batch: shuffled physical placement, N(0, 1) values."""
    rng = np.random.default_rng(seed)
    per = [max(1, -(-n // bs)) for n in lens]
    nb = sum(per) + slack
    perm = rng.permutation(nb)
    width = max(per)
    tables = np.full((len(lens), width), -1, dtype=np.int32)
    pos = 0
    for i, k in enumerate(per):
        tables[i, :k] = perm[pos:pos + k]
        pos += k
    g = torch.Generator(device="cpu").manual_seed(seed)
    k_cache = torch.randn(nb, Hkv, bs, hd, generator=g).to(dtype).to(device)
    v_cache = torch.randn(nb, Hkv, bs, hd, generator=g).to(dtype).to(device)
    q = torch.randn(len(lens), Hq, hd, generator=g).to(dtype).to(device)
    tables_t = torch.from_numpy(tables).to(device)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=device)
    if nan_tails:
        fill_tails_with_nan(k_cache, v_cache, tables_t, lens_t)
    return q, k_cache, v_cache, tables_t, lens_t
