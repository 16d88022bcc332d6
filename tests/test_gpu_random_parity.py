"""Seeded random sweep of pa_decode configurations against the fp64 oracle:
dtype, head_dim, block size, group size (1..40, several head tiles), partition
size, lengths (0, 1, block edges, long), block placement, NaN tails, fused or
separate cache write, tensor-core or SIMT products for bf16.  Every case must meet the tolerance and leave the
status word clear."""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_decode_close, make_case, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    from paged_kv_cache_237_gb300 import binding
    return binding


def draw(rng, fma_pass=False):
    """One configuration; fma_pass draws only cases of the fp32-FMA pass (fp32
    inputs, or bf16 with simt)."""
    dtype = torch.bfloat16 if rng.random() < 0.75 else torch.float32
    if fma_pass:
        dtype = torch.float32 if rng.random() < 0.7 else torch.bfloat16
    hd = int(rng.choice([64, 128]))
    bs = int(rng.choice([16, 32]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    group = int(rng.choice([1, 2, 3, 4, 5, 8, 12, 16, 20, 40]))
    P = int(rng.choice([0, 16, 48, 128, 512, 4096]))
    S = int(rng.integers(1, 9))
    lens = []
    for _ in range(S):
        r = rng.random()
        if r < 0.08:
            lens.append(0)
        elif r < 0.3:
            lens.append(int(rng.choice([1, bs - 1, bs, bs + 1, 2 * bs])))
        else:
            lens.append(int(rng.integers(1, 3000)))
    fused = bool(rng.random() < 0.5)
    simt = dtype == torch.bfloat16 and (fma_pass or bool(rng.random() < 0.3))
    return dtype, hd, bs, Hkv, group * Hkv, P, lens, fused, simt


@pytest.mark.parametrize("seed", range(40))
def test_random_configuration_matches_oracle(pa, seed):
    check_random_case(pa, seed, np.random.default_rng(1000 + seed), fma_pass=False)


@pytest.mark.parametrize("seed", range(24))
def test_random_fma_pass_configuration_matches_oracle(pa, seed):
    """The same sweep restricted to the fp32-FMA pass (head tiles of 1, 2, 4
    and 8 query heads, both head_dims, packed-FMA products)."""
    check_random_case(pa, 500 + seed, np.random.default_rng(5000 + seed), fma_pass=True)


def check_random_case(pa, seed, rng, fma_pass):
    dtype, hd, bs, Hkv, Hq, P, lens, fused, simt = draw(rng, fma_pass)
    q, kc, vc, tables, lens_t = make_case(lens, Hq, Hkv, hd, bs, dtype, seed=seed, slack=int(rng.integers(0, 9)))
    scale = float(rng.uniform(0.02, 0.2)) if rng.random() < 0.9 else 1.0 / math.sqrt(hd)
    max_ctx = max(lens) if max(lens) > 0 else 1
    status = pa.DeviceStatus()
    out = torch.empty_like(q)
    S = len(lens)
    if fused and max(lens) > 0:
        g = torch.Generator().manual_seed(seed)
        k_new = torch.randn(S, Hkv, hd, generator=g).to(dtype)
        v_new = torch.randn(S, Hkv, hd, generator=g).to(dtype)
        tab = tables.cpu()
        slots = torch.tensor([int(tab[i, (n - 1) // bs]) * bs + (n - 1) % bs if n > 0 else -1
                              for i, n in enumerate(lens)], dtype=torch.int64)
        kc_ref, vc_ref = kc.cpu(), vc.cpu()
        oracle.reshape_and_cache(k_new, v_new, kc_ref, vc_ref, slots)
        pa.pa_decode(out, q, kc, vc, tables, lens_t, scale, max_context_len=max_ctx, partition_size=P,
                     status=status, k_new=k_new.cuda(), v_new=v_new.cuda(), slot_mapping=slots.cuda(), simt=simt)
        torch.cuda.synchronize()
        assert torch.equal(kc.cpu().view(torch.uint8), kc_ref.view(torch.uint8))
    else:
        kc_ref, vc_ref = kc, vc
        pa.pa_decode(out, q, kc, vc, tables, lens_t, scale, max_context_len=max_ctx, partition_size=P,
                     status=status, simt=simt)
        torch.cuda.synchronize()
    assert status.read() == 0
    ref = oracle_decode(q, kc_ref, vc_ref, tables, lens_t, scale)
    assert_decode_close(out, ref, dtype,
                        what=f"seed {seed}: {dtype} hd{hd} bs{bs} {Hq}/{Hkv} P={P} lens={lens} fused={fused} simt={simt}")
