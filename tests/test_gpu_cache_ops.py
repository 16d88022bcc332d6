"""pa_reshape_and_cache and pa_copy_blocks on the GPU: bit-exact against the
oracle's host copies, including untouched blocks, padding slots and the
rejected cases."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    from paged_kv_cache_237_gb300 import binding
    return binding


def bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("hd,bs,Hkv", [(128, 16, 8), (64, 32, 4), (128, 32, 1)])
def test_reshape_and_cache_is_bit_exact(pa, dtype, hd, bs, Hkv):
    nb, T = 40, 57
    g = torch.Generator().manual_seed(hd + bs)
    kc = torch.randn(nb, Hkv, bs, hd, generator=g).to(dtype)
    vc = torch.randn(nb, Hkv, bs, hd, generator=g).to(dtype)
    k = torch.randn(T, Hkv, hd, generator=g).to(dtype)
    v = torch.randn(T, Hkv, hd, generator=g).to(dtype)
    slots = np.random.default_rng(hd).choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[::9] = -1
    sm = torch.from_numpy(slots)
    ek, ev = kc.clone(), vc.clone()
    oracle.reshape_and_cache(k, v, ek, ev, sm)
    dk, dv = kc.cuda(), vc.cuda()
    status = pa.DeviceStatus()
    pa.pa_reshape_and_cache(k.cuda(), v.cuda(), dk, dv, sm.cuda(), status=status)
    torch.cuda.synchronize()
    assert status.read() == 0
    assert torch.equal(bits(dk.cpu()), bits(ek)) and torch.equal(bits(dv.cpu()), bits(ev))


def test_reshape_and_cache_flags_slot_past_the_pool(pa):
    kc = torch.zeros(4, 2, 16, 64, device="cuda")
    vc = torch.zeros_like(kc)
    k = torch.ones(2, 2, 64, device="cuda")
    status = pa.DeviceStatus()
    pa.pa_reshape_and_cache(k, k, kc, vc, torch.tensor([3, 4 * 16 + 7], device="cuda"), status=status)
    torch.cuda.synchronize()
    assert status.read() & pa.STATUS_BAD_SLOT
    assert kc[0, :, 3].eq(1).all() and kc.sum().item() == 2 * 64


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_copy_blocks_is_bit_exact(pa, dtype):
    nb, Hkv, bs, hd = 30, 8, 16, 128
    g = torch.Generator().manual_seed(1)
    kc = torch.randn(nb, Hkv, bs, hd, generator=g).to(dtype)
    vc = torch.randn(nb, Hkv, bs, hd, generator=g).to(dtype)
    pairs = torch.tensor([[3, 20], [3, 21], [7, 22], [0, 29], [5, 5]], dtype=torch.int64)
    ek, ev = kc.clone(), vc.clone()
    oracle.copy_blocks(ek, ev, pairs)
    dk, dv = kc.cuda(), vc.cuda()
    status = pa.DeviceStatus()
    pa.pa_copy_blocks(dk, dv, pairs.cuda(), status=status)
    torch.cuda.synchronize()
    assert status.read() == 0
    assert torch.equal(bits(dk.cpu()), bits(ek)) and torch.equal(bits(dv.cpu()), bits(ev))


def test_copy_blocks_rejects_racing_and_out_of_range_pairs(pa):
    nb = 8
    kc = torch.arange(nb, dtype=torch.float32).view(nb, 1, 1, 1).expand(nb, 1, 16, 64).contiguous().cuda()
    vc = kc.clone()
    status = pa.DeviceStatus()
    # pair 0 writes block 2, which pair 1 reads; pair 2 is out of range; pair 3 is fine
    pairs = torch.tensor([[1, 2], [2, 3], [0, 99], [4, 5]], dtype=torch.int64, device="cuda")
    pa.pa_copy_blocks(kc, vc, pairs, status=status)
    torch.cuda.synchronize()
    assert status.read() & pa.STATUS_BAD_PAIR
    got = kc[:, 0, 0, 0].cpu().tolist()
    assert got[2] == 2.0          # skipped: its dst is another pair's src
    assert got[3] == 2.0          # pair 1 copied the untouched block 2
    assert got[5] == 4.0          # valid pair applied


def test_bounded_wait_gives_up_and_reports(pa):
    """The decode kernels' bounded wait, on a barrier nothing completes, gives
    up after its limit, flags PA_STATUS_WAIT_TIMEOUT and lets the kernel end;
    the context stays usable."""
    import ctypes
    import time
    status = pa.DeviceStatus()
    t0 = time.perf_counter()
    rc = pa._lib.pa_selftest_wait_timeout(ctypes.c_void_p(status.ptr()), 20000, None)
    assert rc == 0
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert status.read() & pa.STATUS_WAIT_TIMEOUT
    assert 0.015 < dt < 5.0
    x = torch.ones(1024, device="cuda")
    assert float((x * 2).sum()) == 2048.0       # the GPU still runs work
