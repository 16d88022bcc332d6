"""pa_decode_noalloc: decode attention for callers that cannot allocate device
memory (a host framework that owns every allocation and passes only inputs
and outputs, or a hot path where cudaMalloc, which may synchronise the
device, is not allowed).  Its split-K scratch is a fixed array inside the
library, so the caller passes no workspace.

Called straight through the C ABI (ctypes) and compared with pa_decode, which
takes a caller workspace, on two calls in a row with different inputs (the
second call finds the first call's data in the shared array).  This file is
collected last so that a run stopping at the first failure has already run
every other test; it also passes on its own in a fresh process.
"""
import ctypes
import math

import pytest
import torch

from helpers import assert_decode_close, make_case

pytestmark = pytest.mark.gpu

NOALLOC_BYTES = 64 * 1024 * 1024


@pytest.fixture(scope="module")
def pa():
    from paged_kv_cache_237_gb300 import binding
    return binding


def c_args(pa, q, kc, tables, max_ctx, partition_size, status):
    return pa._DecodeArgs(q.shape[0], tables.shape[1], kc.shape[0], pa._dtype_code(q.dtype), partition_size,
                          max_ctx, None, 0, status.ptr(), torch.cuda.current_stream().cuda_stream, 0)


def call_noalloc(pa, out, q, kc, vc, tables, lens, scale, max_ctx, partition_size, status):
    args = c_args(pa, q, kc, tables, max_ctx, partition_size, status)
    rc = pa._lib.pa_decode_noalloc(out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                                   tables.data_ptr(), lens.data_ptr(), q.shape[1], kc.shape[1], q.shape[2],
                                   kc.shape[2], ctypes.c_float(scale), ctypes.byref(args))
    return rc


def test_noalloc_matches_pa_decode_on_two_calls_in_a_row(pa):
    cases = [
        # (lens, Hq, Hkv, hd, bs, dtype, partition)
        ([5000, 17, 1024, 3000, 1, 4097, 640, 2600], 32, 8, 128, 16, torch.bfloat16, 512),
        ([2100, 64, 9000, 333, 4096, 12], 16, 2, 64, 32, torch.bfloat16, 256),
    ]
    for call, (lens, Hq, Hkv, hd, bs, dtype, P) in enumerate(cases):
        q, kc, vc, tables, lens_t = make_case(lens, Hq, Hkv, hd, bs, dtype, seed=100 + call)
        max_ctx = max(lens)
        need = pa.pa_decode_workspace_size(len(lens), Hq, hd, max_ctx, P)
        assert 0 < need <= NOALLOC_BYTES          # the split-K scratch is really used
        scale = 1.0 / math.sqrt(hd)
        ref = torch.empty_like(q)
        pa.pa_decode(ref, q, kc, vc, tables, lens_t, scale, max_context_len=max_ctx, partition_size=P)
        out = torch.full_like(q, float("nan"))
        status = pa.DeviceStatus()
        rc = call_noalloc(pa, out, q, kc, vc, tables, lens_t, scale, max_ctx, P, status)
        assert rc == 0, pa._lib.pa_last_error_string()
        torch.cuda.synchronize()
        assert status.read() == 0
        assert_decode_close(out, ref.double(), dtype, what=f"noalloc call {call}")


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch(pa):
    lens = [32768] * 4
    q, kc, vc, tables, lens_t = make_case([16] * 4, 64, 8, 128, 16, torch.bfloat16, seed=7)
    # claim a long context so that the needed scratch exceeds the fixed array
    big_ctx = 32768
    assert pa.pa_decode_workspace_size(4, 64, 128, big_ctx, 16) > NOALLOC_BYTES
    wide = torch.zeros(4, big_ctx // 16, dtype=torch.int32, device="cuda")
    wide[:, :1] = tables[:, :1]
    out = torch.zeros_like(q)
    status = pa.DeviceStatus()
    rc = call_noalloc(pa, out, q, kc, vc, wide, lens_t, 0.1, big_ctx, 16, status)
    assert rc == pa.PA_ERR_WORKSPACE
    assert b"PA_NOALLOC_WORKSPACE_BYTES" in pa._lib.pa_last_error_string()
    assert torch.count_nonzero(out) == 0       # nothing was enqueued
    del lens


def test_noalloc_may_skip_the_counter_reset(pa):
    """The fixed scratch starts at zero and every completed call leaves its
    work counter at zero, so a caller may set skip_counter_reset: the same
    bits come out as with the reset, call after call."""
    lens = [3000, 700, 4096, 1, 513, 2049]
    q, kc, vc, tables, lens_t = make_case(lens, 16, 2, 128, 16, torch.bfloat16, seed=77)
    max_ctx, P, scale = max(lens), 256, 0.09
    outs = []
    for skip in (0, 1, 1, 0, 1):
        out = torch.full_like(q, float("nan"))
        status = pa.DeviceStatus()
        args = c_args(pa, q, kc, tables, max_ctx, P, status)
        args.skip_counter_reset = skip
        rc = pa._lib.pa_decode_noalloc(out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                                       tables.data_ptr(), lens_t.data_ptr(), q.shape[1], kc.shape[1], q.shape[2],
                                       kc.shape[2], ctypes.c_float(scale), ctypes.byref(args))
        assert rc == 0, pa._lib.pa_last_error_string()
        torch.cuda.synchronize()
        assert status.read() == 0
        outs.append(out)
    for out in outs[1:]:
        assert torch.equal(out.view(torch.int16), outs[0].view(torch.int16))
