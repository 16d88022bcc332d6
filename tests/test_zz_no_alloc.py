"""pa_decode_noalloc: decode attention for callers that cannot allocate device
memory (a host framework that owns every allocation and passes only inputs
and outputs, or a hot path where cudaMalloc, which may synchronise the
device, is not allowed).  Its split-K scratch is a fixed array inside the
library, so the caller passes no workspace.

Called straight through the C ABI (ctypes) and compared with pa_decode, which
takes a caller workspace.  Both run the same deterministic kernels at the same
partition size, so the outputs must be identical bit for bit; each output is
also checked against the fp64 oracle at the usual tolerance.  Calls come in
pairs with different inputs, so the second finds the first call's data in the
shared array.  This file is collected last so that a run stopping at the
first failure has already run every other test; it also passes on its own in
a fresh process.
"""
import ctypes
import math

import pytest
import torch

from helpers import assert_decode_close, make_case, oracle_decode

pytestmark = pytest.mark.gpu

NOALLOC_BYTES = 64 * 1024 * 1024


@pytest.fixture(scope="module")
def pa():
    from paged_kv_cache_237_gb300 import binding
    return binding


def c_args(pa, q, kc, tables, max_ctx, partition_size, status, phase=0):
    return pa._DecodeArgs(q.shape[0], tables.shape[1], kc.shape[0], pa._dtype_code(q.dtype), partition_size,
                          max_ctx, None, 0, status.ptr(), torch.cuda.current_stream().cuda_stream, phase)


def call_noalloc(pa, out, q, kc, vc, tables, lens, scale, max_ctx, partition_size, status, phase=0):
    args = c_args(pa, q, kc, tables, max_ctx, partition_size, status, phase)
    rc = pa._lib.pa_decode_noalloc(out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                                   tables.data_ptr(), lens.data_ptr(), q.shape[1], kc.shape[1], q.shape[2],
                                   kc.shape[2], ctypes.c_float(scale), ctypes.byref(args))
    return rc


def same_bits(a, b):
    ia = a.view(torch.int32) if a.dtype == torch.float32 else a.view(torch.int16)
    ib = b.view(torch.int32) if b.dtype == torch.float32 else b.view(torch.int16)
    return torch.equal(ia, ib)


CASES = [
    # (lens, Hq, Hkv, hd, bs, dtype, partition)
    ([5000, 17, 1024, 3000, 1, 4097, 640, 2600], 32, 8, 128, 16, torch.bfloat16, 512),
    ([2100, 64, 9000, 333, 4096, 12], 16, 2, 64, 32, torch.bfloat16, 256),
    ([1500, 3, 700, 2049, 260], 8, 8, 128, 16, torch.float32, 256),
    ([999, 31, 1600], 12, 4, 64, 32, torch.float32, 128),
]


def test_noalloc_matches_pa_decode_bit_for_bit_on_calls_in_a_row(pa):
    for call, (lens, Hq, Hkv, hd, bs, dtype, P) in enumerate(CASES):
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
        assert same_bits(out, ref), f"noalloc call {call} differs from pa_decode"
        assert_decode_close(out, oracle_decode(q, kc, vc, tables, lens_t, scale), dtype,
                            what=f"noalloc call {call} vs oracle")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_noalloc_split_phases_read_the_partials_left_in_the_array(pa, dtype):
    """PA_PHASE_PARTITIONS then PA_PHASE_REDUCE as two calls on one stream: the
    merge reads the partials the first call left in the shared array."""
    lens = [3000, 700, 4096, 1, 513, 2049]
    q, kc, vc, tables, lens_t = make_case(lens, 16, 4, 128, 16, dtype, seed=55)
    max_ctx, P, scale = max(lens), 512, 1 / math.sqrt(128)
    ref = torch.empty_like(q)
    pa.pa_decode(ref, q, kc, vc, tables, lens_t, scale, max_context_len=max_ctx, partition_size=P)
    # a call with other inputs first, so the array holds stale partials
    q2, kc2, vc2, tables2, lens2 = make_case([4000, 2500], 16, 4, 128, 16, dtype, seed=56)
    other = torch.empty_like(q2)
    status = pa.DeviceStatus()
    assert call_noalloc(pa, other, q2, kc2, vc2, tables2, lens2, scale, 4000, P, status) == 0
    out = torch.full_like(q, float("nan"))
    for phase in (pa.PA_PHASE_PARTITIONS, pa.PA_PHASE_REDUCE):
        rc = call_noalloc(pa, out, q, kc, vc, tables, lens_t, scale, max_ctx, P, status, phase)
        assert rc == 0, pa._lib.pa_last_error_string()
    torch.cuda.synchronize()
    assert status.read() == 0
    assert same_bits(out, ref)
    assert_decode_close(out, oracle_decode(q, kc, vc, tables, lens_t, scale), dtype, what="split phases")


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch(pa):
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


def test_noalloc_reports_a_bad_partition_size_as_such(pa):
    """A partition size outside the supported range is an argument error, even
    where the scratch it would need is larger than the fixed array."""
    q, kc, vc, tables, lens_t = make_case([16] * 4, 64, 8, 128, 16, torch.bfloat16, seed=8)
    big_ctx = 32768
    wide = torch.zeros(4, big_ctx // 16, dtype=torch.int32, device="cuda")
    wide[:, :1] = tables[:, :1]
    out = torch.zeros_like(q)
    status = pa.DeviceStatus()
    for P in (8, 1, 24):
        rc = call_noalloc(pa, out, q, kc, vc, wide, lens_t, 0.1, big_ctx, P, status)
        assert rc == pa.PA_ERR_INVALID_ARG, (P, pa._lib.pa_last_error_string())
    assert torch.count_nonzero(out) == 0


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
        assert same_bits(out, outs[0])
