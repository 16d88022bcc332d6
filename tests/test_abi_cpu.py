"""The C-ABI library builds, loads without a GPU and exports every function
include/pa.h declares; host-side argument checks fail before any launch."""
import ctypes

import pytest
import torch

from paged_kv_cache_237_gb300 import build as pa_build


@pytest.fixture(scope="module")
def lib():
    pa_build.build()
    from paged_kv_cache_237_gb300 import binding
    return binding


def test_every_declared_function_is_exported(lib):
    names = lib.declared_functions()
    assert "pa_decode" in names and "pa_reshape_and_cache" in names and "pa_copy_blocks" in names
    raw = ctypes.CDLL(lib.library_path())
    missing = [n for n in names if not hasattr(raw, n)]
    assert not missing, missing


def test_version_and_error_string(lib):
    assert lib._lib.pa_version() >> 16 == 1
    assert isinstance(lib._lib.pa_last_error_string(), bytes)


def _args(lib, **kw):
    a = lib._DecodeArgs(kw.get("num_seqs", 2), kw.get("max_blocks", 4), kw.get("num_blocks", 8),
                        kw.get("dtype", lib.PA_BF16), kw.get("partition_size", 0),
                        kw.get("max_context_len", 64), kw.get("workspace", None),
                        kw.get("workspace_bytes", 0), None, None, kw.get("phase", 0))
    return a


FAKE = 0x10000  # a 16-byte aligned non-null value; no call below reaches a kernel


@pytest.mark.parametrize("change,code", [
    (dict(head_dim=96), -2), (dict(block_size=8), -2), (dict(num_q_heads=6, num_kv_heads=4), -1),
    (dict(dtype=7), -1), (dict(partition_size=24), -1), (dict(partition_size=8192), -1),
    (dict(max_context_len=4096, partition_size=512), -7), (dict(null_q=True), -1),
    (dict(misaligned=True), -1), (dict(phase=3), -1),
])
def test_pa_decode_rejects_bad_arguments_on_the_host(lib, change, code):
    hd = change.get("head_dim", 128)
    bs = change.get("block_size", 16)
    hq, hkv = change.get("num_q_heads", 8), change.get("num_kv_heads", 2)
    a = _args(lib, dtype=change.get("dtype", lib.PA_BF16), partition_size=change.get("partition_size", 0),
              max_context_len=change.get("max_context_len", 64), max_blocks=256,
              phase=change.get("phase", 0))
    q = None if change.get("null_q") else FAKE + (4 if change.get("misaligned") else 0)
    rc = lib._lib.pa_decode(FAKE, q, FAKE, FAKE, FAKE, FAKE, hq, hkv, hd, bs, 0.1, ctypes.byref(a))
    assert rc == code, lib._lib.pa_last_error_string()
    assert lib._lib.pa_last_error_string()


def test_empty_batch_is_a_no_op(lib):
    a = _args(lib, num_seqs=0)
    assert lib._lib.pa_decode(None, None, None, None, None, None, 8, 2, 128, 16, 0.1, ctypes.byref(a)) == 0


def test_workspace_size_formula(lib):
    # no split needed
    assert lib.pa_decode_workspace_size(4, 8, 128, 512, 512) == 0
    # 3 partitions of 512 for 1025 tokens: a 256-byte header (the work counter),
    # then ml = 4*3*8*2 floats and acc = 4*3*8*128 floats, each padded to 256 bytes
    rows = 4 * 3 * 8
    a256 = lambda x: (x + 255) // 256 * 256
    assert lib.pa_decode_workspace_size(4, 8, 128, 1025, 512) == 256 + a256(rows * 8) + a256(rows * 128 * 4)
    assert lib.pa_decode_workspace_size(3, 5, 64, 1025, 512) == 256 + a256(45 * 8) + a256(45 * 64 * 4)
    assert lib.pa_decode_workspace_size(4, 8, 128, 1025, 0) == lib.pa_decode_workspace_size(4, 8, 128, 1025, 512)


def test_cache_ops_reject_bad_arguments_on_the_host(lib):
    L = lib._lib
    assert L.pa_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 128, 16, 4, 9, None, None) == -1
    assert L.pa_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 2, 128, 16, 4, 1, None, None) == 0
    assert L.pa_reshape_and_cache(FAKE + 2, FAKE, FAKE, FAKE, FAKE, 1, 2, 128, 16, 4, 1, None, None) == -1
    assert L.pa_copy_blocks(FAKE, FAKE, None, 1, 2, 128, 16, 4, 1, None, None) == -1
    assert L.pa_copy_blocks(FAKE, FAKE, FAKE, 0, 2, 128, 16, 4, 1, None, None) == 0


def test_binding_refuses_cpu_tensors(lib):
    q = torch.zeros(1, 2, 64)
    with pytest.raises(ValueError):
        lib.pa_decode(q, q, torch.zeros(1, 2, 16, 64), torch.zeros(1, 2, 16, 64),
                      torch.zeros(1, 1, dtype=torch.int32), torch.ones(1, dtype=torch.int32), 0.1,
                      max_context_len=1)


def test_workspace_size_at_the_largest_context_length(lib):
    """The partition count is taken in 64 bits: a context bound of INT_MAX does
    not overflow."""
    int_max = 2**31 - 1
    parts = -(-int_max // 512)
    a256 = lambda x: (x + 255) // 256 * 256
    assert lib.pa_decode_workspace_size(1, 1, 64, int_max, 512) == 256 + a256(parts * 8) + a256(parts * 64 * 4)
    assert lib.pa_decode_workspace_size(1, 1, 64, int_max, 4096) == \
        256 + a256(-(-int_max // 4096) * 8) + a256(-(-int_max // 4096) * 256)


@pytest.mark.parametrize("change,code", [
    (dict(partition_size=8), -1), (dict(partition_size=1), -1), (dict(partition_size=24), -1),
    (dict(head_dim=96), -2), (dict(block_size=8), -2), (dict(dtype=7), -1), (dict(num_seqs=-1), -1),
    (dict(max_context_len=1 << 20, partition_size=16), -7),
])
def test_noalloc_checks_arguments_before_sizing_its_scratch(lib, change, code):
    """pa_decode_noalloc reports a bad size with the code pa_decode gives, not as
    a scratch too small for it; only sizes that are valid but too large for its
    fixed array get PA_ERR_WORKSPACE."""
    a = _args(lib, num_seqs=change.get("num_seqs", 4), dtype=change.get("dtype", lib.PA_BF16),
              partition_size=change.get("partition_size", 0),
              max_context_len=change.get("max_context_len", 32768), max_blocks=1 << 16)
    rc = lib._lib.pa_decode_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 8, change.get("head_dim", 128),
                                    change.get("block_size", 16), 0.1, ctypes.byref(a))
    assert rc == code, lib._lib.pa_last_error_string()
