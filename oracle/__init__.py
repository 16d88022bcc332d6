"""fp64 CPU oracle for paged decode attention, the cache write and the block copy.

TEST INFRASTRUCTURE ONLY.  The tests, the package smoke check and the CPU
baseline leg of the benchmark may import this package; the library itself never
does, and this package never touches the CUDA library.  It shares no code with
the GPU path: the arithmetic lives in ``paged_ref.c`` (plain C, fp64), the
block-manager model in ``block_manager_ref.py`` and the byte accounting in
``accounting.py``.

What the oracle computes follows the pages on PagedAttention:
"PagedAttention et RadixAttention : parlons de KV Cache" (aitalk.it), section
"PagedAttention : la memoire comme un systeme d'exploitation" -- attention
gathers the fixed-size blocks through a per-sequence table and paging leaves
the model's outputs unchanged -- so the oracle resolves the table into a
contiguous K/V and applies the textbook softmax(scale q K^T) V in fp64.

Every function takes CPU torch tensors and checks their dtype and layout.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "paged_ref.c")
_LIB_PATH = os.path.join(_HERE, "libpa_oracle.so")

F32, BF16 = 0, 1
_ERRORS = {-1: "invalid argument", -4: "index out of range", -9: "out of memory"}

_lib = None
_lock = threading.Lock()


def build_oracle(force: bool = False, out_path: str | None = None, source: str | None = None) -> str:
    """Compile ``paged_ref.c`` with gcc into a shared object and return its path.

    ``source``/``out_path`` let a test compile a modified copy elsewhere.
    """
    src = source or _SRC
    dst = out_path or _LIB_PATH
    if (not force and os.path.exists(dst)
            and os.path.getmtime(dst) >= os.path.getmtime(src)):
        return dst
    tmp = dst + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
           "-ffp-contract=off", src, "-o", tmp, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, dst)
    return dst


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.oracle_paged_decode.restype = i32
    lib.oracle_paged_decode.argtypes = [vp, vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32,
                                        i32, i32, dbl, vp, i64, i32]
    lib.oracle_reshape_and_cache.restype = i32
    lib.oracle_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32]
    lib.oracle_copy_blocks.restype = i32
    lib.oracle_copy_blocks.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32]
    lib.oracle_swap_blocks.restype = i32
    lib.oracle_swap_blocks.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32]
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library.  With ``path`` a
    separately built copy is loaded and returned without caching."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build_oracle()))
        return _lib


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what}: {_ERRORS.get(rc, rc)}")


def _cpu(t: torch.Tensor, dtypes, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise TypeError(f"{name} must be a CPU torch tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    return t.contiguous()


def _cache_dtype(t: torch.Tensor) -> int:
    return F32 if t.dtype == torch.float32 else BF16


def paged_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                 pairs: torch.Tensor | None = None, threads: int | None = None,
                 lib: ctypes.CDLL | None = None) -> torch.Tensor:
    """fp64 paged decode attention.

    q: [S, Hq, hd] (any float dtype; widened to fp64 exactly).
    k_cache, v_cache: [num_blocks, Hkv, block_size, hd], fp32 or bf16.
    block_tables: [S, max_blocks] int32; context_lens: [S] int32.
    pairs: optional [P, 2] int32 of (seq, q head) to compute; other rows of the
    result are NaN.  Returns [S, Hq, hd] float64.
    """
    lib = lib or load()
    q64 = _cpu(q, (torch.float64, torch.float32, torch.bfloat16), "q").to(torch.float64).contiguous()
    kc = _cpu(k_cache, (torch.float32, torch.bfloat16), "k_cache")
    vc = _cpu(v_cache, (kc.dtype,), "v_cache")
    bt = _cpu(block_tables, (torch.int32,), "block_tables")
    cl = _cpu(context_lens, (torch.int32,), "context_lens")
    S, Hq, hd = q64.shape
    nb, Hkv, bs, hd2 = kc.shape
    if hd2 != hd or vc.shape != kc.shape or bt.dim() != 2 or bt.shape[0] != S or cl.shape != (S,):
        raise ValueError("oracle paged_decode: inconsistent shapes")
    out = torch.full((S, Hq, hd), float("nan"), dtype=torch.float64)
    if pairs is not None:
        pr = _cpu(pairs, (torch.int32,), "pairs")
        pp, npairs = pr.data_ptr(), pr.shape[0]
    else:
        pr, pp, npairs = None, None, 0
    nthreads = threads if threads is not None else min(os.cpu_count() or 1, 64)
    rc = lib.oracle_paged_decode(out.data_ptr(), q64.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                                 _cache_dtype(kc), bt.data_ptr(), bt.shape[1], cl.data_ptr(),
                                 S, Hq, Hkv, hd, bs, nb, float(scale), pp, npairs, nthreads)
    _check(rc, "paged_decode")
    return out


def reshape_and_cache(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                      lib: ctypes.CDLL | None = None) -> None:
    """In-place cache write on CPU tensors: k, v [T, Hkv, hd]; slot_mapping [T] int64."""
    lib = lib or load()
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("caches must be contiguous")
    kk = _cpu(k, (k_cache.dtype,), "k")
    vv = _cpu(v, (k_cache.dtype,), "v")
    sm = _cpu(slot_mapping, (torch.int64,), "slot_mapping")
    nb, Hkv, bs, hd = k_cache.shape
    rc = lib.oracle_reshape_and_cache(kk.data_ptr(), vv.data_ptr(), k_cache.data_ptr(),
                                      v_cache.data_ptr(), sm.data_ptr(), sm.shape[0], Hkv, hd,
                                      bs, nb, k_cache.element_size())
    _check(rc, "reshape_and_cache")


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src_dst_pairs: torch.Tensor,
                lib: ctypes.CDLL | None = None) -> None:
    """In-place block copy on CPU tensors; src_dst_pairs [P, 2] int64."""
    lib = lib or load()
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("caches must be contiguous")
    pr = _cpu(src_dst_pairs, (torch.int64,), "src_dst_pairs")
    nb, Hkv, bs, hd = k_cache.shape
    rc = lib.oracle_copy_blocks(k_cache.data_ptr(), v_cache.data_ptr(), pr.data_ptr(),
                                pr.shape[0], Hkv, hd, bs, nb, k_cache.element_size())
    _check(rc, "copy_blocks")


def swap_blocks(src_k: torch.Tensor, src_v: torch.Tensor, dst_k: torch.Tensor, dst_v: torch.Tensor,
                src_dst_pairs: torch.Tensor, lib: ctypes.CDLL | None = None) -> None:
    """In-place block copy between two CPU pools of the same geometry."""
    lib = lib or load()
    for t in (src_k, src_v, dst_k, dst_v):
        if t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError("pools must be contiguous CPU tensors")
    pr = _cpu(src_dst_pairs, (torch.int64,), "src_dst_pairs")
    nbs, Hkv, bs, hd = src_k.shape
    nbd = dst_k.shape[0]
    rc = lib.oracle_swap_blocks(src_k.data_ptr(), src_v.data_ptr(), dst_k.data_ptr(), dst_v.data_ptr(),
                                pr.data_ptr(), pr.shape[0], nbs, nbd, Hkv, hd, bs, src_k.element_size())
    _check(rc, "swap_blocks")
