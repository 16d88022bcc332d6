"""ctypes binding of the C-ABI library (``include/pa.h``).

Argument marshalling only: every function checks tensor devices, dtypes,
shapes and contiguity, then passes raw pointers, sizes and the current CUDA
stream to the library, whose kernels do all the work.  Importing this module
without the built library raises ImportError; there is no fallback path.

Names follow the C ABI: ``pa_decode``, ``pa_decode_workspace_size``,
``pa_reshape_and_cache``, ``pa_copy_blocks`` and the ``BlockManager`` class
over ``pa_bm_*``.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from . import build as _build

PA_OK = 0
PA_ERR_INVALID_ARG = -1
PA_ERR_UNSUPPORTED = -2
PA_ERR_CUDA = -3
PA_ERR_BAD_INDEX = -4
PA_ERR_NO_BLOCKS = -5
PA_ERR_REFCOUNT = -6
PA_ERR_WORKSPACE = -7

PA_F32, PA_BF16 = 0, 1
PA_PHASE_ALL, PA_PHASE_PARTITIONS, PA_PHASE_REDUCE = 0, 1, 2

STATUS_BAD_BLOCK_ID = 1
STATUS_BAD_CONTEXT_LEN = 2
STATUS_BAD_SLOT = 4
STATUS_BAD_PAIR = 8
STATUS_WAIT_TIMEOUT = 16


class PAError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


class _DecodeArgs(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int),
        ("max_blocks_per_seq", ctypes.c_int),
        ("num_blocks", ctypes.c_int),
        ("dtype", ctypes.c_int),
        ("partition_size", ctypes.c_int),
        ("max_context_len", ctypes.c_int),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("dev_status", ctypes.c_void_p),
        ("stream", ctypes.c_void_p),
        ("phase", ctypes.c_int),
        ("k_new", ctypes.c_void_p),
        ("v_new", ctypes.c_void_p),
        ("slot_mapping", ctypes.c_void_p),
        ("simt", ctypes.c_int),
        ("skip_counter_reset", ctypes.c_int),
    ]


def library_path() -> str:
    return _build.LIB_PATH


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.pa_decode.restype = i32
    lib.pa_decode.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, ctypes.POINTER(_DecodeArgs)]
    lib.pa_decode_noalloc.restype = i32
    lib.pa_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32,
                                      ctypes.POINTER(_DecodeArgs)]
    lib.pa_decode_workspace_size.restype = sz
    lib.pa_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    lib.pa_reshape_and_cache.restype = i32
    lib.pa_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp]
    lib.pa_copy_blocks.restype = i32
    lib.pa_copy_blocks.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp]
    lib.pa_swap_blocks.restype = i32
    lib.pa_swap_blocks.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp]
    lib.pa_bm_move_seq.restype = i32
    lib.pa_bm_move_seq.argtypes = [vp, vp, i32, vp, i32, ctypes.POINTER(i32)]
    lib.pa_selftest_wait_timeout.restype = i32
    lib.pa_selftest_wait_timeout.argtypes = [vp, i32, vp]
    lib.pa_bm_create.restype = vp
    lib.pa_bm_create.argtypes = [i32, i32]
    lib.pa_bm_destroy.restype = None
    lib.pa_bm_destroy.argtypes = [vp]
    lib.pa_bm_add_seq.restype = i32
    lib.pa_bm_add_seq.argtypes = [vp, i32, i32]
    lib.pa_bm_fork.restype = i32
    lib.pa_bm_fork.argtypes = [vp, i32, i32]
    lib.pa_bm_append_slot.restype = i32
    lib.pa_bm_append_slot.argtypes = [vp, i32, ctypes.POINTER(i64), ctypes.POINTER(ctypes.c_int32),
                                      ctypes.POINTER(ctypes.c_int32)]
    lib.pa_bm_free_seq.restype = i32
    lib.pa_bm_free_seq.argtypes = [vp, i32]
    lib.pa_bm_block_table.restype = i32
    lib.pa_bm_block_table.argtypes = [vp, i32, vp, i32]
    lib.pa_bm_num_tokens.restype = i32
    lib.pa_bm_num_tokens.argtypes = [vp, i32]
    lib.pa_bm_num_free.restype = i32
    lib.pa_bm_num_free.argtypes = [vp]
    lib.pa_bm_refcount.restype = i32
    lib.pa_bm_refcount.argtypes = [vp, i32]
    lib.pa_bm_append_slots.restype = i32
    lib.pa_bm_append_slots.argtypes = [vp, vp, i32, vp, vp, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    lib.pa_bm_add_seq_cached.restype = i32
    lib.pa_bm_add_seq_cached.argtypes = [vp, i32, vp, i32, ctypes.c_uint64, ctypes.POINTER(i32)]
    lib.pa_bm_register_blocks.restype = i32
    lib.pa_bm_register_blocks.argtypes = [vp, i32, vp, i32, ctypes.c_uint64]
    lib.pa_bm_num_cached.restype = i32
    lib.pa_bm_num_cached.argtypes = [vp]
    lib.pa_bm_build_tables.restype = i32
    lib.pa_bm_build_tables.argtypes = [vp, vp, i32, vp, i32, vp]
    lib.pa_last_error_string.restype = ctypes.c_char_p
    lib.pa_last_error_string.argtypes = []
    lib.pa_version.restype = i32
    lib.pa_version.argtypes = []
    return lib


def load_library() -> ctypes.CDLL:
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(f"{path} is not built; run `python -m paged_kv_cache_237_gb300.build` "
                          "or __graft_entry__.build() first")
    return _declare(ctypes.CDLL(path))


_lib = load_library()


def declared_functions(header: str | None = None) -> list[str]:
    """Names of the functions include/pa.h declares (used by the ABI tests)."""
    header = header or os.path.join(_build.INCLUDE, "pa.h")
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def _raise(rc: int):
    if rc != PA_OK:
        raise PAError(rc, _lib.pa_last_error_string().decode())


def _stream_ptr(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check_cuda(t: torch.Tensor, name: str, dtypes, dev=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if dev is not None and t.device != dev:
        raise ValueError(f"{name} is on {t.device}, expected {dev}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return PA_F32
    if dt == torch.bfloat16:
        return PA_BF16
    raise TypeError(f"unsupported dtype {dt}")


class DeviceStatus:
    """A device int32 word that kernels OR PA_STATUS_* bits into."""

    def __init__(self, device="cuda"):
        self.tensor = torch.zeros(1, dtype=torch.int32, device=device)

    def ptr(self) -> int:
        return self.tensor.data_ptr()

    def read(self, clear: bool = True) -> int:
        v = int(self.tensor.item())
        if clear:
            self.tensor.zero_()
        return v


def pa_decode_workspace_size(num_seqs: int, num_q_heads: int, head_dim: int, max_context_len: int,
                             partition_size: int = 0) -> int:
    return int(_lib.pa_decode_workspace_size(num_seqs, num_q_heads, head_dim, max_context_len,
                                             partition_size))


def pa_decode(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
              block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float, *,
              max_context_len: int, partition_size: int = 0, workspace: torch.Tensor | None = None,
              status: DeviceStatus | None = None, stream=None, phase: int = 0,
              k_new: torch.Tensor | None = None, v_new: torch.Tensor | None = None,
              slot_mapping: torch.Tensor | None = None, simt: bool = False,
              skip_counter_reset: bool = False) -> torch.Tensor:
    """Paged decode attention; writes ``out`` [S, Hq, hd] and returns it.

    q [S, Hq, hd]; k_cache, v_cache [num_blocks, Hkv, block_size, hd];
    block_tables [S, max_blocks] int32; context_lens [S] int32.  When any
    sequence may span more than one partition a workspace of
    ``pa_decode_workspace_size`` bytes is needed; if none is given one is
    allocated (zeroed) with torch for this call.  ``skip_counter_reset=True``
    skips the reset of the workspace's work counter; valid when the counter is
    zero (a zeroed workspace, or one a completed call has used).

    With k_new, v_new [S, Hkv, hd] and slot_mapping [S] int64, each
    sequence's new (last) token is written into the caches and attended in the
    same launch (fused cache write).  ``simt=True`` (bf16 only) computes the
    products with fp32 FMAs instead of tensor-core MMAs.
    """
    fdt = (torch.float32, torch.bfloat16)
    _check_cuda(q, "q", fdt)
    dev = q.device
    _check_cuda(out, "out", (q.dtype,), dev)
    _check_cuda(k_cache, "k_cache", (q.dtype,), dev)
    _check_cuda(v_cache, "v_cache", (q.dtype,), dev)
    _check_cuda(block_tables, "block_tables", (torch.int32,), dev)
    _check_cuda(context_lens, "context_lens", (torch.int32,), dev)
    if q.dim() != 3 or k_cache.dim() != 4 or block_tables.dim() != 2:
        raise ValueError("q must be [S, Hq, hd], caches [num_blocks, Hkv, bs, hd], tables [S, max_blocks]")
    S, Hq, hd = q.shape
    nb, Hkv, bs, hd2 = k_cache.shape
    if (hd2 != hd or tuple(v_cache.shape) != tuple(k_cache.shape) or tuple(out.shape) != tuple(q.shape)
            or block_tables.shape[0] != S or tuple(context_lens.shape) != (S,)):
        raise ValueError("inconsistent shapes")
    need = pa_decode_workspace_size(S, Hq, hd, max_context_len, partition_size)
    if need and workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=dev)
        skip_counter_reset = True
    if workspace is not None:
        _check_cuda(workspace, "workspace", (torch.uint8,), dev)
    fused = (k_new, v_new, slot_mapping)
    if any(t is not None for t in fused):
        if any(t is None for t in fused):
            raise ValueError("k_new, v_new and slot_mapping go together")
        _check_cuda(k_new, "k_new", (q.dtype,), dev)
        _check_cuda(v_new, "v_new", (q.dtype,), dev)
        _check_cuda(slot_mapping, "slot_mapping", (torch.int64,), dev)
        if tuple(k_new.shape) != (S, Hkv, hd) or tuple(v_new.shape) != (S, Hkv, hd) or \
                tuple(slot_mapping.shape) != (S,):
            raise ValueError("k_new, v_new must be [S, Hkv, hd] and slot_mapping [S]")
    args = _DecodeArgs(S, block_tables.shape[1], nb, _dtype_code(q.dtype), partition_size,
                       max_context_len,
                       workspace.data_ptr() if workspace is not None else None,
                       workspace.numel() if workspace is not None else 0,
                       status.ptr() if status is not None else None,
                       _stream_ptr(stream, dev), phase,
                       k_new.data_ptr() if k_new is not None else None,
                       v_new.data_ptr() if v_new is not None else None,
                       slot_mapping.data_ptr() if slot_mapping is not None else None,
                       1 if simt else 0, 1 if skip_counter_reset else 0)
    with torch.cuda.device(dev):
        rc = _lib.pa_decode(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                            block_tables.data_ptr(), context_lens.data_ptr(), Hq, Hkv, hd, bs,
                            float(scale), ctypes.byref(args))
    _raise(rc)
    return out


def pa_reshape_and_cache(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                         slot_mapping: torch.Tensor, *, status: DeviceStatus | None = None,
                         stream=None) -> None:
    """Write k, v [T, Hkv, hd] into the caches at slot_mapping [T] int64."""
    _check_cuda(k_cache, "k_cache", (torch.float32, torch.bfloat16))
    dev = k_cache.device
    for name, t in (("k", k), ("v", v), ("v_cache", v_cache)):
        _check_cuda(t, name, (k_cache.dtype,), dev)
    _check_cuda(slot_mapping, "slot_mapping", (torch.int64,), dev)
    nb, Hkv, bs, hd = k_cache.shape
    T = slot_mapping.shape[0]
    if tuple(k.shape) != (T, Hkv, hd) or tuple(v.shape) != (T, Hkv, hd) or v_cache.shape != k_cache.shape:
        raise ValueError("inconsistent shapes")
    with torch.cuda.device(dev):
        rc = _lib.pa_reshape_and_cache(k.data_ptr(), v.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                       slot_mapping.data_ptr(), T, Hkv, hd, bs, nb,
                                       _dtype_code(k_cache.dtype),
                                       status.ptr() if status is not None else None,
                                       _stream_ptr(stream, dev))
    _raise(rc)


def pa_copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src_dst_pairs: torch.Tensor, *,
                   status: DeviceStatus | None = None, stream=None) -> None:
    """Copy whole blocks src -> dst in both caches; src_dst_pairs [P, 2] int64."""
    _check_cuda(k_cache, "k_cache", (torch.float32, torch.bfloat16))
    dev = k_cache.device
    _check_cuda(v_cache, "v_cache", (k_cache.dtype,), dev)
    _check_cuda(src_dst_pairs, "src_dst_pairs", (torch.int64,), dev)
    if src_dst_pairs.dim() != 2 or src_dst_pairs.shape[1] != 2 or v_cache.shape != k_cache.shape:
        raise ValueError("inconsistent shapes")
    nb, Hkv, bs, hd = k_cache.shape
    with torch.cuda.device(dev):
        rc = _lib.pa_copy_blocks(k_cache.data_ptr(), v_cache.data_ptr(), src_dst_pairs.data_ptr(),
                                 src_dst_pairs.shape[0], Hkv, hd, bs, nb, _dtype_code(k_cache.dtype),
                                 status.ptr() if status is not None else None,
                                 _stream_ptr(stream, dev))
    _raise(rc)


def pa_swap_blocks(src_k: torch.Tensor, src_v: torch.Tensor, dst_k: torch.Tensor, dst_v: torch.Tensor,
                   src_dst_pairs: torch.Tensor, *, status: DeviceStatus | None = None, stream=None) -> None:
    """Copy whole blocks between two pools of the same geometry, each on the
    GPU or in pinned host memory (swap out / swap in).  src_dst_pairs [P, 2]
    int64, on the GPU or pinned."""
    pools = (("src_k", src_k), ("src_v", src_v), ("dst_k", dst_k), ("dst_v", dst_v))
    for name, t in pools:
        if not isinstance(t, torch.Tensor) or t.dtype not in (torch.float32, torch.bfloat16):
            raise TypeError(f"{name} must be an fp32 or bf16 tensor")
        if not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous [num_blocks, Hkv, bs, hd] tensor")
        if t.device.type == "cpu" and not t.is_pinned():
            raise ValueError(f"{name} is pageable host memory; pin it (pin_memory()) so the GPU can address it")
    if src_k.shape[1:] != dst_k.shape[1:] or src_v.shape != src_k.shape or dst_v.shape != dst_k.shape \
            or len({t.dtype for _, t in pools}) != 1:
        raise ValueError("pools must share block geometry and dtype")
    if src_dst_pairs.dtype != torch.int64 or src_dst_pairs.dim() != 2 or src_dst_pairs.shape[1] != 2:
        raise ValueError("src_dst_pairs must be int64 [P, 2]")
    if src_dst_pairs.device.type == "cpu" and not src_dst_pairs.is_pinned():
        raise ValueError("src_dst_pairs must be on the GPU or pinned")
    devs = {t.device for _, t in pools if t.device.type == "cuda"}
    if src_dst_pairs.device.type == "cuda":
        devs.add(src_dst_pairs.device)
    if len(devs) > 1:
        raise ValueError("all device tensors must be on one GPU")
    dev = devs.pop() if devs else torch.device("cuda", torch.cuda.current_device())
    nbs, Hkv, bs, hd = src_k.shape
    with torch.cuda.device(dev):
        rc = _lib.pa_swap_blocks(src_k.data_ptr(), src_v.data_ptr(), dst_k.data_ptr(), dst_v.data_ptr(),
                                 src_dst_pairs.data_ptr(), src_dst_pairs.shape[0], nbs, dst_k.shape[0], Hkv, hd,
                                 bs, _dtype_code(src_k.dtype), status.ptr() if status is not None else None,
                                 _stream_ptr(stream, dev))
    _raise(rc)


class BlockManager:
    """Host block manager (``pa_bm_*``): free pool, refcounts, copy-on-write."""

    def __init__(self, num_blocks: int, block_size: int):
        self._h = _lib.pa_bm_create(num_blocks, block_size)
        if not self._h:
            raise PAError(PA_ERR_INVALID_ARG, _lib.pa_last_error_string().decode())
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self):
        if self._h:
            _lib.pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_seq(self, seq_id: int, num_tokens: int) -> None:
        _raise(_lib.pa_bm_add_seq(self._h, seq_id, num_tokens))

    def fork(self, parent: int, child: int) -> None:
        _raise(_lib.pa_bm_fork(self._h, parent, child))

    def append_slot(self, seq_id: int):
        slot = ctypes.c_int64()
        src, dst = ctypes.c_int32(), ctypes.c_int32()
        _raise(_lib.pa_bm_append_slot(self._h, seq_id, ctypes.byref(slot), ctypes.byref(src),
                                      ctypes.byref(dst)))
        return slot.value, src.value, dst.value

    def append_slots(self, seq_ids):
        """Batched append; returns (slots int64 [n], cow_pairs int64 [P, 2])."""
        ids = torch.tensor(list(seq_ids), dtype=torch.int32)
        n = ids.numel()
        slots = torch.empty(n, dtype=torch.int64)
        pairs = torch.empty(max(n, 1), 2, dtype=torch.int64)
        npairs, ndone = ctypes.c_int(), ctypes.c_int()
        rc = _lib.pa_bm_append_slots(self._h, ids.data_ptr(), n, slots.data_ptr(), pairs.data_ptr(),
                                     ctypes.byref(npairs), ctypes.byref(ndone))
        _raise(rc)
        return slots, pairs[:npairs.value].clone()

    def add_seq_cached(self, seq_id: int, tokens, salt: int = 0) -> int:
        """New sequence over token ids, sharing cached prefix blocks (chained
        block keys, tenant salt).  Returns the number of leading tokens whose
        K/V are already in the cache."""
        t = torch.as_tensor(list(tokens) if not isinstance(tokens, torch.Tensor) else tokens,
                            dtype=torch.int32).contiguous()
        cached = ctypes.c_int()
        _raise(_lib.pa_bm_add_seq_cached(self._h, seq_id, t.data_ptr() if t.numel() else None, t.numel(),
                                         ctypes.c_uint64(salt & (2**64 - 1)), ctypes.byref(cached)))
        return cached.value

    def register_blocks(self, seq_id: int, tokens, salt: int = 0) -> int:
        """Key the sequence's full blocks not keyed yet; returns how many."""
        t = torch.as_tensor(list(tokens) if not isinstance(tokens, torch.Tensor) else tokens,
                            dtype=torch.int32).contiguous()
        n = _lib.pa_bm_register_blocks(self._h, seq_id, t.data_ptr() if t.numel() else None, t.numel(),
                                       ctypes.c_uint64(salt & (2**64 - 1)))
        if n < 0:
            _raise(n)
        return n

    def num_cached(self) -> int:
        return _lib.pa_bm_num_cached(self._h)

    def move_seq(self, to: "BlockManager", seq_id: int) -> torch.Tensor:
        """Move a sequence into another manager's pool; returns the int64
        [P, 2] (block here, block there) pairs for pa_swap_blocks."""
        cap = max(1, len(self.block_table(seq_id)))
        pairs = torch.empty(cap, 2, dtype=torch.int64)
        n = ctypes.c_int()
        _raise(_lib.pa_bm_move_seq(self._h, to._h, seq_id, pairs.data_ptr(), cap, ctypes.byref(n)))
        return pairs[:n.value].clone()

    def free_seq(self, seq_id: int) -> None:
        _raise(_lib.pa_bm_free_seq(self._h, seq_id))

    def block_table(self, seq_id: int) -> list[int]:
        cap = max(1, self.num_blocks)
        buf = (ctypes.c_int32 * cap)()
        n = _lib.pa_bm_block_table(self._h, seq_id, buf, cap)
        if n < 0:
            _raise(n)
        return list(buf[:n])

    def num_tokens(self, seq_id: int) -> int:
        n = _lib.pa_bm_num_tokens(self._h, seq_id)
        if n < 0:
            _raise(n)
        return n

    def num_free(self) -> int:
        return _lib.pa_bm_num_free(self._h)

    def refcount(self, block: int) -> int:
        r = _lib.pa_bm_refcount(self._h, block)
        if r < 0:
            _raise(r)
        return r

    def build_tables(self, seq_ids, max_blocks_per_seq: int):
        """Padded int32 tables [n, max_blocks_per_seq] and context lengths [n] (host)."""
        ids = torch.tensor(list(seq_ids), dtype=torch.int32)
        n = ids.numel()
        tables = torch.empty(n, max_blocks_per_seq, dtype=torch.int32)
        lens = torch.empty(n, dtype=torch.int32)
        _raise(_lib.pa_bm_build_tables(self._h, ids.data_ptr(), n, tables.data_ptr(),
                                       max_blocks_per_seq, lens.data_ptr()))
        return tables, lens
