"""Seeded synthetic workloads shaped like the pages' decode scenarios.

This module only draws random inputs (context lengths, physical block
placement, cache/query values, cache-write slots).  It holds none of the
attention, cache-write or block-copy arithmetic, so both the CUDA path and the
oracle can be fed from it.

Workloads (sizes fixed here; the pages name the shapes only loosely):

``tiny_f32``
    fp32, 4 sequences of {7, 16, 33, 50} tokens, 4 query = 4 KV heads,
    head_dim 64, block_size 16, scale 1/8.  A pool of 32 physical blocks; a
    seeded permutation of the pool hands out the 9 needed blocks in
    sequence/logical order.  Four cache writes go to 4 distinct random slots.
``mha_llama2_7b``
    bf16, 64 sequences, 32 query = 32 KV heads, head_dim 128, block_size 16,
    lengths uniform in [128, 2048], pool of ceil(1.2 x need) blocks, shuffled.
``gqa_llama3_70b``
    bf16, 32 sequences, 64 query / 8 KV heads, head_dim 128, block_size 16,
    lengths round(4096 * exp(sigma Z)), Z ~ N(0, 1), sigma 1 (0.5 as a
    sensitivity case), clipped to [256, 32768]; pool of ceil(1.05 x need)
    blocks, shuffled.
``prefix_share``
    bf16, 50 sequences, 32 query / 8 KV heads, head_dim 128, block_size 16: 25
    sampled pairs share one 2048-token prefix; each pair also shares a suffix
    of uniform 0..512 tokens (the pair's last block is partial and shared, so
    the decode step's write triggers copy-on-write).  The block layout itself
    is produced by the block manager from ``prefix_share_layout``.
``long_context``
    bf16, 256 sequences, 64 query / 8 KV heads, head_dim 128, block_size 32:
    8 sequences of 131072 tokens and 248 of uniform 16..32768 tokens; split-K
    partitions of 512 tokens; the pool is sized so that the sequences fill
    ~96% of it, with blocks scattered at random.

``mha_llama2_7b_f32``, ``gqa_llama3_70b_f32``
    The MHA and GQA batches above with fp32 K/V, q and output: the same
    seeds, so the same lengths and placement, and the values before rounding
    to bf16.

All values are N(0, 1) cast to the workload dtype.  Context lengths include the
token written by the step (a decode step first writes the new token's K/V, then
attends over every token present).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: torch.dtype
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    partition_size: int = 512
    seed: int = 0
    notes: str = ""
    extra: dict = field(default_factory=dict)
    recipe: str = ""          # length and pool recipe, when it is another workload's

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def kind(self) -> str:
        return self.recipe or self.name


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", torch.float32, 4, 4, 4, 64, 16, 512, 1),
    "mha_llama2_7b": Workload("mha_llama2_7b", torch.bfloat16, 64, 32, 32, 128, 16, 512, 2),
    "gqa_llama3_70b": Workload("gqa_llama3_70b", torch.bfloat16, 32, 64, 8, 128, 16, 512, 3),
    "prefix_share": Workload("prefix_share", torch.bfloat16, 50, 32, 8, 128, 16, 512, 4),
    "long_context": Workload("long_context", torch.bfloat16, 256, 64, 8, 128, 32, 512, 5),
    "mha_llama2_7b_f32": Workload("mha_llama2_7b_f32", torch.float32, 64, 32, 32, 128, 16, 512, 2,
                                  recipe="mha_llama2_7b"),
    "gqa_llama3_70b_f32": Workload("gqa_llama3_70b_f32", torch.float32, 32, 64, 8, 128, 16, 512, 3,
                                   recipe="gqa_llama3_70b"),
}


def context_lengths(w: Workload, rng: np.random.Generator, gqa_sigma: float = 1.0) -> np.ndarray:
    """Context length per sequence (int64), drawn per the workload's recipe.
    ``gqa_sigma`` is the log-space spread of the GQA batch's lognormal (the
    recipe leaves it open: 1.0 by default, 0.5 as a sensitivity case; the
    same normal draws are scaled, so both cases share one median)."""
    if w.kind == "tiny_f32":
        return np.array([7, 16, 33, 50], dtype=np.int64)
    if w.kind == "mha_llama2_7b":
        return rng.integers(128, 2048, size=w.num_seqs, endpoint=True).astype(np.int64)
    if w.kind == "gqa_llama3_70b":
        z = rng.standard_normal(w.num_seqs)
        return np.clip(np.rint(4096.0 * np.exp(gqa_sigma * z)), 256, 32768).astype(np.int64)
    if w.kind == "long_context":
        short = rng.integers(16, 32768, size=w.num_seqs - 8, endpoint=True)
        lens = np.concatenate([np.full(8, 131072), short]).astype(np.int64)
        return lens[rng.permutation(w.num_seqs)]
    raise ValueError(f"{w.name}: lengths come from prefix_share_layout")


def pool_blocks(w: Workload, need: int) -> int:
    """Physical pool size for a workload needing `need` blocks."""
    if w.kind == "tiny_f32":
        return 32
    if w.kind == "mha_llama2_7b":
        return math.ceil(1.2 * need)
    if w.kind == "gqa_llama3_70b":
        return math.ceil(1.05 * need)
    if w.kind == "long_context":
        return math.ceil(need / 0.96)
    return need


def place_blocks(lens: np.ndarray, block_size: int, num_blocks: int,
                 rng: np.random.Generator, shuffle: bool = True):
    """Hand out physical blocks to each sequence's logical blocks.

    A permutation of the pool (identity when shuffle is False) is consumed in
    sequence order, logical block order.  Returns (block_tables [S, max_blocks]
    int32 padded with -1, blocks_needed).
    """
    per_seq = [(int(n) + block_size - 1) // block_size for n in lens]
    need = sum(per_seq)
    if need > num_blocks:
        raise ValueError("pool too small")
    order = rng.permutation(num_blocks) if shuffle else np.arange(num_blocks)
    max_blocks = max(1, max(per_seq) if per_seq else 1)
    tables = np.full((len(lens), max_blocks), -1, dtype=np.int32)
    pos = 0
    for i, nb in enumerate(per_seq):
        tables[i, :nb] = order[pos:pos + nb]
        pos += nb
    return tables, need


def randn(shape, dtype: torch.dtype, seed: int, device, chunk_elems: int = 1 << 28) -> torch.Tensor:
    """N(0, 1) values cast to dtype, drawn in chunks (bounded temporary memory)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    for start in range(0, flat.numel(), chunk_elems):
        stop = min(flat.numel(), start + chunk_elems)
        flat[start:stop] = torch.randn(stop - start, generator=gen, device=device,
                                       dtype=torch.float32).to(dtype)
    return out


def new_token_slots(lens: np.ndarray, tables: np.ndarray, block_size: int) -> np.ndarray:
    """Physical slot of each sequence's last token (the one a decode step writes)."""
    slots = np.empty(len(lens), dtype=np.int64)
    for i, n in enumerate(lens):
        t = int(n) - 1
        slots[i] = int(tables[i, t // block_size]) * block_size + t % block_size
    return slots


def decode_inputs(name: str, device="cpu", seed: int | None = None, shuffle: bool = True,
                  lens_override=None, block_size: int | None = None, gqa_sigma: float = 1.0,
                  num_seqs: int | None = None) -> dict:
    """All inputs of one decode step of a workload (except prefix_share).

    Returns a dict with q [S, Hq, hd], k_cache/v_cache [num_blocks, Hkv, bs, hd],
    block_tables [S, max_blocks] int32, context_lens [S] int32, k_new/v_new
    [T, Hkv, hd] and slot_mapping [T] int64 (the step's cache writes), plus the
    workload record and host copies of lengths and tables.  ``shuffle=False``
    places every sequence's blocks consecutively (identity placement);
    ``block_size`` overrides the workload's block size (same lengths, same
    pool fill); ``gqa_sigma`` sets the GQA batch's lognormal spread;
    ``num_seqs`` keeps only the first sequences of the drawn batch (a smaller
    slice of the same length mix, its pool sized by the same rule).
    """
    w = WORKLOADS[name]
    if block_size is not None and block_size != w.block_size:
        w = Workload(w.name, w.dtype, w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, block_size,
                     w.partition_size, w.seed, w.notes, w.extra, w.recipe)
    seed = w.seed if seed is None else seed
    rng = np.random.default_rng(seed)
    lens = context_lengths(w, rng, gqa_sigma) if lens_override is None else np.asarray(lens_override, np.int64)
    if num_seqs is not None:
        lens = lens[:num_seqs]
    need = sum((int(n) + w.block_size - 1) // w.block_size for n in lens)
    nb = pool_blocks(w, need)
    tables, _ = place_blocks(lens, w.block_size, nb, rng, shuffle=shuffle)
    S, Hq, Hkv, hd, bs = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size
    S = len(lens)
    if w.kind == "tiny_f32":
        # four writes to distinct random slots of the 32-block pool
        slots = rng.choice(nb * bs, size=4, replace=False).astype(np.int64)
    else:
        slots = new_token_slots(lens, tables, bs)
    T = len(slots)
    k_cache = randn((nb, Hkv, bs, hd), w.dtype, seed * 1000 + 1, device)
    v_cache = randn((nb, Hkv, bs, hd), w.dtype, seed * 1000 + 2, device)
    q = randn((S, Hq, hd), w.dtype, seed * 1000 + 3, device)
    k_new = randn((T, Hkv, hd), w.dtype, seed * 1000 + 4, device)
    v_new = randn((T, Hkv, hd), w.dtype, seed * 1000 + 5, device)
    return dict(
        workload=w, q=q, k_cache=k_cache, v_cache=v_cache,
        block_tables=torch.from_numpy(tables).to(device),
        context_lens=torch.from_numpy(lens.astype(np.int32)).to(device),
        k_new=k_new, v_new=v_new, slot_mapping=torch.from_numpy(slots).to(device),
        lens=lens, tables=tables, num_blocks=nb, scale=w.scale,
        max_context_len=int(lens.max()) if len(lens) else 0,
    )


def prefix_share_layout(seed: int | None = None) -> dict:
    """Structure of the prefix-sharing workload: 25 sampled pairs, one shared
    2048-token prefix, a per-pair shared suffix of uniform 0..512 tokens."""
    w = WORKLOADS["prefix_share"]
    rng = np.random.default_rng(w.seed if seed is None else seed)
    suffix = rng.integers(0, 512, size=w.num_seqs // 2, endpoint=True).astype(np.int64)
    prefix = 2048
    need = prefix // w.block_size + int(sum(-(-int(u) // w.block_size) for u in suffix))
    return dict(workload=w, prefix_len=prefix, pair_suffix=suffix,
                num_blocks=need + 2 * len(suffix) + 16)


def fill_values(shape, dtype, seed, device) -> torch.Tensor:
    """Alias of randn for callers that fill pools built elsewhere."""
    return randn(shape, dtype, seed, device)
