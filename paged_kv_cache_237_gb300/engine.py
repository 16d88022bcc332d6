"""One decode step of one layer over a paged KV cache, built from the C-ABI
calls: copy-on-write block copies, the new tokens' cache writes, then decode
attention, all enqueued on one stream in that order.

This follows the order the pages give for a shared block ("PagedAttention",
robocikowo.com, "Jak dziala": a write into a shared block triggers the copy;
"PagedAttention et RadixAttention : parlons de KV Cache", aitalk.it, fourth
step) and the reading that a step writes its token before attending over every
token present.
"""
from __future__ import annotations

import torch

from . import binding
from .workloads import WORKLOADS, prefix_share_layout, randn


class DecodeStep:
    """Holds the device buffers a repeated decode step needs (output,
    split-K workspace, status word) so that the timed calls allocate nothing.

    The workspace is zeroed once here, so the calls skip the per-call reset of
    its work counter (every completed call leaves the counter zero).  Steps
    that run one after another on one stream may share a workspace and a
    status word: pass them in."""

    def __init__(self, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                 max_context_len: int, partition_size: int = 0, simt: bool = False,
                 workspace: torch.Tensor | None = None, status: binding.DeviceStatus | None = None):
        self.q, self.k_cache, self.v_cache = q, k_cache, v_cache
        self.block_tables, self.context_lens = block_tables, context_lens
        self.scale = scale
        self.max_context_len = max_context_len
        self.partition_size = partition_size
        self.simt = simt
        self.out = torch.empty_like(q)
        S, Hq, hd = q.shape
        ws = binding.pa_decode_workspace_size(S, Hq, hd, max_context_len, partition_size)
        if workspace is not None and workspace.numel() < ws:
            raise ValueError(f"workspace has {workspace.numel()} bytes, {ws} needed")
        if workspace is None and ws:
            workspace = torch.zeros(ws, dtype=torch.uint8, device=q.device)
        self.workspace = workspace if ws else None
        self.status = status if status is not None else binding.DeviceStatus(q.device)

    def decode(self, stream=None, phase: int = binding.PA_PHASE_ALL, k_new=None, v_new=None,
               slot_mapping=None) -> torch.Tensor:
        return binding.pa_decode(self.out, self.q, self.k_cache, self.v_cache, self.block_tables,
                                 self.context_lens, self.scale, max_context_len=self.max_context_len,
                                 partition_size=self.partition_size, workspace=self.workspace,
                                 status=self.status, stream=stream, phase=phase, k_new=k_new,
                                 v_new=v_new, slot_mapping=slot_mapping, simt=self.simt,
                                 skip_counter_reset=True)

    def run_fused(self, k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                  cow_pairs: torch.Tensor | None = None, stream=None,
                  phase: int = binding.PA_PHASE_ALL) -> torch.Tensor:
        """Copy-on-write copies, then one decode launch that also writes each
        sequence's new token (one token per sequence, slot of its last position)."""
        if cow_pairs is not None and cow_pairs.numel() and phase != binding.PA_PHASE_REDUCE:
            binding.pa_copy_blocks(self.k_cache, self.v_cache, cow_pairs, status=self.status, stream=stream)
        return self.decode(stream, phase, k_new, v_new, slot_mapping)

    def write_tokens(self, k_new, v_new, slot_mapping, cow_pairs=None, stream=None) -> None:
        """The step's cache updates: copy-on-write copies, then the new rows."""
        if cow_pairs is not None and cow_pairs.numel():
            binding.pa_copy_blocks(self.k_cache, self.v_cache, cow_pairs, status=self.status, stream=stream)
        if slot_mapping.numel():
            binding.pa_reshape_and_cache(k_new, v_new, self.k_cache, self.v_cache, slot_mapping,
                                         status=self.status, stream=stream)

    def run(self, k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
            cow_pairs: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        self.write_tokens(k_new, v_new, slot_mapping, cow_pairs, stream)
        return self.decode(stream)


def prefix_share_state(device="cuda", seed: int | None = None) -> dict:
    """The prefix-sharing workload driven through the host block manager.

    One root holds a 2048-token prompt; each of 25 pairs forks it, grows a
    pair suffix (uniform 0..512 tokens) and forks again, so the pair shares
    its partial last block; the root is then dropped (prompt refcount 50).  The
    decode step appends one token to each of the 50 sequences: the first of a
    pair whose last block is partial triggers a copy-on-write.
    Returns host-side step inputs (slots, copy pairs, tables, lengths) and
    device tensors (caches, q, new K/V).
    """
    lay = prefix_share_layout(seed)
    w = lay["workload"]
    bs, nb = w.block_size, lay["num_blocks"]
    bm = binding.BlockManager(nb, bs)
    root = 1 << 20
    bm.add_seq(root, lay["prefix_len"])
    for p, u in enumerate(lay["pair_suffix"].tolist()):
        a, b = 2 * p, 2 * p + 1
        bm.fork(root, a)
        for _ in range(u):
            _, src, _ = bm.append_slot(a)
            assert src < 0, "a fresh suffix never needs a copy"
        bm.fork(a, b)
    bm.free_seq(root)
    seqs = list(range(w.num_seqs))
    prompt_blocks = bm.block_table(0)[: lay["prefix_len"] // bs]
    slots, pairs = bm.append_slots(seqs)
    max_blocks = max(len(bm.block_table(s)) for s in seqs)
    tables, lens = bm.build_tables(seqs, max_blocks)
    s0 = (w.seed if seed is None else seed) * 1000
    Hkv, hd = w.num_kv_heads, w.head_dim
    return dict(
        workload=w, block_manager=bm, num_blocks=nb, prompt_blocks=prompt_blocks,
        slots=slots, pairs=pairs, tables=tables, lens=lens,
        k_cache=randn((nb, Hkv, bs, hd), w.dtype, s0 + 1, device),
        v_cache=randn((nb, Hkv, bs, hd), w.dtype, s0 + 2, device),
        q=randn((w.num_seqs, w.num_q_heads, hd), w.dtype, s0 + 3, device),
        k_new=randn((w.num_seqs, Hkv, hd), w.dtype, s0 + 4, device),
        v_new=randn((w.num_seqs, Hkv, hd), w.dtype, s0 + 5, device),
        scale=w.scale, max_context_len=int(lens.max()),
    )


__all__ = ["DecodeStep", "prefix_share_state", "WORKLOADS"]
