"""Byte and memory accounting for a paged KV cache, written as plain definitions.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources:
- "PagedAttention et RadixAttention : parlons de KV Cache" (aitalk.it), opening
  section: a Llama-3.1-70B cache in bf16 costs roughly 0.31 MB per token, so a
  128k-token context needs about 40 GB.
- "PagedAttention" (ayinedjimi-consultants.fr), "Definition", and the
  analyticslegends.ai concept sheet, "Points cles": contiguous allocation sized
  to the maximum length wastes 60-80% of the cache; with fixed-size blocks of
  16 or 32 tokens allocated on demand, a sequence wastes less than one block
  (utilisation above 96%).
- analyticslegends.ai concept sheet, "Points cles": a 2k-token system prompt
  shared by 50 requests is stored once instead of once per request.
"""
from __future__ import annotations


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    """Bytes of K plus V that one token adds to the cache across all layers."""
    return num_layers * num_kv_heads * head_dim * 2 * elem_bytes


def blocks_for_tokens(num_tokens: int, block_size: int) -> int:
    """Physical blocks a sequence of num_tokens occupies (the last may be partial)."""
    return -(-num_tokens // block_size) if num_tokens > 0 else 0


def paged_slack_tokens(context_lens, block_size: int) -> int:
    """Token slots allocated but unused when every sequence holds whole blocks."""
    return sum(blocks_for_tokens(n, block_size) * block_size - n for n in context_lens)


def contiguous_slack_tokens(context_lens, max_len: int) -> int:
    """Token slots unused when every sequence reserves max_len slots up front."""
    return sum(max_len - n for n in context_lens)


def shared_prefix_blocks(prefix_len: int, private_lens, block_size: int) -> int:
    """Blocks held by requests that share one prefix (stored once) and own their
    private suffixes; the prefix must end on a block boundary to be shareable
    without a copy."""
    if prefix_len % block_size:
        raise ValueError("prefix must fill whole blocks")
    return prefix_len // block_size + sum(blocks_for_tokens(u, block_size) for u in private_lens)


def decode_algorithmic_bytes(context_lens, num_q_heads: int, num_kv_heads: int, head_dim: int,
                             block_size: int, kv_elem: int, q_elem: int, out_elem: int) -> int:
    """Bytes one decode-attention call must move at minimum: the K and V rows of
    every attended token, q, the output, the used block-table entries and the
    context lengths."""
    kv = sum(context_lens) * num_kv_heads * head_dim * 2 * kv_elem
    qo = len(context_lens) * num_q_heads * head_dim * (q_elem + out_elem)
    tables = sum(blocks_for_tokens(n, block_size) for n in context_lens) * 4
    return kv + qo + tables + len(context_lens) * 4

