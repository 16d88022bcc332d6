"""Byte accounting pinned to figures the pages print.

Golden files under tests/golden/ carry the page figure and its source.
"""
import json
import os

import numpy as np
import pytest

from oracle import accounting as acc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_llama31_70b_bytes_per_token_matches_page():
    g = load("kv_bytes_llama31_70b.json")
    m = g["model_shape"]
    b = acc.kv_bytes_per_token(m["num_layers"], m["num_kv_heads"], m["head_dim"], m["elem_bytes"])
    assert b == 327680                       # 80 * 8 * 128 * 2 (K and V) * 2 bytes
    mib = b / 2**20
    assert abs(mib - g["page_values"]["mb_per_token"]) / g["page_values"]["mb_per_token"] < 0.02
    gib = b * g["page_values"]["context_tokens"] / 2**30
    assert abs(gib - g["page_values"]["gb_for_context"]) / g["page_values"]["gb_for_context"] < 0.03
    # one layer: 4096 bytes per token
    assert acc.kv_bytes_per_token(1, 8, 128, 2) == 4096


def test_shared_prompt_is_stored_once():
    g = load("prefix_sharing_50x2k.json")
    n, p = g["page_values"]["requests"], g["page_values"]["prefix_tokens"]
    rng = np.random.default_rng(0)
    private = rng.integers(0, 513, size=n).tolist()
    shared = acc.shared_prefix_blocks(p, private, 16)
    unshared = sum(acc.blocks_for_tokens(p + u, 16) for u in private)
    assert unshared - shared == (n - 1) * (p // 16)
    assert shared == 128 + sum(acc.blocks_for_tokens(u, 16) for u in private)


def test_paged_slack_is_below_one_block_per_sequence():
    rng = np.random.default_rng(1)
    lens = rng.integers(1, 32768, size=500).tolist()
    for bs in (16, 32):
        slack = acc.paged_slack_tokens(lens, bs)
        assert 0 <= slack < bs * len(lens)
        # utilisation above 96% once sequences are long against the block size
        assert sum(lens) / (sum(lens) + slack) > 0.96


def test_contiguous_reservation_wastes_most_of_the_cache_for_mixed_lengths():
    """Reserving the maximum length per request leaves most slots unused when
    lengths are spread out (the pages quote 60-80% waste)."""
    rng = np.random.default_rng(2)
    lens = rng.integers(16, 32768, size=40).tolist()
    waste = acc.contiguous_slack_tokens(lens, 131072) / (40 * 131072)
    assert 0.6 < waste < 1.0


def test_decode_bytes_hand_computed():
    # lens 7 and 16, Hq 4, Hkv 2, hd 64, bs 16, bf16 everywhere:
    # K/V 23*2*64*2*2 = 11776; q+out 2*4*64*(2+2) = 2048; tables 2*4 = 8; lens 8
    assert acc.decode_algorithmic_bytes([7, 16], 4, 2, 64, 16, 2, 2, 2) == 13840
