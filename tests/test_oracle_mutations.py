"""Planted mistakes in a copy of the oracle must be caught by its pins.

Each case copies ``oracle/paged_ref.c``, plants one plausible mistake (a wrong
head mapping, a shifted slot, a swapped layout, a dropped scale or
normalisation, keys read from the value cache, a transposed query index),
compiles the copy into a temporary directory and runs the contiguous-attention
pin (torch SDPA on the same data, fp64) against it.  The unmodified copy must
pass and every mutant must fail.  Nothing here touches the real oracle build.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from test_oracle_pins import place_contiguous, rand_case, sdpa_reference

SRC = os.path.join(os.path.dirname(oracle.__file__), "paged_ref.c")

MUTANTS = {
    "gqa_mapping": ("int kv = h / group;", "int kv = h % j->num_kv_heads;"),
    "slot_shift": ("* bs + (t % bs)) * hd;", "* bs + ((t + 1) % bs)) * hd;"),
    "block_index": ("int32_t phys = table[t / bs];", "int32_t phys = table[t % bs];"),
    "layout_swap": ("(((int64_t)phys * num_kv_heads + kv_head) * bs + (t % bs)) * hd",
                    "(((int64_t)phys * bs + (t % bs)) * num_kv_heads + kv_head) * hd"),
    "dropped_scale": ("s[t] = scale * acc;", "s[t] = acc;"),
    "no_normalisation": ("double p = s[t] / denom;", "double p = s[t];"),
    "keys_from_values": ("acc += q[d] * K[(int64_t)t * hd + d];",
                         "acc += q[d] * V[(int64_t)t * hd + d];"),
    "short_context": ("attend_contiguous(j->out + row, j->q + row, K, V, n, hd,",
                      "attend_contiguous(j->out + row, j->q + row, K, V, n > 1 ? n - 1 : n, hd,"),
    "query_transposed": ("int64_t row = ((int64_t)i * j->num_q_heads + h) * hd;",
                         "int64_t row = ((int64_t)h * j->num_seqs + i) * hd;"),
}


def pin_battery(lib) -> bool:
    """True when the library passes the contiguous-equivalence pin."""
    lens = [1, 17, 33, 40]
    Hq, Hkv, hd, bs = 8, 2, 64, 16
    q, K, V = rand_case(77, lens, Hq, Hkv, hd, torch.float32)
    need = sum(-(-n // bs) for n in lens)
    perm = np.random.default_rng(5).permutation(need + 3)
    kc, vc, tables = place_contiguous(K, V, bs, need + 3, perm, torch.float32)
    kc = torch.nan_to_num(kc, nan=1e3)   # defined values in unused slots
    vc = torch.nan_to_num(vc, nan=1e3)
    scale = 1.0 / math.sqrt(hd)
    try:
        out = oracle.paged_decode(q, kc, vc, tables, torch.tensor(lens, dtype=torch.int32), scale,
                                  threads=1, lib=lib)
    except ValueError:
        return False
    for i in range(len(lens)):
        ref = sdpa_reference(q[i], K[i], V[i], scale)
        if not torch.allclose(out[i], ref, rtol=0, atol=1e-12):
            return False
    return True


def build_variant(tmp_path, name, edit):
    text = open(SRC).read()
    if edit is not None:
        old, new = edit
        assert text.count(old) == 1, f"mutation anchor for {name} not found exactly once"
        text = text.replace(old, new)
    src = tmp_path / f"{name}.c"
    src.write_text(text)
    so = tmp_path / f"lib{name}.so"
    oracle.build_oracle(force=True, out_path=str(so), source=str(src))
    return oracle.load(str(so))


def test_unmodified_copy_passes(tmp_path):
    assert pin_battery(build_variant(tmp_path, "clean", None))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    assert not pin_battery(build_variant(tmp_path, name, MUTANTS[name]))
