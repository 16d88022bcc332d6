"""KV-memory utilisation of contiguous reservation vs on-demand paging over a
continuous batch, simulated on the host with the library's block manager.

What is compared (the pages' framing):
- "PagedAttention" (ayinedjimi-consultants.fr), "Definition", and the
  analyticslegends.ai sheet, "Pourquoi c'est important": engines before paging
  reserved, at admission, one contiguous region sized for the maximum length,
  and most of it stayed unused for requests of varied lengths.
- The same sheet and "PagedAttention et RadixAttention" (aitalk.it), step
  three: with paging, fixed-size blocks are allocated as a sequence grows and
  released block by block when it ends, so a sequence wastes less than one
  block.

The simulation admits requests in arrival order while memory allows (first
come, first served, no preemption), grows every running request by one token
per step, and releases a request when it has produced its output.  The
contiguous allocator must reserve ``max_len`` slots per request at admission;
the paged allocator reserves the prompt's blocks at admission and one block
whenever a sequence crosses a block boundary (a request is admitted only if
the pool can also hold one more block per running request, so that growth never
stalls).  Both see the same memory budget (in token slots) and the same
request stream.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import binding


@dataclass
class SimResult:
    steps: int
    mean_running: float
    mean_utilisation: float      # tokens held / slots reserved, averaged over steps with work
    peak_running: int
    finished: int


def request_stream(num_requests: int, seed: int = 0, max_len: int = 32768):
    """Prompt and output lengths for a mixed-length workload: prompts uniform in
    16..max_len/2, outputs uniform in 16..1024, capped so prompt + output <=
    max_len."""
    rng = np.random.default_rng(seed)
    prompts = rng.integers(16, max_len // 2, size=num_requests, endpoint=True)
    outputs = rng.integers(16, 1024, size=num_requests, endpoint=True)
    outputs = np.minimum(outputs, max_len - prompts)
    return prompts.astype(np.int64), outputs.astype(np.int64)


def simulate_contiguous(prompts, outputs, budget_slots: int, max_len: int, max_steps: int = 10**7) -> SimResult:
    waiting = list(range(len(prompts)))
    running = {}                      # id -> tokens held
    done, step, util_sum, run_sum, busy, peak = 0, 0, 0.0, 0, 0, 0
    while (waiting or running) and step < max_steps:
        while waiting and (len(running) + 1) * max_len <= budget_slots:
            r = waiting.pop(0)
            running[r] = int(prompts[r])
        if not running:
            raise ValueError("budget smaller than one request's reservation")
        for r in list(running):
            running[r] += 1
            if running[r] >= prompts[r] + outputs[r]:
                del running[r]
                done += 1
        step += 1
        if running:
            busy += 1
            util_sum += sum(running.values()) / (len(running) * max_len)
            run_sum += len(running)
            peak = max(peak, len(running))
    return SimResult(step, run_sum / max(busy, 1), util_sum / max(busy, 1), peak, done)


def simulate_paged(prompts, outputs, budget_slots: int, block_size: int, max_steps: int = 10**7,
                   check=None) -> SimResult:
    """Same stream through the library's block manager (pa_bm_*).  ``check`` is
    called after every step with (block_manager, {id: tokens}) for tests."""
    num_blocks = budget_slots // block_size
    bm = binding.BlockManager(num_blocks, block_size)
    waiting = list(range(len(prompts)))
    running = {}
    done, step, util_sum, run_sum, busy, peak = 0, 0, 0.0, 0, 0, 0
    try:
        while (waiting or running) and step < max_steps:
            while waiting:
                r = waiting[0]
                need = -(-int(prompts[r]) // block_size)
                if need + len(running) + 1 > bm.num_free():
                    break
                bm.add_seq(r, int(prompts[r]))
                running[r] = int(prompts[r])
                waiting.pop(0)
            if not running:
                raise ValueError("budget smaller than one request's prompt")
            for r in list(running):
                bm.append_slot(r)
                running[r] += 1
                if running[r] >= prompts[r] + outputs[r]:
                    bm.free_seq(r)
                    del running[r]
                    done += 1
            step += 1
            if check is not None:
                check(bm, running)
            if running:
                busy += 1
                held = sum(running.values())
                util_sum += held / ((num_blocks - bm.num_free()) * block_size)
                run_sum += len(running)
                peak = max(peak, len(running))
    finally:
        bm.close()
    return SimResult(step, run_sum / max(busy, 1), util_sum / max(busy, 1), peak, done)
