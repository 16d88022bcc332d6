#!/usr/bin/env python
"""Paged decode attention benchmark on one node (one process per GPU).

A step is one layer of one decode step for the whole batch: the new tokens'
K/V written into their slots (plus copy-on-write block copies when the batch
shares blocks), the per-partition decode pass, and the split-K merge.  The
default workload is the long-context continuous batch (256 sequences, 8 at
131072 tokens, 248 uniform in 16..32768; 64 query / 8 KV heads, head_dim 128,
block_size 32, bf16, partitions of 512); its K/V (~21 GB) is far larger than
L2, so no flush is needed between steps.  Smaller workloads get an L2 flush
(a 512 MB write) between timed steps, outside the timed events.

Metric: paged decode attention KV GB/s = algorithmic bytes of the decode call
(K and V rows of every attended token, q, output, used block-table entries,
context lengths) / step time; plus sequence-layer decode steps/s.

``--impl reference`` times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (there is no other reference implementation).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "paged decode attention KV GB/s (% of GB300 HBM peak); seq-layer decode steps/s"
L2_BYTES = 129 * 2**20

# DRAM read+write bytes of one partition-pass launch (with the fused cache
# write), per workload, from ncu's dram__bytes_read.sum + dram__bytes_write.sum
# on one launch.  Captures stay small (a few GB on the device): the GQA batch is
# captured whole (0.9 GB of K/V); the long-context figure is a capture of a
# seeded slice of the same length mix (--num-seqs), scaled to the full launch
# by the ratio of algorithmic bytes.  Valid only while the kernel source is
# the one captured.
TRAFFIC_CAPTURE = {"source_sha256_prefix": "d2092055b73d411c",
                   # 48-sequence slice: 4,143,338,496 B read + 26,150,400 B written
                   # over 4,141,526,704 algorithmic bytes, scaled to 20,791,665,640
                   "bytes_per_launch": {"long_context": 20932043957,
                                        "gqa_llama3_70b": 902361344 + 6061312}}


KERNEL_FILES = ("pa_decode.cu", "pa_decode_common.cuh", "pa_internal.h")


def kernel_source(*texts: bytes) -> bytes:
    """The code the bf16 partition pass is built and launched from
    (pa_decode.cu, pa_decode_common.cuh and pa_internal.h: kernels, helpers,
    launch shapes), with comments and whitespace removed so that only code
    changes count."""
    import re
    out = []
    for text in texts:
        code = re.sub(rb"/\*.*?\*/", b"", text, flags=re.S)
        code = re.sub(rb"//[^\n]*", b"", code)
        out.append(re.sub(rb"\s+", b" ", code).strip())
    return b"\n".join(out)


def captured_traffic(workload: str):
    """Measured DRAM bytes of one partition-pass launch of `workload`, or None
    when there is no capture of it or the kernel changed since."""
    import hashlib
    csrc = os.path.join(ROOT, "paged_kv_cache_237_gb300", "csrc")
    try:
        texts = []
        for name in KERNEL_FILES:
            with open(os.path.join(csrc, name), "rb") as f:
                texts.append(f.read())
        digest = hashlib.sha256(kernel_source(*texts)).hexdigest()[:16]
    except OSError:
        return None
    c = TRAFFIC_CAPTURE
    if digest != c["source_sha256_prefix"] or workload not in c["bytes_per_launch"]:
        return None
    return int(c["bytes_per_launch"][workload])


# ------------------------------------------------------------ accounting ---
def decode_bytes(lens, num_q_heads, num_kv_heads, head_dim, block_size, kv_elem, q_elem, out_elem):
    """Minimum bytes one decode call moves: K and V rows of every attended
    token, q, the output, used block-table entries and the context lengths."""
    lens = [int(n) for n in lens]
    kv = sum(lens) * num_kv_heads * head_dim * 2 * kv_elem
    qo = len(lens) * num_q_heads * head_dim * (q_elem + out_elem)
    tables = sum(-(-n // block_size) for n in lens) * 4
    return kv + qo + tables + 4 * len(lens)


def decode_bytes_pages(lens, num_q_heads, num_kv_heads, head_dim, block_size, kv_elem, q_elem, out_elem):
    """decode_bytes with K/V counted by whole pages: every used block's
    block_size rows, so a partial last block counts in full (secondary)."""
    lens = [int(n) for n in lens]
    pages = sum(-(-n // block_size) for n in lens)
    return (decode_bytes(lens, num_q_heads, num_kv_heads, head_dim, block_size, kv_elem, q_elem, out_elem)
            + (pages * block_size - sum(lens)) * num_kv_heads * head_dim * 2 * kv_elem)


def partition_pass_bytes(lens, num_q_heads, num_kv_heads, head_dim, block_size, kv_elem, q_elem):
    """Algorithmic bytes of the per-partition pass alone: K/V rows, q, table
    entries, lengths (its partial/output writes are not counted)."""
    lens = [int(n) for n in lens]
    return (sum(lens) * num_kv_heads * head_dim * 2 * kv_elem
            + len(lens) * num_q_heads * head_dim * q_elem
            + sum(-(-n // block_size) for n in lens) * 4 + 4 * len(lens))


NOMINAL_HBM_GBPS = 7900.0     # GB300 HBM3e, datasheet figure


def fractions(gbps: float, peak: float) -> dict:
    """A bandwidth as a fraction of the measured copy peak (the roofline
    denominator; a read-only stream may exceed it, since a copy also writes)
    and of the datasheet HBM bandwidth."""
    return {"of_measured_copy_peak": round(gbps / peak, 4),
            "of_datasheet_7900_GBps": round(gbps / NOMINAL_HBM_GBPS, 4)}


def load_peak():
    """(HBM copy peak in GB/s, 'measured' | 'fallback')."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
        return float(peaks["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return 6800.0, "fallback"


# ---------------------------------------------------------------- clocks ---
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            if uuid:
                cmd += ["-i", uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"]
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- workloads ---
def build_workload(name: str, device, seed_offset: int, gqa_sigma: float = 1.0, num_seqs=None):
    from paged_kv_cache_237_gb300 import engine, workloads
    if name == "prefix_share":
        if num_seqs is not None:
            raise ValueError("--num-seqs does not apply to the prefix-sharing batch")
        st = engine.prefix_share_state(device, seed=workloads.WORKLOADS[name].seed + seed_offset)
        w = st["workload"]
        d = dict(workload=w, q=st["q"], k_cache=st["k_cache"], v_cache=st["v_cache"],
                 block_tables=st["tables"].to(device), context_lens=st["lens"].to(device),
                 k_new=st["k_new"], v_new=st["v_new"], slot_mapping=st["slots"].to(device),
                 cow_pairs=st["pairs"].to(device), lens=st["lens"].numpy(), scale=st["scale"],
                 max_context_len=st["max_context_len"])
    else:
        d = workloads.decode_inputs(name, device=device, seed=workloads.WORKLOADS[name].seed + seed_offset,
                                    gqa_sigma=gqa_sigma, num_seqs=num_seqs)
        d["cow_pairs"] = None
    return d


def combine_ranks(ms_local: float, bytes_local: int, dist=None, device="cpu"):
    """Step time and bytes for the whole job: the slowest rank's time (MAX)
    and every rank's bytes (SUM).  Without a process group, the local values."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return ms_local, bytes_local
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    b = torch.tensor([float(bytes_local)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), int(b.item())


def workload_config(w, d, world: int, gqa_sigma: float = 1.0) -> dict:
    """The `config` object of the JSON line (the same for both arms)."""
    lens = d["lens"]
    elem = torch.tensor([], dtype=w.dtype).element_size()
    working_set = d["k_cache"].numel() * elem * 2
    extra = {"lognormal_sigma": gqa_sigma} if w.name == "gqa_llama3_70b" else {}
    return {
        "workload": w.name, **extra,
        "num_seqs": len(lens), "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
        "head_dim": w.head_dim, "block_size": w.block_size, "partition_size": w.partition_size,
        "total_context_tokens": int(sum(int(n) for n in lens)),
        "max_context_len": int(d["max_context_len"]),
        "bytes_per_step": decode_bytes(lens, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                       elem, elem, elem),
        "l2": "inputs larger than L2 (no flush)" if working_set > 2 * L2_BYTES
              else "512 MB L2 flush between steps",
        "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
    }


def flush_l2(buf):
    if buf is not None:
        buf.add_(1)


# ------------------------------------------------------------- CPU legs ---
def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(d, seqs):
    """Host copies of the blocks the sampled sequences use (gathered with torch
    indexing on the device), ready for the oracle."""
    bs = d["k_cache"].shape[2]
    lens = d["lens"]
    tab = d["block_tables"].cpu().numpy()
    rows = [tab[s, :-(-int(lens[s]) // bs)] for s in seqs]
    uniq = np.unique(np.concatenate(rows)) if rows else np.zeros(0, np.int64)
    remap = {int(b): i for i, b in enumerate(uniq)}
    idx = torch.from_numpy(uniq.astype(np.int64)).to(d["k_cache"].device)
    kc = d["k_cache"].index_select(0, idx).cpu()
    vc = d["v_cache"].index_select(0, idx).cpu()
    t = np.full((len(seqs), max(1, max(len(r) for r in rows))), -1, np.int32)
    for i, r in enumerate(rows):
        t[i, :len(r)] = [remap[int(b)] for b in r]
    q = d["q"][list(seqs)].cpu()
    return q, kc, vc, torch.from_numpy(t), torch.tensor([int(lens[s]) for s in seqs], dtype=torch.int32)


def time_oracle(d, seqs, threads):
    import oracle
    q, kc, vc, t, ln = oracle_sample(d, seqs)
    t0 = time.perf_counter()
    oracle.paged_decode(q, kc, vc, t, ln, d["scale"], threads=threads)
    return time.perf_counter() - t0


def pick_sample(d, target_s: float, threads: int):
    """Sequences (seeded random order) whose oracle time is about target_s.
    The rate per token comes from one probe sequence, then from one timed run
    of the picked sample if that overshoots by more than a quarter."""
    lens = d["lens"]
    rng = np.random.default_rng(1234)
    order = [int(i) for i in rng.permutation(len(lens))]

    def pick(per_token):
        budget = target_s / per_token
        seqs, tok = [], 0
        for s in order:
            if tok + int(lens[s]) > budget and seqs:
                continue
            seqs.append(s)
            tok += int(lens[s])
            if tok >= 0.9 * budget:
                break
        return seqs, tok

    probe = order[:1]
    dt = max(time_oracle(d, probe, threads), 1e-4)
    seqs, tok = pick(dt / max(1, int(lens[probe[0]])))
    if len(seqs) > 1:
        dt = time_oracle(d, seqs, threads)
        if dt > 1.25 * target_s:
            seqs, _ = pick(dt / max(1, tok))
    return seqs


def sample_kv_bytes(d, seqs):
    w = d["workload"]
    e = torch.tensor([], dtype=w.dtype).element_size()
    return decode_bytes([d["lens"][s] for s in seqs], w.num_q_heads, w.num_kv_heads, w.head_dim,
                        w.block_size, e, e, e)


# ------------------------------------------------------------------ main ---
def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long_context",
                    choices=["tiny_f32", "mha_llama2_7b", "gqa_llama3_70b", "prefix_share", "long_context",
                             "mha_llama2_7b_f32", "gqa_llama3_70b_f32"])
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="keep only the first N sequences of the drawn batch (a smaller slice of the same "
                         "length mix, for profiler captures)")
    ap.add_argument("--profile", action="store_true",
                    help="run the warm-up steps and one more step of the workload, print nothing and exit: "
                         "a short program for profiler captures (the last step's partition pass is launch "
                         "number 2 * (warmup + 1) of decode_*_kernel and the merge kernel together)")
    ap.add_argument("--gqa-sigma", type=float, default=1.0,
                    help="log-space spread of the GQA batch's lognormal lengths (1.0; 0.5 is the sensitivity case)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target oracle time of the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the same-run measurements of the other workloads and of the placement, cache-op, "
                         "prefix-cache and swap studies")
    ap.add_argument("--simt", action="store_true",
                    help="bf16 products on plain fp32 FMAs (SIMT kernel) instead of tensor-core MMAs")
    ap.add_argument("--unfused", action="store_true",
                    help="write the new tokens with a separate pa_reshape_and_cache launch instead of inside "
                         "the decode launch")
    ap.add_argument("--study", choices=["placement", "prefix_cache", "swap", "mma", "cache_ops"], default=None,
                    help="instead of the benchmark line, print one study line: 'placement' times the partition "
                         "pass with shuffled vs identity block placement at block sizes 32 and 16; "
                         "'prefix_cache' admits a multi-tenant batch through the chained-key prefix cache and "
                         "times its decode step; 'swap' times block copies between the device cache and pinned "
                         "host memory; 'mma' times the bf16 partition pass on tensor-core MMAs vs SIMT FMAs; "
                         "'cache_ops' times the cache write and the block copy at step and streaming sizes")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.study == "placement":
        run_placement_study(args)
        return
    if args.study == "prefix_cache":
        run_prefix_cache_study(args)
        return
    if args.study == "swap":
        run_swap_study(args)
        return
    if args.study == "cache_ops":
        run_cache_ops_study(args)
        return
    if args.study == "mma":
        run_mma_study(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist  # noqa: F811
        if torch.cuda.is_available():
            torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")

    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        if dist is not None:
            dist.destroy_process_group()
        return

    from paged_kv_cache_237_gb300 import build as pa_build
    pa_build.build()
    from paged_kv_cache_237_gb300 import binding
    from paged_kv_cache_237_gb300.engine import DecodeStep

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    d = build_workload(args.workload, device, seed_offset=rank, gqa_sigma=args.gqa_sigma, num_seqs=args.num_seqs)
    w = d["workload"]
    elem = torch.tensor([], dtype=w.dtype).element_size()
    lens = d["lens"]
    B = decode_bytes(lens, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, elem, elem, elem)
    B_part = partition_pass_bytes(lens, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, elem, elem)
    step = DecodeStep(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"], d["scale"],
                      d["max_context_len"], w.partition_size, simt=args.simt)
    split = binding.pa_decode_workspace_size(len(lens), w.num_q_heads, w.head_dim, d["max_context_len"],
                                             w.partition_size) > 0
    stream = torch.cuda.current_stream(device)
    working_set = d["k_cache"].numel() * elem * 2
    flush = None if working_set > 2 * L2_BYTES else torch.empty(512 * 2**20 // 4, dtype=torch.float32,
                                                                  device=device)
    cow = d["cow_pairs"]

    # The fused launch writes each sequence's last position; a workload whose
    # writes go elsewhere (the tiny fp32 case writes 4 random slots) runs unfused.
    from paged_kv_cache_237_gb300.workloads import new_token_slots
    last_slots = new_token_slots(lens, d["block_tables"].cpu().numpy(), w.block_size)
    fused = (not args.unfused and d["slot_mapping"].numel() == len(lens)
             and bool(np.array_equal(last_slots, d["slot_mapping"].cpu().numpy())))
    new_tok = (d["k_new"], d["v_new"], d["slot_mapping"]) if fused else (None, None, None)

    def cache_updates(st):
        if fused:
            if cow is not None and cow.numel():
                binding.pa_copy_blocks(step.k_cache, step.v_cache, cow, status=step.status, stream=st)
        else:
            step.write_tokens(d["k_new"], d["v_new"], d["slot_mapping"], cow, st)

    def partition_pass(st):
        step.decode(st, binding.PA_PHASE_PARTITIONS, *new_tok)

    def merge(st):
        step.decode(st, binding.PA_PHASE_REDUCE)

    def one_step(st):
        cache_updates(st)
        partition_pass(st)
        merge(st)

    for _ in range(args.warmup):
        one_step(stream)
        flush_l2(flush)
    torch.cuda.synchronize(device)
    if step.status.read():
        raise RuntimeError("device status flagged an input error")
    if args.profile:
        one_step(stream)
        torch.cuda.synchronize(device)
        if step.status.read():
            raise RuntimeError("device status flagged an input error")
        if dist is not None:
            dist.destroy_process_group()
        return

    # The timed step is a CUDA graph of the step's launches (how a decode loop
    # runs in production): replays leave no host gaps between kernels, so the
    # events measure the GPU alone.  Single-phase graphs time the phases.
    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            fn(None)
        return g

    has_updates = (not fused and d["slot_mapping"].numel() > 0) or (cow is not None and cow.numel() > 0)
    g_step, g_part = capture(one_step), capture(partition_pass)
    g_merge = capture(merge) if split else None
    g_upd = capture(cache_updates) if has_updates else None

    def timed_replays(g, n):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in ev:
            a.record(stream)
            g.replay()
            b.record(stream)
            flush_l2(flush)
        torch.cuda.synchronize(device)
        return [a.elapsed_time(b) for a, b in ev]

    def back_to_back(g, n):
        """Mean time of n replays enqueued back to back between one pair of
        events: everything between the first step's start and the last one's
        end, launch gaps included (inputs larger than L2 only)."""
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize(device)
        return a.elapsed_time(b) / n

    K = args.steps
    for g in (g_step, g_part, g_merge, g_upd):
        if g is not None:
            timed_replays(g, 2)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(device)
    clocks = ClockSampler(local_rank)
    time.sleep(0.2)
    step_ms = timed_replays(g_step, K)
    # The K timed steps as the run contract brackets them: back to back between
    # one pair of events.  A workload that needs an L2 flush between steps
    # keeps the per-step events, which leave the flush outside.
    run_ms = back_to_back(g_step, K) if flush is None else statistics.mean(step_ms)
    clk = clocks.stop()
    if dist is not None:
        dist.barrier()
    part_ms = timed_replays(g_part, K)
    red_ms = timed_replays(g_merge, K) if g_merge is not None else [0.0]
    write_ms = timed_replays(g_upd, K) if g_upd is not None else [0.0]
    if step.status.read():
        raise RuntimeError("device status flagged an input error")
    # the same step launched eagerly from Python, for comparison
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in ev:
        a.record(stream)
        one_step(stream)
        b.record(stream)
        flush_l2(flush)
    torch.cuda.synchronize(device)
    eager_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    ms, B_job = combine_ranks(run_ms, B, dist, device)
    _, B_pages = combine_ranks(ms, decode_bytes_pages(lens, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                                      w.block_size, elem, elem, elem), dist, device)
    launches_per_step = (0 if fused or not d["slot_mapping"].numel() else 1) + 1 + (1 if split else 0) + \
        (1 if cow is not None and cow.numel() else 0)

    # ---- end to end through the public API, host buffers in pinned memory.
    # Each step copies its inputs (q, block tables, lengths, new K/V, slots,
    # copy pairs) from pinned host memory and reads its output back.  As in a
    # serving loop, two buffer sets alternate: step i+1's inputs are copied on a
    # side stream while step i computes, and step i's output is read back there
    # too; the timed region runs from the first input copy to the last read.
    hq = d["q"].cpu().pin_memory()
    htab = d["block_tables"].cpu().pin_memory()
    hlen = d["context_lens"].cpu().pin_memory()
    hk = d["k_new"].cpu().pin_memory()
    hv = d["v_new"].cpu().pin_memory()
    hslot = d["slot_mapping"].cpu().pin_memory()
    hcow = cow.cpu().pin_memory() if cow is not None and cow.numel() else None
    houts = [torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in (hq, htab, hlen, hk, hv, hslot)) + \
        (hcow.numel() * 8 if hcow is not None else 0)
    d2h = houts[0].numel() * houts[0].element_size()
    sets = []
    for j in range(2):
        # steps run one after another on one stream: they share the workspace and status word
        sj = DecodeStep(torch.empty_like(d["q"]), d["k_cache"], d["v_cache"], torch.empty_like(d["block_tables"]),
                        torch.empty_like(d["context_lens"]), d["scale"], d["max_context_len"], w.partition_size,
                        simt=args.simt, workspace=step.workspace, status=step.status)
        sets.append(dict(step=sj, k=torch.empty_like(d["k_new"]), v=torch.empty_like(d["v_new"]),
                         slots=torch.empty_like(d["slot_mapping"]),
                         cow=torch.empty_like(cow) if hcow is not None else None,
                         in_ready=torch.cuda.Event(), done=torch.cuda.Event()))
    copy_stream = torch.cuda.Stream(device)
    torch.cuda.synchronize(device)      # nothing allocated above is still being written by another stream

    def h2d_inputs(bs):
        st = bs["step"]
        st.q.copy_(hq, non_blocking=True)
        st.block_tables.copy_(htab, non_blocking=True)
        st.context_lens.copy_(hlen, non_blocking=True)
        bs["k"].copy_(hk, non_blocking=True)
        bs["v"].copy_(hv, non_blocking=True)
        bs["slots"].copy_(hslot, non_blocking=True)
        if hcow is not None:
            bs["cow"].copy_(hcow, non_blocking=True)
        bs["in_ready"].record(copy_stream)

    def e2e_loop(n):
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(copy_stream):
            start.record(copy_stream)
            h2d_inputs(sets[0])
        for i in range(n):
            cur, nxt = sets[i % 2], sets[(i + 1) % 2]
            stream.wait_event(cur["in_ready"])
            if fused:
                cur["step"].run_fused(cur["k"], cur["v"], cur["slots"], cur["cow"], stream)
            else:
                cur["step"].run(cur["k"], cur["v"], cur["slots"], cur["cow"], stream)
            cur["done"].record(stream)
            with torch.cuda.stream(copy_stream):
                if i + 1 < n:
                    if i >= 1:
                        copy_stream.wait_event(nxt["done"])     # step i-1 no longer reads these inputs
                    h2d_inputs(nxt)
                copy_stream.wait_event(cur["done"])
                houts[i % 2].copy_(cur["step"].out, non_blocking=True)
        with torch.cuda.stream(copy_stream):
            stop.record(copy_stream)
        torch.cuda.synchronize(device)
        return start.elapsed_time(stop) / n

    e2e_loop(max(args.warmup, 2))
    e2e_ms, _ = combine_ranks(e2e_loop(K), B, dist, device)
    if step.status.read():
        raise RuntimeError("device status flagged an input error")

    # ---- CPU baseline: the oracle as it stands, on a bounded sample
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = host_cores()
        seqs = pick_sample(d, args.cpu_seconds, threads)
        dt = time_oracle(d, seqs, threads)
        sb = sample_kv_bytes(d, seqs)
        one = pick_sample(d, min(3.0, args.cpu_seconds), 1)
        dt1 = time_oracle(d, one, 1)
        cpu = {"value": round(sb / dt / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"{len(seqs)} of {len(lens)} sequences ({int(sum(lens[s] for s in seqs))} tokens, "
                         f"all {w.num_q_heads} query heads) of the same workload, fp64 C oracle, "
                         f"{dt:.1f} s",
               "single_core_value": round(sample_kv_bytes(d, one) / dt1 / 1e9, 4),
               "single_core_sample": f"{len(one)} sequences, 1 thread, {dt1:.1f} s"}

    secondary = placement = cache_ops = prefix_cache = swap = None
    peak, peak_src = load_peak()
    if rank == 0 and world == 1 and args.workload == "long_context" and args.num_seqs is None \
            and not args.no_secondary:
        # every other workload's step, in the same run (the long-context batch is the line's own)
        n2 = max(args.steps, 100)
        secondary = {}
        for key, name, sigma in (("tiny_f32", "tiny_f32", 1.0), ("mha_llama2_7b", "mha_llama2_7b", 1.0),
                                 ("gqa_llama3_70b", "gqa_llama3_70b", 1.0),
                                 ("gqa_llama3_70b_sigma0.5", "gqa_llama3_70b", 0.5),
                                 ("prefix_share", "prefix_share", 1.0),
                                 ("mha_llama2_7b_f32", "mha_llama2_7b_f32", 1.0),
                                 ("gqa_llama3_70b_f32", "gqa_llama3_70b_f32", 1.0)):
            secondary[key] = measure_step(name, n2, gqa_sigma=sigma, peak=peak)
        # the pages' gather-overhead figures, measured on this kernel
        placement = placement_block("long_context", 40, args.warmup)
        # cache write and block copy at a decode step's size and at streaming sizes
        cache_ops = cache_ops_block(100, args.warmup, tokens=(256, 65536), pairs=(24, 2048))
        # prefix caching over a multi-tenant batch, and block swaps to pinned host memory
        prefix_cache = prefix_cache_block(100, args.warmup)
        swap = swap_block(20, args.warmup)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    part_avg = statistics.mean(part_ms)
    achieved = B_part / (part_avg * 1e-3) / 1e9
    value = B_job / (ms * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "ms_per_step_events_each": round(statistics.mean(step_ms), 4),
        "median_ms_per_step_events_each": round(statistics.median(step_ms), 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32",
        "data": "synthetic",
        "config": workload_config(w, d, world, args.gqa_sigma),
        "hbm_fraction": fractions(B / (ms * 1e-3) / 1e9, peak),
        "page_granular": {"bytes_per_step": B_pages, "GBps": round(B_pages / (ms * 1e-3) / 1e9, 2),
                          "what": "K/V counted by whole pages (partial last blocks in full)"},
        "seq_layer_steps_per_s": round(world * len(lens) / (ms * 1e-3), 1),
        "step": "copy-on-write copies + decode launch that also writes the new tokens + split-K merge" if fused
                else "copy-on-write copies + cache write + decode + split-K merge",
        "timing": ("CUDA graph of the step; K replays back to back between one pair of events" if flush is None
                   else "CUDA graph of the step; events around each replay, a 512 MB write between replays"),
        "eager_ms_per_step": round(eager_ms, 4),
        "phases_ms": {"cache_updates": round(statistics.mean(write_ms), 4),
                      "partition_pass": round(part_avg, 4), "split_k_reduce": round(statistics.mean(red_ms), 4)},
        "roofline": {"bound": "hbm", "kernel": "decode_bf16_kernel (partition pass)"
                     if w.dtype == torch.bfloat16 and not args.simt else "decode_simt_kernel (partition pass)",
                     "peak_what": "HBM copy bandwidth (read + write), so a read-only stream may exceed 1",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_src,
                     "bytes_per_launch": B_part,
                     "traffic": None if args.simt or args.unfused else captured_traffic(w.name)},
        "e2e": {"value": round(B_job / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "public Python API; pinned host inputs copied and output read back every step, "
                       "double-buffered so copies overlap the previous step's compute"},
        "gpu_launches": K * launches_per_step,
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    if cow is not None:
        # prefix sharing: K/V bytes of the distinct blocks the step reads
        bs = w.block_size
        tab = d["block_tables"].cpu().numpy()
        used = {int(b) for i, n in enumerate(lens) for b in tab[i, :-(-int(n) // bs)]}
        uniq = len(used) * w.num_kv_heads * bs * w.head_dim * 2 * elem
        line["unique_kv_bytes"] = uniq
        line["unique_kv_GBps"] = round(uniq / (ms * 1e-3) / 1e9, 1)
    if secondary is not None:
        line["secondary_workloads"] = secondary
    if placement is not None:
        line["placement"] = placement
    if cache_ops is not None:
        line["cache_ops"] = cache_ops
    if prefix_cache is not None:
        line["prefix_cache"] = prefix_cache
    if swap is not None:
        line["swap"] = swap
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def time_partition_pass(d, steps: int, warmup: int) -> float:
    """Mean CUDA-event time (ms) of the per-partition decode pass alone."""
    from paged_kv_cache_237_gb300 import binding
    from paged_kv_cache_237_gb300.engine import DecodeStep
    w = d["workload"]
    step = DecodeStep(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"], d["scale"],
                      d["max_context_len"], w.partition_size)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        step.decode(stream, binding.PA_PHASE_PARTITIONS)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        a.record(stream)
        step.decode(stream, binding.PA_PHASE_PARTITIONS)
        b.record(stream)
    torch.cuda.synchronize()
    if step.status.read():
        raise RuntimeError("device status flagged an input error")
    return statistics.mean(a.elapsed_time(b) for a, b in ev)


def placement_block(name: str, steps: int, warmup: int) -> dict:
    """Gather overhead and block-size trade-off on the same kernel: the
    partition pass over one workload's lengths with every sequence's blocks
    shuffled across the pool or laid out consecutively, at block size 32 and
    16 (CUDA events, mean of `steps` launches)."""
    from paged_kv_cache_237_gb300 import workloads
    rows = {}
    for bs in (32, 16):
        for shuffle in (True, False):
            d = workloads.decode_inputs(name, device="cuda", shuffle=shuffle, block_size=bs)
            w = d["workload"]
            e = torch.tensor([], dtype=w.dtype).element_size()
            B = partition_pass_bytes(d["lens"], w.num_q_heads, w.num_kv_heads, w.head_dim, bs, e, e)
            ms = time_partition_pass(d, steps, warmup)
            rows[f"bs{bs}_{'shuffled' if shuffle else 'identity'}"] = {
                "ms": round(ms, 4), "GBps": round(B / (ms * 1e-3) / 1e9, 1),
                "table_entries": int(sum(-(-int(n) // bs) for n in d["lens"]))}
            del d
            torch.cuda.empty_cache()
    return {"workload": name, "steps": steps, "kernel": "partition pass", "results": rows,
            "gather_overhead_bs32": round(rows["bs32_shuffled"]["ms"] / rows["bs32_identity"]["ms"] - 1, 4),
            "gather_overhead_bs16": round(rows["bs16_shuffled"]["ms"] / rows["bs16_identity"]["ms"] - 1, 4),
            "bs16_vs_bs32_shuffled": round(rows["bs16_shuffled"]["ms"] / rows["bs32_shuffled"]["ms"] - 1, 4),
            "what": "partition pass with blocks shuffled across the pool vs laid out consecutively; "
                    "overhead = shuffled / identity time - 1"}


def run_placement_study(args):
    from paged_kv_cache_237_gb300 import build as pa_build
    pa_build.build()
    torch.cuda.set_device(0)
    print(json.dumps({"study": "placement", **placement_block(args.workload, args.steps, args.warmup)}),
          flush=True)


def run_prefix_cache_study(args):
    from paged_kv_cache_237_gb300 import build as pa_build
    pa_build.build()
    torch.cuda.set_device(0)
    print(json.dumps({"study": "prefix_cache", **prefix_cache_block(args.steps, args.warmup)}), flush=True)


def prefix_cache_block(steps: int, warmup: int, tenants: int = 4, per_tenant: int = 64,
                       prompt_len: int = 2048) -> dict:
    """A multi-tenant batch admitted through the chained-key prefix cache: each
    tenant has its own 2048-token system prompt (salted by tenant), each
    request adds a private question of 16..512 tokens.  Reports host admission
    cost, blocks held with and without sharing, and the decode step over the
    shared blocks (GQA 64/8, head_dim 128, bs 16, bf16)."""
    from paged_kv_cache_237_gb300 import binding
    from paged_kv_cache_237_gb300.engine import DecodeStep
    from paged_kv_cache_237_gb300.workloads import randn
    rng = np.random.default_rng(7)
    bs, Hq, Hkv, hd = 16, 64, 8, 128
    systems = [rng.integers(0, 128000, size=prompt_len).tolist() for _ in range(tenants)]
    reqs = []
    for t in range(tenants):
        for _ in range(per_tenant):
            reqs.append((t, systems[t] + rng.integers(0, 128000, size=int(rng.integers(16, 513))).tolist()))
    order = rng.permutation(len(reqs))
    unshared = sum(-(-(len(r[1]) + 1) // bs) for r in reqs)
    bm = binding.BlockManager(unshared + 64, bs)
    t0 = time.perf_counter()
    cached_tokens = 0
    for sid in order:
        t, toks = reqs[sid]
        cached_tokens += bm.add_seq_cached(int(sid), toks, salt=1000 + t)
    admit_s = time.perf_counter() - t0
    seqs = list(range(len(reqs)))
    slots, pairs = bm.append_slots(seqs)
    held = bm.num_blocks - bm.num_free()
    max_blocks = max(len(bm.block_table(s)) for s in seqs)
    tables, lens = bm.build_tables(seqs, max_blocks)
    dev = torch.device("cuda", torch.cuda.current_device())
    nb = bm.num_blocks
    q = randn((len(seqs), Hq, hd), torch.bfloat16, 71, dev)
    kc = randn((nb, Hkv, bs, hd), torch.bfloat16, 72, dev)
    vc = randn((nb, Hkv, bs, hd), torch.bfloat16, 73, dev)
    kn = randn((len(seqs), Hkv, hd), torch.bfloat16, 74, dev)
    vn = randn((len(seqs), Hkv, hd), torch.bfloat16, 75, dev)
    step = DecodeStep(q, kc, vc, tables.to(dev), lens.to(dev), 1 / math.sqrt(hd), int(lens.max()))
    sl = slots.to(dev)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        step.run_fused(kn, vn, sl, stream=stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        a.record(stream)
        step.run_fused(kn, vn, sl, stream=stream)
        b.record(stream)
    torch.cuda.synchronize()
    if step.status.read():
        raise RuntimeError("device status flagged an input error")
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    logical = decode_bytes(lens.tolist(), Hq, Hkv, hd, bs, 2, 2, 2)
    unique_kv = held * Hkv * bs * hd * 2 * 2
    bm.close()
    del q, kc, vc, kn, vn, step
    torch.cuda.empty_cache()
    return {
        "tenants": tenants, "requests": len(reqs), "system_prompt_tokens": prompt_len,
        "copy_on_write_pairs": int(pairs.shape[0]),
        "host_admission_us_per_request": round(admit_s / len(reqs) * 1e6, 2),
        "cached_tokens_at_admission": int(cached_tokens),
        "blocks_held": int(held), "blocks_without_sharing": int(unshared),
        "memory_saved": round(1 - held / unshared, 4),
        "decode_step_ms": round(ms, 4), "logical_kv_GBps": round(logical / (ms * 1e-3) / 1e9, 1),
        "unique_kv_bytes": int(unique_kv), "unique_kv_GBps": round(unique_kv / (ms * 1e-3) / 1e9, 1),
        "timing": "eager decode steps (fused write), events around each"}


def run_swap_study(args):
    from paged_kv_cache_237_gb300 import build as pa_build
    pa_build.build()
    torch.cuda.set_device(0)
    print(json.dumps({"study": "swap", **swap_block(args.steps, args.warmup)}), flush=True)


def swap_block(steps: int, warmup: int, num_blocks: int = 4096) -> dict:
    """Swap-out (device -> pinned host) and swap-in (host -> device) of
    `num_blocks` scattered blocks of the long-context geometry (8 KV heads,
    block_size 32, head_dim 128, bf16: 128 KB of K+V per block), and the copy
    engines on one contiguous range of the same size for comparison."""
    from paged_kv_cache_237_gb300 import binding
    from paged_kv_cache_237_gb300.workloads import randn
    dev = torch.device("cuda", torch.cuda.current_device())
    Hkv, bs, hd = 8, 32, 128
    pool = 3 * num_blocks
    dk = randn((pool, Hkv, bs, hd), torch.bfloat16, 81, dev)
    dv = randn((pool, Hkv, bs, hd), torch.bfloat16, 82, dev)
    hk = torch.empty((num_blocks, Hkv, bs, hd), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty((num_blocks, Hkv, bs, hd), dtype=torch.bfloat16).pin_memory()
    rng = np.random.default_rng(9)
    dev_ids = rng.choice(pool, size=num_blocks, replace=False)
    out_pairs = torch.from_numpy(np.stack([dev_ids, rng.permutation(num_blocks)], 1).astype(np.int64)).to(dev)
    in_pairs = torch.from_numpy(np.stack([np.arange(num_blocks), rng.choice(pool, size=num_blocks, replace=False)],
                                         1).astype(np.int64)).to(dev)
    status = binding.DeviceStatus(dev)
    stream = torch.cuda.current_stream()
    nbytes = num_blocks * Hkv * bs * hd * 2 * 2

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in ev:
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    ms_out = timed(lambda: binding.pa_swap_blocks(dk, dv, hk, hv, out_pairs, status=status, stream=stream))
    ms_in = timed(lambda: binding.pa_swap_blocks(hk, hv, dk, dv, in_pairs, status=status, stream=stream))
    if status.read():
        raise RuntimeError("device status flagged an input error")
    # the copy engines on one contiguous range of the same size, for comparison
    half = hk.numel()
    dflat_k, dflat_v = dk.view(-1)[:half], dv.view(-1)[:half]
    hflat_k, hflat_v = hk.view(-1), hv.view(-1)

    def memcpy_out():
        hflat_k.copy_(dflat_k, non_blocking=True)
        hflat_v.copy_(dflat_v, non_blocking=True)

    def memcpy_in():
        dflat_k.copy_(hflat_k, non_blocking=True)
        dflat_v.copy_(hflat_v, non_blocking=True)
    mc_out, mc_in = timed(memcpy_out), timed(memcpy_in)
    del dk, dv, hk, hv
    torch.cuda.empty_cache()
    return {"blocks": num_blocks, "bytes_each_way": nbytes,
            "swap_out_ms": round(ms_out, 4), "swap_out_GBps": round(nbytes / (ms_out * 1e-3) / 1e9, 1),
            "swap_in_ms": round(ms_in, 4), "swap_in_GBps": round(nbytes / (ms_in * 1e-3) / 1e9, 1),
            "contiguous_memcpy_out_GBps": round(nbytes / (mc_out * 1e-3) / 1e9, 1),
            "contiguous_memcpy_in_GBps": round(nbytes / (mc_in * 1e-3) / 1e9, 1)}


def cache_ops_block(steps: int, warmup: int, tokens=(256, 4096, 65536), pairs=(24, 256, 2048)) -> dict:
    """pa_reshape_and_cache and pa_copy_blocks at decode-step sizes (latency)
    and at sizes where they stream HBM: the long-context geometry (8 KV heads,
    block_size 32, head_dim 128, bf16), distinct random slots and pairs, CUDA
    graphs of single launches, inputs larger than L2 where the size allows
    (a 512 MB buffer is written between launches otherwise).  Bytes are read +
    written bytes of the cache rows or blocks moved."""
    from paged_kv_cache_237_gb300 import binding
    from paged_kv_cache_237_gb300.workloads import randn
    dev = torch.device("cuda", torch.cuda.current_device())
    Hkv, bs, hd = 8, 32, 128
    pool = 40000                                  # 2.6 GB per cache
    kc = randn((pool, Hkv, bs, hd), torch.bfloat16, 91, dev)
    vc = randn((pool, Hkv, bs, hd), torch.bfloat16, 92, dev)
    flush = torch.empty(512 * 2**20 // 4, dtype=torch.float32, device=dev)
    status = binding.DeviceStatus(dev)
    stream = torch.cuda.current_stream()
    rng = np.random.default_rng(13)
    peak, _ = load_peak()

    def timed(fn, flush_between):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):          # fn launches on the current (capturing) stream
            fn()
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in ev:
            a.record(stream)
            g.replay()
            b.record(stream)
            if flush_between:
                flush_l2(flush)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    rows = {}
    for T in tokens:
        k = randn((T, Hkv, hd), torch.bfloat16, 93, dev)
        v = randn((T, Hkv, hd), torch.bfloat16, 94, dev)
        slots = torch.from_numpy(rng.choice(pool * bs, size=T, replace=False).astype(np.int64)).to(dev)
        nbytes = T * Hkv * hd * 2 * 2 * 2 + T * 8
        ms = timed(lambda: binding.pa_reshape_and_cache(k, v, kc, vc, slots, status=status),
                   nbytes < 2 * L2_BYTES)
        rows[f"reshape_and_cache_T{T}"] = {"us": round(ms * 1e3, 2), "GBps": round(nbytes / (ms * 1e-3) / 1e9, 1),
                                           "frac": round(nbytes / (ms * 1e-3) / 1e9 / peak, 4)}
    for P in pairs:
        ids = rng.choice(pool, size=2 * P, replace=False)
        pr = torch.from_numpy(np.stack([ids[:P], ids[P:]], 1).astype(np.int64)).to(dev)
        nbytes = P * 2 * Hkv * bs * hd * 2 * 2 + P * 16
        ms = timed(lambda: binding.pa_copy_blocks(kc, vc, pr, status=status),
                   nbytes < 2 * L2_BYTES)
        rows[f"copy_blocks_P{P}"] = {"us": round(ms * 1e3, 2), "GBps": round(nbytes / (ms * 1e-3) / 1e9, 1),
                                     "frac": round(nbytes / (ms * 1e-3) / 1e9 / peak, 4)}
    if status.read():
        raise RuntimeError("device status flagged an input error")
    del kc, vc, flush
    torch.cuda.empty_cache()
    return {"geometry": "8 KV heads, block_size 32, head_dim 128, bf16", "peak_GBps": peak,
            "frac_of": "measured copy peak", "results": rows}


def run_cache_ops_study(args):
    from paged_kv_cache_237_gb300 import build as pa_build
    pa_build.build()
    torch.cuda.set_device(0)
    print(json.dumps({"study": "cache_ops", **cache_ops_block(args.steps, args.warmup)}), flush=True)


def measure_step(name: str, steps: int, warmup: int = 5, gqa_sigma: float = 1.0, peak: float | None = None,
                 simt: bool = False) -> dict:
    """Graph-replayed decode step of another workload, timed in the same run:
    step GB/s and the partition pass alone.  The step is the one the main line
    times (copy-on-write copies, the decode launch with the fused cache write,
    the split-K merge); a workload whose writes are not each sequence's last
    position (the tiny fp32 batch) writes them with a separate launch.  Inputs
    smaller than twice L2 get a 512 MB write between replays, outside the
    events."""
    from paged_kv_cache_237_gb300 import binding
    from paged_kv_cache_237_gb300.engine import DecodeStep
    from paged_kv_cache_237_gb300.workloads import new_token_slots
    dev = torch.device("cuda", torch.cuda.current_device())
    d = build_workload(name, dev, 0, gqa_sigma)
    w = d["workload"]
    e = torch.tensor([], dtype=w.dtype).element_size()
    lens = d["lens"]
    B = decode_bytes(lens, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, e, e, e)
    Bp = partition_pass_bytes(lens, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, e, e)
    step = DecodeStep(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"], d["scale"],
                      d["max_context_len"], w.partition_size, simt=simt)
    last = new_token_slots(lens, d["block_tables"].cpu().numpy(), w.block_size)
    fused = (d["slot_mapping"].numel() == len(lens)
             and bool(np.array_equal(last, d["slot_mapping"].cpu().numpy())))
    tok = (d["k_new"], d["v_new"], d["slot_mapping"])
    cow = d["cow_pairs"]
    working_set = d["k_cache"].numel() * e * 2
    flush = None if working_set > 2 * L2_BYTES else torch.empty(512 * 2**20 // 4, dtype=torch.float32,
                                                                  device=dev)

    def full(_):
        if fused:
            step.run_fused(*tok, cow)
        else:
            step.run(*tok, cow)

    def part(_):
        if fused:
            step.decode(None, binding.PA_PHASE_PARTITIONS, *tok)
        else:
            step.decode(None, binding.PA_PHASE_PARTITIONS)

    for _ in range(warmup):
        full(None)
        flush_l2(flush)
    torch.cuda.synchronize()
    if step.status.read():
        raise RuntimeError("device status flagged an input error")
    stream = torch.cuda.current_stream()
    out = {}
    for key, fn in (("step", full), ("partition_pass", part)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            fn(None)
        g.replay()
        flush_l2(flush)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in ev:
            a.record(stream)
            g.replay()
            b.record(stream)
            flush_l2(flush)
        torch.cuda.synchronize()
        out[key] = statistics.mean(a.elapsed_time(b) for a, b in ev)
        if key == "step":
            out["step_events_each"] = out[key]
            if flush is None:
                # the steps back to back between one pair of events, as the main line times them
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(steps):
                    g.replay()
                b.record(stream)
                torch.cuda.synchronize()
                out[key] = a.elapsed_time(b) / steps
                # context only: ten steps captured in one graph, as a serving loop's graph of a whole
                # decode step would hold them (no graph-launch gap between them)
                g10 = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g10, capture_error_mode="relaxed"):
                    for _ in range(10):
                        fn(None)
                g10.replay()
                reps = max(1, steps // 10)
                a.record(stream)
                for _ in range(reps):
                    g10.replay()
                b.record(stream)
                torch.cuda.synchronize()
                out["step_graph_of_10"] = a.elapsed_time(b) / (10 * reps)
                del g10
    if step.status.read():
        raise RuntimeError("device status flagged an input error")
    res = {"dtype": "bf16" if w.dtype == torch.bfloat16 else "f32",
           "kernel": "decode_bf16_kernel" if w.dtype == torch.bfloat16 and not simt else "decode_simt_kernel",
           "ms_per_step": round(out["step"], 4), "us_per_step": round(out["step"] * 1e3, 2),
           "ms_per_step_events_each": round(out["step_events_each"], 4),
           "value": round(B / (out["step"] * 1e-3) / 1e9, 1),
           "partition_pass_ms": round(out["partition_pass"], 4),
           "partition_pass_GBps": round(Bp / (out["partition_pass"] * 1e-3) / 1e9, 1),
           "bytes_per_step": int(B), "total_context_tokens": int(sum(int(n) for n in lens)),
           "l2": "inputs larger than L2 (no flush)" if flush is None else "512 MB L2 flush between steps",
           "timing": "step: replays back to back between one pair of events" if flush is None
                     else "step: events around each replay, L2 flushed between"}
    if "step_graph_of_10" in out:
        res["context_graph_of_10_steps"] = {
            "ms_per_step": round(out["step_graph_of_10"], 4),
            "GBps": round(B / (out["step_graph_of_10"] * 1e-3) / 1e9, 1),
            "what": "ten steps in one CUDA graph (no launch gap between them); context, not the line's figure"}
    if peak:
        res["hbm_fraction"] = fractions(res["value"], peak)
        res["partition_pass_frac"] = round(res["partition_pass_GBps"] / peak, 4)
        if "context_graph_of_10_steps" in res:
            res["context_graph_of_10_steps"]["of_measured_copy_peak"] = round(
                res["context_graph_of_10_steps"]["GBps"] / peak, 4)
    if name.startswith("gqa_llama3_70b"):
        res["lognormal_sigma"] = gqa_sigma
    if cow is not None:
        # prefix sharing: the logical figure counts the shared prompt once per
        # sequence (it is read from L2 after the first); this one counts the
        # distinct blocks the step reads
        bs = w.block_size
        tab = d["block_tables"].cpu().numpy()
        used = {int(b) for i, n in enumerate(lens) for b in tab[i, :-(-int(n) // bs)]}
        uniq = len(used) * w.num_kv_heads * bs * w.head_dim * 2 * e
        res["copy_on_write_pairs"] = int(cow.numel() // 2)
        res["unique_kv_bytes"] = uniq
        res["unique_kv_GBps"] = round(uniq / (out["step"] * 1e-3) / 1e9, 1)
    del d, step, flush
    torch.cuda.empty_cache()
    return res


def run_mma_study(args):
    """Does batching the query-head group into mma tiles pay off?  The bf16
    partition pass with its products on tensor-core MMAs (the default) and on
    plain fp32 FMAs (SIMT kernel), same inputs, CUDA graphs, per workload."""
    from paged_kv_cache_237_gb300 import build as pa_build
    pa_build.build()
    from paged_kv_cache_237_gb300 import binding
    from paged_kv_cache_237_gb300.engine import DecodeStep
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    rows = {}
    for name in ("mha_llama2_7b", "gqa_llama3_70b", "long_context"):
        d = build_workload(name, dev, 0)
        w = d["workload"]
        Bp = partition_pass_bytes(d["lens"], w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, 2, 2)
        row = {"group": w.num_q_heads // w.num_kv_heads}
        outs = {}
        for mode, simt in (("mma", False), ("simt", True)):
            step = DecodeStep(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                              d["scale"], d["max_context_len"], w.partition_size, simt=simt)
            for _ in range(args.warmup):
                step.decode(None, binding.PA_PHASE_PARTITIONS)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="relaxed"):
                step.decode(None, binding.PA_PHASE_PARTITIONS)
            g.replay()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            for a, b in ev:
                a.record(stream)
                g.replay()
                b.record(stream)
            torch.cuda.synchronize()
            ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
            step.decode(None, binding.PA_PHASE_ALL)
            torch.cuda.synchronize()
            if step.status.read():
                raise RuntimeError("device status flagged an input error")
            outs[mode] = step.out.float().clone()
            row[f"{mode}_ms"] = round(ms, 4)
            row[f"{mode}_GBps"] = round(Bp / (ms * 1e-3) / 1e9, 1)
            del step
        row["simt_over_mma_time"] = round(row["simt_ms"] / row["mma_ms"], 3)
        row["max_abs_diff_mma_vs_simt"] = float((outs["mma"] - outs["simt"]).abs().max())
        rows[name] = row
        del d
        torch.cuda.empty_cache()
    print(json.dumps({"study": "mma", "kernel": "partition pass", "steps": args.steps, "results": rows}), flush=True)


def run_reference(args):
    """The fp64 oracle, as it stands, on the host cores: each step is a
    bounded sample of the workload (same metric and unit)."""
    sys.path.insert(0, ROOT)
    from paged_kv_cache_237_gb300 import workloads

    name = args.workload
    w = workloads.WORKLOADS[name]
    if name == "prefix_share":
        print(json.dumps({"impl": "reference", "unavailable": "reference arm samples only the "
                          "decode_inputs workloads"}))
        return
    # Build the workload on the GPU when there is one (same generator as our arm), else on the host.
    device = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    d = workloads.decode_inputs(name, device=device, gqa_sigma=args.gqa_sigma)
    threads = host_cores()
    per_step = max(0.3, min(10.0, 150.0 / (args.steps + args.warmup)))
    seqs = pick_sample(d, per_step, threads)
    sb = sample_kv_bytes(d, seqs)
    import oracle
    q, kc, vc, t, ln = oracle_sample(d, seqs)
    for _ in range(args.warmup):
        oracle.paged_decode(q, kc, vc, t, ln, d["scale"], threads=threads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.paged_decode(q, kc, vc, t, ln, d["scale"], threads=threads)
        times.append(time.perf_counter() - t0)
    ms = statistics.mean(times) * 1e3
    value = sb / (ms * 1e-3) / 1e9
    lens = d["lens"]
    sample = (f"{len(seqs)} of {len(lens)} sequences ({int(sum(lens[s] for s in seqs))} tokens, all "
              f"{w.num_q_heads} query heads) of the same workload per step, fp64 C oracle")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, d, 1, args.gqa_sigma),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


if __name__ == "__main__":
    main()
