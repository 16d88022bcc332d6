"""The benchmark's byte accounting (its own code: the bench may not import the
oracle outside its CPU-baseline leg) against the oracle's pinned definition and
hand-computed cases, and the gate that withholds a traffic figure captured on
other code."""
import os
import shutil

import numpy as np

import bench
from oracle import accounting as acc


def test_decode_bytes_equals_the_pinned_definition():
    assert bench.decode_bytes([7, 16], 4, 2, 64, 16, 2, 2, 2) == 13840        # hand-computed in the accounting pins
    rng = np.random.default_rng(4)
    for _ in range(50):
        lens = rng.integers(0, 5000, size=int(rng.integers(1, 40))).tolist()
        hkv = int(rng.choice([1, 2, 8]))
        args = (int(hkv * rng.choice([1, 4, 8])), hkv, int(rng.choice([64, 128])), int(rng.choice([16, 32])))
        for e in ((2, 2, 2), (4, 4, 4)):
            assert bench.decode_bytes(lens, *args, *e) == acc.decode_algorithmic_bytes(lens, *args, *e)


def test_page_granular_bytes_count_whole_blocks():
    # lens 1, 16, 17 at bs 16: 4 pages = 64 slots for 34 tokens; 30 extra rows x 2 heads x 128 x 2 B x (K, V)
    tok = bench.decode_bytes([1, 16, 17], 8, 2, 128, 16, 2, 2, 2)
    assert bench.decode_bytes_pages([1, 16, 17], 8, 2, 128, 16, 2, 2, 2) - tok == 30 * 2 * 128 * 2 * 2
    assert bench.decode_bytes_pages([32, 64], 8, 2, 128, 32, 2, 2, 2) == bench.decode_bytes([32, 64], 8, 2, 128, 32,
                                                                                            2, 2, 2)


def test_partition_pass_bytes_leave_out_the_output():
    lens = [100, 513, 4096]
    full = bench.decode_bytes(lens, 64, 8, 128, 16, 2, 2, 2)
    assert full - bench.partition_pass_bytes(lens, 64, 8, 128, 16, 2, 2) == 3 * 64 * 128 * 2


def test_traffic_figure_is_withheld_once_the_code_changes(tmp_path, monkeypatch):
    src = os.path.join(bench.ROOT, "paged_kv_cache_237_gb300", "csrc")
    fake = tmp_path / "paged_kv_cache_237_gb300" / "csrc"
    fake.mkdir(parents=True)
    for name in bench.KERNEL_FILES:
        shutil.copy(os.path.join(src, name), fake / name)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    have = bench.captured_traffic("long_context")
    # a comment or whitespace edit keeps the figure; a code edit withholds it
    with open(fake / "pa_decode.cu", "a") as f:
        f.write("\n// a comment\n\n")
    assert bench.captured_traffic("long_context") == have
    with open(fake / "pa_decode.cu", "a") as f:
        f.write("static int an_edit = 1;\n")
    assert bench.captured_traffic("long_context") is None
    assert bench.captured_traffic("no_such_workload") is None


def test_bandwidth_fractions_name_their_denominators():
    f = bench.fractions(6787.6, 6787.6)
    assert f == {"of_measured_copy_peak": 1.0, "of_datasheet_7900_GBps": round(6787.6 / 7900.0, 4)}
    assert bench.fractions(3393.8, 6787.6)["of_measured_copy_peak"] == 0.5
