"""The library from a plain C program: tests/c_client/pa_c_client.c includes
include/pa.h, allocates device memory with the CUDA runtime and runs one
decode step -- copy-on-write block copy, the new tokens' cache write, decode
attention -- with no Python or torch in its process.  Inputs come from the
seeded test generator through files; the caches it writes back must equal the
oracle's copy and write bit for bit, and its outputs the oracle's attention
within the usual tolerance."""
import math
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_decode_close, make_case

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def cuda_home() -> str:
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def cudart_dir(home: str) -> str:
    cands = [os.path.join(home, "lib64")]
    targets = os.path.join(home, "targets")
    if os.path.isdir(targets):
        cands += [os.path.join(targets, t, "lib") for t in sorted(os.listdir(targets))]
    for cand in cands:
        if os.path.exists(os.path.join(cand, "libcudart.so")):
            return cand
    pytest.fail(f"libcudart.so not found under {home}")


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    from paged_kv_cache_237_gb300 import build as pa_build
    lib = pa_build.build()
    libdir = os.path.dirname(lib)
    home = cuda_home()
    rt = cudart_dir(home)
    exe = str(tmp_path_factory.mktemp("c_client") / "pa_c_client")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", f"-I{os.path.join(ROOT, 'include')}", f"-I{os.path.join(home, 'include')}",
           os.path.join(ROOT, "tests", "c_client", "pa_c_client.c"), "-o", exe, f"-L{libdir}", "-lpa_gb300",
           f"-L{rt}", "-lcudart", f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{rt}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def raw(t: torch.Tensor) -> bytes:
    t = t.contiguous().cpu()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.numpy().tobytes()


@pytest.mark.parametrize("dtype,hd,bs,Hq,Hkv,P", [(torch.bfloat16, 128, 16, 16, 2, 512),
                                                   (torch.float32, 64, 32, 8, 8, 128)])
def test_c_program_runs_a_decode_step_through_the_header_alone(client, tmp_path, dtype, hd, bs, Hq, Hkv, P):
    lens = [1, bs + 3, 700, 1500, 2 * bs]
    q, kc, vc, tables, lens_t = make_case(lens, Hq, Hkv, hd, bs, dtype, seed=31, device="cpu", slack=5,
                                          nan_tails=False)
    S, nb = len(lens), kc.shape[0]
    # Copy-on-write: sequence 2's last block moves to a free block, copied first.
    used = {int(b) for i, n in enumerate(lens) for b in tables[i, :-(-n // bs)].tolist()}
    free = [b for b in range(nb) if b not in used]
    last = (lens[2] - 1) // bs
    pairs = torch.tensor([[int(tables[2, last]), free[0]]], dtype=torch.int64)
    tables[2, last] = free[0]
    slots = torch.tensor([int(tables[i, (n - 1) // bs]) * bs + (n - 1) % bs for i, n in enumerate(lens)],
                         dtype=torch.int64)
    g = torch.Generator().manual_seed(32)
    k_new = torch.randn(S, Hkv, hd, generator=g).to(dtype)
    v_new = torch.randn(S, Hkv, hd, generator=g).to(dtype)
    scale = 1.0 / math.sqrt(hd)

    d = str(tmp_path)
    with open(os.path.join(d, "sizes.txt"), "w") as f:
        f.write(f"{S} {Hq} {Hkv} {hd} {bs} {nb} {tables.shape[1]} {0 if dtype == torch.float32 else 1} {P} "
                f"{pairs.shape[0]} {scale!r}\n")
    for name, t in (("q", q), ("k_cache", kc), ("v_cache", vc), ("k_new", k_new), ("v_new", v_new),
                    ("tables", tables.to(torch.int32)), ("lens", lens_t.to(torch.int32)), ("slots", slots),
                    ("pairs", pairs)):
        with open(os.path.join(d, name + ".bin"), "wb") as f:
            f.write(raw(t))
    r = subprocess.run([client, d], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "sequences decoded" in r.stdout

    kc_ref, vc_ref = kc.clone(), vc.clone()
    oracle.copy_blocks(kc_ref, vc_ref, pairs)
    oracle.reshape_and_cache(k_new, v_new, kc_ref, vc_ref, slots)
    np_dt = np.float32 if dtype == torch.float32 else np.int16

    def load(name, like):
        a = np.fromfile(os.path.join(d, name + ".bin"), dtype=np_dt).reshape(like.shape)
        t = torch.from_numpy(a)
        return t if dtype == torch.float32 else t.view(torch.bfloat16)

    assert torch.equal(raw_view(load("k_cache_out", kc)), raw_view(kc_ref))
    assert torch.equal(raw_view(load("v_cache_out", vc)), raw_view(vc_ref))
    ref = oracle.paged_decode(q, kc_ref, vc_ref, tables.to(torch.int32), lens_t.to(torch.int32), scale)
    assert_decode_close(load("out", q), ref, dtype, what=f"C client {dtype}")


def raw_view(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)
