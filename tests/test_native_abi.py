"""The C ABI driven from C++ alone (tests/native/abi_forward.cpp): no Python binding, no torch types.

The program computes the host metadata with the library's own functions, allocates device memory with
cudaMalloc, writes the history with paged_kv_write and runs the layer with paged_kv_write_attn, then the
same attention through paged_attn_varlen_noalloc (no workspace).  The CPU test builds it against
include/pagedkv.h and libpagedkv.so; the GPU test feeds it seeded inputs and compares both outputs with
the oracle, and with each other bit for bit.
"""

import dataclasses
import os
import subprocess

import numpy as np
import pytest
import torch

from paged_kv_cache_181_gb300 import configs, synth

from . import cases

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "paged_kv_cache_181_gb300")
SRC = os.path.join(ROOT, "tests", "native", "abi_forward.cpp")
CUDA = "/usr/local/cuda"

W = dataclasses.replace(configs.GQA_ACTION, name="native-gqa-bf16", num_heads=10, num_kv_heads=2, chunk_tokens=160,
                        window_chunks=2, sink_chunks=1, history_tokens=480, query_tokens=160, action_len=16,
                        spans=((320, 480),), pool_blocks=256)


def _build(tmp_path) -> str:
    from paged_kv_cache_181_gb300 import _lib

    exe = str(tmp_path / "abi_forward")
    cmd = ["g++", "-std=c++17", "-O2", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), "-I",
           os.path.join(CUDA, "include"), SRC, "-o", exe, os.path.dirname(_lib.LIB_PATH) + "/libpagedkv.so",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-Wl,-rpath," + PKG]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr[-3000:]
    return exe


def test_native_program_builds_against_the_header(tmp_path):
    if not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime.h")):
        pytest.skip("no CUDA toolkit headers")
    _build(tmp_path)


@pytest.mark.gpu
def test_native_forward_matches_oracle(tmp_path):
    exe = _build(tmp_path)
    w = W
    d = synth.draw(w, 0, "cpu")
    row_blocks, action_blocks = synth.allocation(w)
    with open(tmp_path / "params.txt", "w") as f:
        vals = [w.batch, w.num_heads, w.num_kv_heads, w.head_dim, w.pool_blocks, w.chunk_tokens, w.sink_tokens,
                w.window_tokens, w.action_len, w.history_tokens, w.query_tokens, len(w.spans)]
        vals += [x for span in w.spans for x in span]
        f.write(" ".join(str(int(v)) for v in vals) + "\n")
    np.concatenate([b.numpy() for b in row_blocks]).astype(np.int32).tofile(tmp_path / "row_blocks.i32")
    if w.action_len:
        np.concatenate([b.numpy() for b in action_blocks]).astype(np.int32).tofile(tmp_path / "action_blocks.i32")
    for name, t in (("q", d.q), ("k_hist", d.k_hist), ("v_hist", d.v_hist), ("k_cur", d.k_cur), ("v_cur", d.v_cur)):
        t.contiguous().view(torch.int16).numpy().tofile(tmp_path / f"{name}.bf16")
    res = subprocess.run([exe, str(tmp_path)], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "device bits 0x0" in res.stdout and "noalloc launches" in res.stdout
    assert res.stdout.rstrip().endswith("device bits 0x0"), res.stdout
    tq = w.batch * w.q_len
    oc = cases.oracle_metadata(w)
    cases.oracle_pools(w, d, oc)
    want = cases.expected(w, oc)
    raws = []
    for name in ("out.bf16", "out_noalloc.bf16"):
        raw = np.fromfile(tmp_path / name, dtype=np.int16).reshape(tq, w.num_heads, w.head_dim)
        raws.append(raw)
        got = torch.from_numpy(raw).view(torch.bfloat16).float().numpy()
        max_abs, mean_abs = cases.compare(got, want, "bf16")
        assert max_abs <= cases.TOL["bf16"][0] and mean_abs <= cases.TOL["bf16"][1], (name, max_abs, mean_abs)
    # Same kernels, same keys (the fused call reads the chunk from k/v, the second call from the pools it
    # wrote), same split plan: the same bits.
    assert np.array_equal(raws[0], raws[1])
