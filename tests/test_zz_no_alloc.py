"""GPU: the allocation-free attention entry point, for callers that cannot allocate device memory.

Such callers (fixed device-memory arenas, real-time loops that must not
allocate, plugin hosts without an allocator) call paged_attn_varlen_noalloc,
which takes no workspace and keeps its split-KV partial results in a fixed
scratch array inside the library.  Its results must match paged_attn_varlen
(given its own workspace) within the tolerance used elsewhere in these tests,
call after call, whatever the previous call left in the shared scratch.

This file is named so that pytest collects it last.
"""

import ctypes as C

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_181_gb300 import _lib

    return _lib


def make_case(seed, dtype, hq, hkv, d, sq, kv, spans):
    """Random pools and a shuffled table; per-row segments from the library's build_segments."""
    from paged_kv_cache_181_gb300 import _lib

    g = torch.Generator().manual_seed(seed)
    B = len(sq)
    W = max(-(-L // 16) for L in kv) + 1
    nblk = B * W + 4
    q = torch.randn(sum(sq), hq, d, generator=g).to(dtype).cuda()
    kp = torch.randn(nblk * 16, hkv, d, generator=g).to(dtype).cuda()
    vp = torch.randn(nblk * 16, hkv, d, generator=g).to(dtype).cuda()
    table = torch.randperm(nblk, generator=g)[: B * W].reshape(B, W).to(torch.int32).cuda()
    qsl = torch.tensor(np.concatenate([[0], np.cumsum(sq)]), dtype=torch.int32).cuda()
    seq = torch.tensor(kv, dtype=torch.int32).cuda()
    rows = [_lib.build_segments(spans[b], kv[b] - sq[b], sq[b], kv[b]) for b in range(B)]
    segs = torch.tensor([s for r in rows for s in r], dtype=torch.int32).reshape(-1, 4).cuda()
    seg_start = torch.tensor(np.concatenate([[0], np.cumsum([len(r) for r in rows])]), dtype=torch.int32).cuda()
    return dict(q=q, kp=kp, vp=vp, table=table, qsl=qsl, seq=seq, segs=segs, seg_start=seg_start,
                max_q=max(sq), max_kv=W * 16)


def run_both(lib, c, flags):
    ws = torch.empty(lib.workspace_size(c["q"].shape[0], c["q"].shape[1], c["q"].shape[2], 1, 1, 1),
                     dtype=torch.uint8, device="cuda")
    args = (c["q"], c["kp"], c["vp"], c["table"], c["qsl"], c["seq"], c["max_q"], c["max_kv"], c["q"].shape[2] ** -0.5)
    ref = lib.paged_attn_varlen(*args, segs=c["segs"], seg_start=c["seg_start"], workspace=ws, flags=flags)
    got = lib.paged_attn_varlen_noalloc(*args, segs=c["segs"], seg_start=c["seg_start"], flags=flags)
    launches = lib.last_launches()
    torch.cuda.synchronize()
    assert lib.check() == 0
    return ref.float().cpu().numpy(), got.float().cpu().numpy(), launches


CASES = [
    # (seed, dtype, Hq, Hkv, D, Sq per row, kv per row, spans per row, splits)
    (1, torch.bfloat16, 8, 2, 128, (300, 212), (900, 700), ([(700, 800)], []), 4),
    (2, torch.bfloat16, 4, 4, 64, (130, 17), (500, 17), ([], [(0, 9)]), 3),
    (3, torch.float32, 4, 2, 64, (40, 33), (120, 90), ([(90, 100)], []), 2),
]


def test_noalloc_matches_workspace_call_on_consecutive_calls(lib):
    # Two passes over the cases: every call after the first finds the previous call's data in the scratch.
    for _ in range(2):
        for seed, dtype, hq, hkv, d, sq, kv, spans, splits in CASES:
            c = make_case(seed, dtype, hq, hkv, d, sq, kv, spans)
            ref, got, launches = run_both(lib, c, lib.PKV_SPLITS(splits))
            assert launches == 2  # split attention + combine: the scratch is in use
            assert np.isfinite(got).all()
            err = np.abs(got - ref)
            if dtype == torch.float32:
                assert err.max() <= 1e-4
            else:
                assert err.max() <= 2e-2 and err.mean() <= 2e-3


PLANNED = [
    CASES[0][:8],
    (4, torch.bfloat16, 8, 8, 64, (256,), (4000,), ([],)),
    (5, torch.float16, 4, 1, 128, (100, 256, 7), (3000, 2100, 900), ([(1000, 1200)], [], [])),
]


def test_noalloc_planned_splits(lib):
    # Few items, so the planner splits every item's key range into the scratch; consecutive calls.
    for _ in range(2):
        for seed, dtype, hq, hkv, d, sq, kv, spans in PLANNED:
            c = make_case(seed, dtype, hq, hkv, d, sq, kv, spans)
            ref, got, launches = run_both(lib, c, 0)
            splits, whole = lib.last_split_plan()
            assert splits > 1 and whole == 0 and launches == 2, (splits, whole, launches)
            err = np.abs(got - ref)
            assert err.max() <= 2e-2 and err.mean() <= 2e-3


def test_noalloc_refuses_splits_beyond_its_scratch(lib):
    # 8 splits x 20000 queries x 16 heads x 129 x 4 bytes >> the fixed scratch: refused before any launch.
    st = lib.lib.paged_attn_varlen_noalloc(None, 20000, 16, None, None, 1, 16, 16, 128, lib.PKV_BF16, None, 1, 1,
                                           None, None, 20000, 20000, 1.0, None, None, None, lib.PKV_SPLITS(8), None)
    assert st == lib.PKV_ERR_CAPACITY
    assert "scratch" in lib.last_error()
    assert lib.last_launches() == 0
