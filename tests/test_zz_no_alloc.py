"""GPU: the allocation-free attention entry point, for callers that cannot allocate device memory.

Such callers (fixed device-memory arenas, real-time loops that must not
allocate, plugin hosts without an allocator) call paged_attn_varlen_noalloc,
which takes no workspace and keeps its split-KV partial results in a fixed
scratch array inside the library.  Its results must match the float64 oracle
within the tolerances used elsewhere in these tests, and be bit-identical to
paged_attn_varlen given its own workspace when both calls run the same split
plan -- call after call, whatever the previous call left in the shared scratch.

This file is named so that pytest collects it last.
"""

import numpy as np
import pytest
import torch

from oracle import pagedattn as pa

from . import cases

pytestmark = pytest.mark.gpu

TOL = {torch.float32: (1e-4, 1e-4), torch.bfloat16: (2e-2, 2e-3), torch.float16: (2e-2, 2e-3)}


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_181_gb300 import _lib

    return _lib


def make_case(seed, dtype, hq, hkv, d, sq, kv, spans):
    """Random pools and a shuffled table; per-row segments from the library's build_segments for the GPU
    calls and from the oracle's for the oracle (the two are compared bit for bit elsewhere)."""
    from paged_kv_cache_181_gb300 import _lib

    g = torch.Generator().manual_seed(seed)
    B = len(sq)
    W = max(-(-L // 16) for L in kv) + 1
    nblk = B * W + 4
    q = torch.randn(sum(sq), hq, d, generator=g).to(dtype)
    kp = torch.randn(nblk * 16, hkv, d, generator=g).to(dtype)
    vp = torch.randn(nblk * 16, hkv, d, generator=g).to(dtype)
    table = torch.randperm(nblk, generator=g)[: B * W].reshape(B, W).to(torch.int32)
    qsl = np.concatenate([[0], np.cumsum(sq)]).astype(np.int32)
    rows = [_lib.build_segments(spans[b], kv[b] - sq[b], sq[b], kv[b]) for b in range(B)]
    segs = torch.tensor([s for r in rows for s in r], dtype=torch.int32).reshape(-1, 4)
    seg_start = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
    oracle = dict(q=q.float().numpy(), kp=kp.float().numpy(), vp=vp.float().numpy(), table=table.numpy().astype(np.int64),
                  qsl=qsl.astype(np.int64), seq=np.array(kv, dtype=np.int64),
                  segments=[pa.build_segments(spans[b], kv[b] - sq[b], sq[b]) for b in range(B)])
    return dict(q=q.cuda(), kp=kp.cuda(), vp=vp.cuda(), table=table.cuda(), qsl=torch.from_numpy(qsl).cuda(),
                seq=torch.tensor(kv, dtype=torch.int32).cuda(), segs=segs.cuda(),
                seg_start=torch.from_numpy(seg_start).cuda(), max_q=max(sq), max_kv=W * 16, oracle=oracle)


def run_both(lib, c, flags):
    """The workspace call, then the allocation-free call, on the same inputs; outputs, launches and plans."""
    tq, hq, d = c["q"].shape
    B = c["table"].shape[0]
    # Room for the most splits either call runs (16), so the workspace never shrinks the plan.
    nbytes = max(lib.workspace_size(tq, hq, d, B, c["max_q"], c["max_kv"]), 16 * tq * hq * (d + 1) * 4)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    args = (c["q"], c["kp"], c["vp"], c["table"], c["qsl"], c["seq"], c["max_q"], c["max_kv"], d ** -0.5)
    ref = lib.paged_attn_varlen(*args, segs=c["segs"], seg_start=c["seg_start"], workspace=ws, flags=flags)
    ref_plan = lib.last_split_plan()
    got = lib.paged_attn_varlen_noalloc(*args, segs=c["segs"], seg_start=c["seg_start"], flags=flags)
    launches, plan = lib.last_launches(), lib.last_split_plan()
    torch.cuda.synchronize()
    assert lib.check() == 0
    return ref.float().cpu().numpy(), got.float().cpu().numpy(), launches, ref_plan, plan


def check_against_oracle(c, got, dtype):
    o = c["oracle"]
    want = pa.paged_attention(o["q"], o["kp"], o["vp"], o["table"], o["qsl"], o["seq"], o["q"].shape[2] ** -0.5, 16,
                              o["segments"])
    assert np.isfinite(got).all()
    err = np.abs(got.astype(np.float64) - want)
    tol_max, tol_mean = TOL[dtype]
    assert err.max() <= tol_max and err.mean() <= tol_mean, (err.max(), err.mean())


CASES = [
    # (seed, dtype, Hq, Hkv, D, Sq per row, kv per row, spans per row, splits)
    (1, torch.bfloat16, 8, 2, 128, (300, 212), (900, 700), ([(700, 800)], []), 4),
    (2, torch.bfloat16, 4, 4, 64, (130, 17), (500, 17), ([], [(0, 9)]), 3),
    (3, torch.float32, 4, 2, 64, (40, 33), (120, 90), ([(90, 100)], []), 2),
    (6, torch.float16, 6, 3, 128, (64, 200), (64, 1000), ([(0, 64)], [(800, 1000)]), 16),
]


def test_noalloc_matches_oracle_and_workspace_call_on_consecutive_calls(lib):
    # Two passes over the cases: every call after the first finds the previous call's data in the scratch.
    for _ in range(2):
        for seed, dtype, hq, hkv, d, sq, kv, spans, splits in CASES:
            c = make_case(seed, dtype, hq, hkv, d, sq, kv, spans)
            ref, got, launches, ref_plan, plan = run_both(lib, c, lib.PKV_SPLITS(splits))
            assert launches == 2  # split attention + combine: the scratch is in use
            assert plan == ref_plan and plan[0] == splits, (plan, ref_plan)
            assert np.array_equal(got, ref)  # same kernels, same plan: the same bits
            check_against_oracle(c, got, dtype)


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
            ref, got, launches, ref_plan, plan = run_both(lib, c, 0)
            splits, whole = plan
            assert splits > 1 and whole == 0 and launches == 2, (splits, whole, launches)
            assert plan == ref_plan, (plan, ref_plan)
            assert np.array_equal(got, ref)
            check_against_oracle(c, got, dtype)


def test_noalloc_cuda_core_split_tail(lib):
    # fp32 runs on the CUDA-core kernel, whose items are 128 queries: 16 heads x 1280 queries = 160 items, one
    # wave of 152 SMs and a tail of 8 that splits into the scratch while the rest run whole.
    c = make_case(8, torch.float32, 16, 4, 64, (1280,), (1400,), ([(120, 1400)],))
    ref, got, launches, ref_plan, plan = run_both(lib, c, 0)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    items = 16 * 1280 // cases.SIMT_ITEM_ROWS
    if items > sms and items % sms:
        assert plan[0] > 1 and plan[1] == items // sms * sms and launches == 2, (plan, launches)
    assert plan == ref_plan, (plan, ref_plan)
    assert np.array_equal(got, ref)
    check_against_oracle(c, got, torch.float32)


def test_noalloc_clamps_forced_splits_like_the_workspace_call(lib):
    # PKV_SPLITS(20) asks for more than the 16 splits either call runs: both take it as 16.
    c = make_case(7, torch.bfloat16, 4, 2, 64, (100,), (3000,), ([(2900, 3000)],))
    ref, got, launches, ref_plan, plan = run_both(lib, c, lib.PKV_SPLITS(20))
    assert plan[0] == 16 and ref_plan[0] == 16 and launches == 2, (plan, ref_plan)
    assert np.array_equal(got, ref)
    check_against_oracle(c, got, torch.bfloat16)


def test_noalloc_refuses_splits_beyond_its_scratch(lib):
    # 8 splits x 20000 queries x 16 heads x 129 x 4 bytes >> the fixed scratch: refused before any launch.
    st = lib.lib.paged_attn_varlen_noalloc(None, 20000, 16, None, None, 1, 16, 16, 128, lib.PKV_BF16, None, 1, 1,
                                           None, None, 20000, 20000, 1.0, None, None, None, lib.PKV_SPLITS(8), None)
    assert st == lib.PKV_ERR_CAPACITY
    assert "scratch" in lib.last_error()
    assert lib.last_launches() == 0
