"""GPU parity: the CUDA path (through the C ABI) against the oracle, element by element.

The write and the host metadata must be bit-exact; attention must be within
max-abs 2e-2 / mean-abs 2e-3 of the float64 oracle for bf16/f16 inputs and
within 1e-4 for fp32.  Pools are NaN-poisoned, so reading any unwritten slot,
the evicted gap between the sink and the window, or table padding (block 0,
never allocated) turns an output NaN and fails.
"""

import dataclasses

import numpy as np
import pytest
import torch

from paged_kv_cache_181_gb300 import configs

from . import cases

pytestmark = pytest.mark.gpu

SMALL = [configs.TINY, configs.ONE_FRAME, configs.ONE_FRAME_PARTIAL, configs.GQA_ACTION, configs.MIXED_MASK]


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_181_gb300 import _lib

    return _lib


def run_case(w, flags=0, poison=True):
    from paged_kv_cache_181_gb300 import workload

    case = workload.build_case(w, poison=poison, keep_draws=True, layers=1)
    case.write(0, flags)
    out = case.attend(0, flags)
    torch.cuda.synchronize()
    from paged_kv_cache_181_gb300 import _lib

    assert _lib.check() == 0, "device error word set"
    return case, out


def check_metadata(case, oc):
    assert np.array_equal(case.meta.table, oc.table)
    assert np.array_equal(case.meta.seq_lens, oc.seq_lens)
    assert np.array_equal(case.meta.query_start_loc, oc.qsl)
    assert np.array_equal(case.meta.slots, oc.slots)
    if oc.segments is None:
        assert case.meta.segments is None
    else:
        want = [[(s.q_start, s.q_end, s.kv_end, 0 if s.mode == "causal" else 1) for s in row] for row in oc.segments]
        assert case.meta.segments == want


def check_pools(case, oc):
    # Bit-exact write: every slot equals the oracle's (NaN where never written).
    for gpu_pool, want in ((case.k_pools[0], oc.k_pool), (case.v_pools[0], oc.v_pool)):
        got = gpu_pool.float().cpu().numpy()
        both_nan = np.isnan(got) & np.isnan(want)
        assert (both_nan | (got == want)).all()


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_workload_parity(lib, w):
    case, out = run_case(w)
    oc = cases.oracle_metadata(w)
    check_metadata(case, oc)
    cases.oracle_pools(w, case.draws[0], oc)
    check_pools(case, oc)
    full = w.batch * w.q_len * w.num_heads * w.q_len <= 2_000_000 or w.name == "one-frame-bf16"
    sample = None if full else cases.sample_rows(w, 48)
    want = cases.expected(w, oc, sample)
    got = out.float().cpu().numpy()
    mask = None if sample is None else ~np.isnan(want)
    max_abs, mean_abs = cases.compare(got, want, w.dtype, mask)
    tol_max, tol_mean = cases.TOL[w.dtype]
    assert max_abs <= tol_max and mean_abs <= tol_mean, (max_abs, mean_abs)
    assert torch.isfinite(out).all()


@pytest.mark.parametrize("w", [configs.GQA_ACTION, configs.ONE_FRAME_PARTIAL], ids=lambda w: w.name)
@pytest.mark.parametrize("mode", ["splits3", "simt", "nosplit"])
def test_variants_agree(lib, w, mode):
    flags = {"splits3": lib.PKV_SPLITS(3), "simt": lib.PKV_FORCE_SIMT, "nosplit": lib.PKV_NO_SPLIT}[mode]
    case, out = run_case(w, flags)
    oc = cases.oracle_metadata(w)
    cases.oracle_pools(w, case.draws[0], oc)
    sample = cases.sample_rows(w, 16, seed=3)
    want = cases.expected(w, oc, sample)
    max_abs, mean_abs = cases.compare(out.float().cpu().numpy(), want, w.dtype, ~np.isnan(want))
    tol_max, tol_mean = cases.TOL[w.dtype]
    assert max_abs <= tol_max and mean_abs <= tol_mean, (max_abs, mean_abs)


def test_repeat_runs_are_bit_identical(lib):
    w = configs.MIXED_MASK
    case, out1 = run_case(w, poison=False)
    out1 = out1.clone()
    out2 = case.attend(0).clone()
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


EDGE = cases.EDGE


@pytest.mark.parametrize("w", EDGE, ids=lambda w: w.name)
def test_edge_cases(lib, w):
    case, out = run_case(w)
    oc = cases.oracle_metadata(w)
    check_metadata(case, oc)
    cases.oracle_pools(w, case.draws[0], oc)
    check_pools(case, oc)
    want = cases.expected(w, oc)
    max_abs, mean_abs = cases.compare(out.float().cpu().numpy(), want, w.dtype)
    tol_max, tol_mean = cases.TOL[w.dtype]
    assert max_abs <= tol_max and mean_abs <= tol_mean, (max_abs, mean_abs)


MEDIUM = [
    # D=64 (10-slot ring, many wraps), GQA 2, one-frame geometry
    dataclasses.replace(configs.ONE_FRAME, name="one-frame-d64-bf16", head_dim=64, num_heads=12, num_kv_heads=6,
                        seed=41),
    # fp16 end to end on the one-frame geometry
    dataclasses.replace(configs.ONE_FRAME, name="one-frame-f16", dtype="f16", seed=42),
    # fp32 at full size: the CUDA-core kernel's 64-key tiles (98 per row) through its asynchronous copies
    dataclasses.replace(configs.ONE_FRAME, name="one-frame-f32", dtype="f32", seed=43),
]


@pytest.mark.parametrize("w", MEDIUM, ids=lambda w: w.name)
@pytest.mark.parametrize("fused", [False, True], ids=["two-call", "fused"])
def test_medium_workloads_sampled_parity(lib, w, fused):
    from paged_kv_cache_181_gb300 import workload

    case = workload.build_case(w, poison=True, keep_draws=True, layers=1)
    if fused:
        out = case.write_attend(0, flags=lib.PKV_CHECK_BOUNDS)
    else:
        case.write(0, lib.PKV_CHECK_BOUNDS)
        out = case.attend(0, lib.PKV_CHECK_BOUNDS)
    torch.cuda.synchronize()
    assert lib.check() == 0
    oc = cases.oracle_metadata(w)
    cases.oracle_pools(w, case.draws[0], oc)
    sample = cases.sample_rows(w, 24)
    want = cases.expected(w, oc, sample)
    max_abs, mean_abs = cases.compare(out.float().cpu().numpy(), want, w.dtype, ~np.isnan(want))
    tol_max, tol_mean = cases.TOL[w.dtype]
    assert max_abs <= tol_max and mean_abs <= tol_mean, (max_abs, mean_abs)


def _tail_workload():
    # One more row than fills every SM once: 8 heads x (SMs // 8 + 1) rows of one 224-query item
    # each, so the launch runs whole items on every SM and splits the last row's 8 over their keys.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return dataclasses.replace(configs.GQA_ACTION, name="tail-split-gqa", batch=sms // 8 + 1, num_heads=8,
                               num_kv_heads=2, chunk_tokens=208, window_chunks=6, sink_chunks=1,
                               history_tokens=8 * 208, query_tokens=208, action_len=16, spans=((1248, 1456),),
                               pool_blocks=4096, seed=51)


def _run_tail(lib, w, fused, workspace_splits=None, scale_sign=1.0, flags=0):
    from paged_kv_cache_181_gb300 import workload

    case = workload.build_case(w, poison=True, keep_draws=True, layers=1)
    if workspace_splits is not None:
        tq = w.batch * w.q_len
        case.workspace = case.workspace[: workspace_splits * tq * w.num_heads * (w.head_dim + 1) * 4]
    case.scale *= scale_sign
    if fused:
        out = case.write_attend(0, flags=lib.PKV_CHECK_BOUNDS | flags)
    else:
        case.write(0, lib.PKV_CHECK_BOUNDS)
        out = case.attend(0, lib.PKV_CHECK_BOUNDS | flags)
    launches, plan = lib.last_launches(), lib.last_split_plan()
    torch.cuda.synchronize()
    assert lib.check() == 0
    oc = cases.oracle_metadata(w)
    cases.oracle_pools(w, case.draws[0], oc)
    want = cases.expected(w, oc, scale=case.scale)
    max_abs, mean_abs = cases.compare(out.float().cpu().numpy(), want, w.dtype)
    tol_max, tol_mean = cases.TOL[w.dtype]
    assert max_abs <= tol_max and mean_abs <= tol_mean, (max_abs, mean_abs)
    return launches, plan


@pytest.mark.parametrize("fused", [False, True], ids=["two-call", "fused"])
def test_split_tail_parity(lib, fused):
    """Whole items on every SM plus a key-split tail and its combine: every output against the oracle."""
    w = _tail_workload()
    launches, (splits, whole) = _run_tail(lib, w, fused)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert splits > 2 and whole == sms, (splits, whole)
    assert launches == 2  # attention + combine


def test_split_tail_shrinks_to_the_workspace(lib):
    """A workspace holding two splits' partials: the tail splits in two, the whole items stay whole."""
    w = _tail_workload()
    launches, (splits, whole) = _run_tail(lib, w, False, workspace_splits=2)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert splits == 2 and whole == sms and launches == 2, (splits, whole, launches)


def _simt_whole_items(w, sms):
    """Items the CUDA-core kernel runs whole: its whole waves of items (one CTA per SM)."""
    items = w.batch * w.num_heads * -(-w.q_len // cases.SIMT_ITEM_ROWS)
    return items // sms * sms, items


def test_negative_scale_plans_for_the_kernel_that_runs(lib):
    """A negative softmax scale on bf16 is refused unless the CUDA-core kernel is asked for by name; then it
    runs there, with that kernel's split plan (its own items of 128 queries: two whole waves and a split
    tail of 16), and matches the oracle."""
    from paged_kv_cache_181_gb300 import workload

    w = _tail_workload()
    case = workload.build_case(w, layers=1)
    case.scale = -case.scale
    with pytest.raises(lib.PkvError) as e:
        case.attend(0)
    assert e.value.status == lib.PKV_ERR_UNSUPPORTED and lib.last_launches() == 0
    del case
    launches, (splits, whole) = _run_tail(lib, w, False, scale_sign=-1.0, flags=lib.PKV_FORCE_SIMT)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    want_whole, items = _simt_whole_items(w, sms)
    assert items > want_whole > 0 and whole == want_whole and splits > 1 and launches == 2, (splits, whole)


@pytest.mark.parametrize("fused", [False, True], ids=["two-call", "fused"])
def test_cuda_core_split_tail_long_window_f32(lib, fused):
    """fp32 at the long window's full size: 1040 CUDA-core items of 128 queries are 6 waves of 152 SMs and
    128 more; those 128 split their 415 key tiles and the combine merges them, the rest run whole.  Sampled
    rows of every (row, head) -- the tail's included -- against the float64 oracle."""
    from paged_kv_cache_181_gb300 import workload

    w = configs.LONG_WINDOW_F32
    case = workload.build_case(w, poison=True, keep_draws=True, layers=1)
    if fused:
        out = case.write_attend(0, flags=lib.PKV_CHECK_BOUNDS)
    else:
        case.write(0, lib.PKV_CHECK_BOUNDS)
        out = case.attend(0, lib.PKV_CHECK_BOUNDS)
    launches, (splits, whole) = lib.last_launches(), lib.last_split_plan()
    torch.cuda.synchronize()
    assert lib.check() == 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    want_whole, items = _simt_whole_items(w, sms)
    if items % sms:
        assert whole == want_whole and splits > 1 and launches == 2, (splits, whole, launches)
    oc = cases.oracle_metadata(w)
    cases.oracle_pools(w, case.draws[0], oc)
    sample = cases.sample_rows(w, 12)
    want = cases.expected(w, oc, sample)
    max_abs, mean_abs = cases.compare(out.float().cpu().numpy(), want, w.dtype, ~np.isnan(want))
    tol_max, tol_mean = cases.TOL[w.dtype]
    assert max_abs <= tol_max and mean_abs <= tol_mean, (max_abs, mean_abs)
