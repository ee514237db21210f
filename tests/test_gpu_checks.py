"""GPU: bounds-check mode, empty rows, ragged batches, and the long-window workload at full size
(40 layers on sampled rows; one layer on every output).

Bad metadata is only ever handed to kernels with PKV_CHECK_BOUNDS set: they
skip the offending access and raise the device error word (no fault, no trap).
"""

import numpy as np
import pytest
import torch

from paged_kv_cache_181_gb300 import configs

from . import cases

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_181_gb300 import _lib

    return _lib


def small_inputs(dtype=torch.bfloat16, B=2, hq=4, hkv=2, d=64, nblk=32, sq=(20, 0), L=(40, 5), W=4):
    g = torch.Generator().manual_seed(77)
    tq = sum(sq)
    q = torch.randn(tq, hq, d, generator=g).to(dtype).cuda()
    kp = torch.randn(nblk * 16, hkv, d, generator=g).to(dtype).cuda()
    vp = torch.randn(nblk * 16, hkv, d, generator=g).to(dtype).cuda()
    perm = torch.randperm(nblk, generator=g)
    table = perm[: B * W].reshape(B, W).to(torch.int32).cuda()
    qsl = torch.tensor(np.concatenate([[0], np.cumsum(sq)]), dtype=torch.int32).cuda()
    seq = torch.tensor(L, dtype=torch.int32).cuda()
    return q, kp, vp, table, qsl, seq


def test_clean_run_in_check_mode_raises_nothing(lib):
    q, kp, vp, table, qsl, seq = small_inputs()
    lib.paged_attn_varlen(q, kp, vp, table, qsl, seq, 20, 64, 0.125, flags=lib.PKV_CHECK_BOUNDS)
    assert lib.check() == 0


def test_bad_block_id_is_flagged_not_read(lib):
    q, kp, vp, table, qsl, seq = small_inputs()
    table[0, 1] = 10_000  # outside the 32-block pool
    out = lib.paged_attn_varlen(q, kp, vp, table, qsl, seq, 20, 64, 0.125, flags=lib.PKV_CHECK_BOUNDS)
    bits = lib.check()
    assert bits & lib.PKV_DEVERR_BLOCK
    assert lib.check() == 0  # cleared
    # the context is still usable
    table[0, 1] = 3
    lib.paged_attn_varlen(q, kp, vp, table, qsl, seq, 20, 64, 0.125, out=out, flags=lib.PKV_CHECK_BOUNDS)
    assert lib.check() == 0


def test_seq_len_past_table_is_flagged(lib):
    q, kp, vp, table, qsl, seq = small_inputs()
    seq[0] = 100  # > W * 16 = 64
    lib.paged_attn_varlen(q, kp, vp, table, qsl, seq, 20, 64, 0.125, flags=lib.PKV_CHECK_BOUNDS)
    assert lib.check() & lib.PKV_DEVERR_SEQLEN


def test_bad_slot_is_flagged_and_skipped(lib):
    k = torch.randn(3, 2, 64).to(torch.bfloat16).cuda()
    v = torch.randn(3, 2, 64).to(torch.bfloat16).cuda()
    kp = torch.zeros(64, 2, 64, dtype=torch.bfloat16).cuda()
    vp = torch.zeros_like(kp)
    slots = torch.tensor([5, 64, -1], dtype=torch.int64).cuda()
    lib.paged_kv_write(k, v, slots, kp, vp, flags=lib.PKV_CHECK_BOUNDS)
    assert lib.check() & lib.PKV_DEVERR_SLOT
    assert torch.equal(kp[5], k[0]) and torch.equal(vp[5], v[0])
    kp[5] = 0
    assert (kp == 0).all()  # the bad and the skipped token wrote nothing


def test_empty_row_and_ragged_batch_match_oracle(lib):
    from oracle import pagedattn as pa

    # D 64 and 128; every row of at most 64 queries, so the CUDA-core kernel runs its 64-row CTAs.
    for d, dtype, flags in ((64, torch.bfloat16, 0), (64, torch.float32, 0), (64, torch.bfloat16, lib.PKV_FORCE_SIMT),
                            (128, torch.float32, 0), (128, torch.bfloat16, lib.PKV_FORCE_SIMT)):
        q, kp, vp, table, qsl, seq = small_inputs(dtype=dtype, d=d, B=3, sq=(20, 0, 3), L=(40, 5, 17), W=4)
        out = lib.paged_attn_varlen(q, kp, vp, table, qsl, seq, 20, 64, 0.3, flags=flags)
        torch.cuda.synchronize()
        want = pa.paged_attention(q.float().cpu().numpy(), kp.float().cpu().numpy(), vp.float().cpu().numpy(),
                                  table.cpu().numpy(), qsl.cpu().numpy(), seq.cpu().numpy(), 0.3, 16)
        tol = 1e-4 if dtype == torch.float32 else 2e-2
        assert np.abs(out.float().cpu().numpy() - want).max() <= tol


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "two-call"])
def test_long_window_forty_layers_full_size(lib, fused):
    """The benchmarked workload in its benchmarked launch configuration: 40 layers, one forward
    (the fused write + attention call per layer, as bench.py times it, and the two-call form).

    Each checked layer is compared on sampled query rows against the float64
    oracle over all 26520 keys; the write is checked bit-exactly at every
    current-chunk slot.
    """
    from paged_kv_cache_181_gb300 import synth, workload

    w = configs.LONG_WINDOW
    case = workload.build_case(w, device="cuda", poison=False)
    case.step(fused=fused)
    torch.cuda.synchronize()
    assert lib.check() == 0
    oc0 = cases.oracle_metadata(w)
    assert np.array_equal(case.meta.table, oc0.table) and np.array_equal(case.meta.seq_lens, oc0.seq_lens)
    assert int(oc0.seq_lens[0]) == 26520
    for layer in (0, w.layers - 1):
        d = synth.draw(w, layer, device="cuda")
        d = synth.Draw(w, layer, d.row_blocks, d.action_blocks, d.q.cpu(), d.k_hist.cpu(), d.v_hist.cpu(),
                       d.k_cur.cpu(), d.v_cur.cpu())
        assert torch.equal(d.q, case.q[layer].cpu())
        oc = cases.oracle_metadata(w)
        cases.oracle_pools(w, d, oc)
        slots = torch.from_numpy(oc.slots)
        got_k = case.k_pools[layer][slots.cuda()].float().cpu().numpy()
        assert np.array_equal(got_k, oc.k_pool[oc.slots])
        sample = cases.sample_rows(w, 6, seed=layer)
        want = cases.expected(w, oc, sample)
        max_abs, mean_abs = cases.compare(case.out[layer].float().cpu().numpy(), want, w.dtype, ~np.isnan(want))
        assert max_abs <= 2e-2 and mean_abs <= 2e-3, (layer, max_abs, mean_abs)


def test_long_window_layer_zero_every_output(lib):
    """Every output of one layer of the benchmarked workload, through the call bench.py times
    (the fused write + attention with its split tail): 2 rows x 40 heads x 1560 queries over
    26520 keys, against the float32 oracle twin (within 1e-5 of float64, pinned on the CPU)."""
    from paged_kv_cache_181_gb300 import synth, workload

    w = configs.LONG_WINDOW
    case = workload.build_case(w, device="cuda", poison=False, layers=1, data_device="cpu")
    case.step(fused=True)
    torch.cuda.synchronize()
    assert lib.check() == 0
    splits, whole = lib.last_split_plan()
    assert splits > 1 and whole > 0  # the split tail behind whole waves, as in the bench
    d = synth.draw(w, 0, device="cpu")  # the same seeded draw the case made
    assert torch.equal(d.q, case.q[0].cpu())
    oc = cases.oracle_metadata(w)
    cases.oracle_pools(w, d, oc)
    want = cases.expected(w, oc, dtype=np.float32).astype(np.float64)
    assert not np.isnan(want).any()
    max_abs, mean_abs = cases.compare(case.out[0].float().cpu().numpy(), want, w.dtype)
    assert max_abs <= 2e-2 and mean_abs <= 2e-3, (max_abs, mean_abs)


def test_expired_wait_reports_timeout_and_leaves_the_context_usable(lib):
    # The kernels' bounded pipeline wait, made to run out on a barrier nothing completes.
    import time

    from paged_kv_cache_181_gb300 import workload

    t0 = time.perf_counter()
    lib.selftest_wait(50_000_000)  # 50 ms
    bits = lib.check()
    elapsed = time.perf_counter() - t0
    assert bits & lib.PKV_DEVERR_TIMEOUT
    assert 0.04 < elapsed < 5.0
    assert lib.check() == 0  # check() cleared the word
    # The context still works: a normal call runs and matches the oracle.
    w = configs.TINY
    case = workload.build_case(w, poison=True, keep_draws=True, layers=1)
    case.write(0)
    out = case.attend(0)
    torch.cuda.synchronize()
    assert lib.check() == 0
    oc = cases.oracle_metadata(w)
    cases.oracle_pools(w, case.draws[0], oc)
    max_abs, _ = cases.compare(out.float().cpu().numpy(), cases.expected(w, oc), w.dtype)
    assert max_abs <= cases.TOL[w.dtype][0]
