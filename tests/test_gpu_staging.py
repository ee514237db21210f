"""Contiguous K/V: the block gather into staging buffers and attention on staged K/V.

The pages stage the visible window of a layer into contiguous buffers (an
``index_select`` of the visible blocks) and run the same varlen attention on
them, re-gathering only the current chunk's blocks when the history is already
staged (``paged_attention.py``, ``_stage_window`` and the contiguous gather
branch of ``ar_diffusion_paged_attention``; ``test_paged_attention.py``,
gather path vs paged path).

* the gather is a bit copy: the staged rows equal the oracle's
  ``gather_row_kv`` of the oracle's pools, bit for bit;
* a re-gather from the chunk's first block after the chunk was rewritten gives
  the oracle's gather of the rewritten pools;
* attention on the staged K/V (``PKV_CONTIGUOUS_KV``) is within the bf16/f16
  tolerance of the float64 oracle, and bit-identical to the paged mode on the
  same data (same kernel, same summation order: only the copies differ);
* a table that is not consecutive under ``PKV_CONTIGUOUS_KV`` is flagged in
  check mode and still gives the right answer.
"""

import dataclasses

import numpy as np
import pytest
import torch

from oracle import pagedattn as pa
from paged_kv_cache_181_gb300 import configs, synth

from . import cases

pytestmark = pytest.mark.gpu

SMALL = [configs.ONE_FRAME, configs.ONE_FRAME_PARTIAL, configs.GQA_ACTION, configs.MIXED_MASK, cases.EDGE[0],
         cases.EDGE[1], cases.EDGE[4]]


def _build(w):
    from paged_kv_cache_181_gb300 import workload

    case = workload.build_case(w, poison=True, keep_draws=True, layers=1)
    case.write(0)
    st = case.make_staging()
    return case, st


def _oracle(w, case):
    oc = cases.oracle_metadata(w)
    cases.oracle_pools(w, case.draws[0], oc)
    return oc


def _staged_equals_oracle(case, st, oc, w):
    for b in range(w.batch):
        L = int(oc.seq_lens[b])
        for got_t, pool in ((st.k, oc.k_pool), (st.v, oc.v_pool)):
            got = got_t[b, :L].float().cpu().numpy()
            want = pa.gather_row_kv(pool, oc.table[b], L, w.block_size)
            assert np.array_equal(got, want), f"row {b}: staged rows differ from the oracle's gather"


@pytest.mark.parametrize("w", SMALL[:4], ids=lambda w: w.name)
def test_gather_is_bit_exact(w):
    from paged_kv_cache_181_gb300 import _lib

    case, st = _build(w)
    case.stage(0, st)
    torch.cuda.synchronize()
    assert _lib.last_launches() == 1
    _staged_equals_oracle(case, st, _oracle(w, case), w)


def test_regather_from_the_chunk_refreshes_only_what_moved():
    from paged_kv_cache_181_gb300 import _lib

    w = configs.GQA_ACTION
    case, st = _build(w)
    case.stage(0, st)
    # A later probe of the same chunk: new K/V for the chunk, history unchanged.
    d2 = synth.draw(dataclasses.replace(w, seed=w.seed + 100), 0)
    case.k_new[0].copy_(d2.k_cur)
    case.v_new[0].copy_(d2.v_cur)
    case.write(0)
    case.stage(0, st, reuse_history=True)
    torch.cuda.synchronize()
    assert _lib.check() == 0
    oc = cases.oracle_metadata(w)
    d_mixed = dataclasses.replace(case.draws[0], k_cur=d2.k_cur, v_cur=d2.v_cur)
    cases.oracle_pools(w, d_mixed, oc)
    assert st.first_block > 0
    _staged_equals_oracle(case, st, oc, w)


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_contiguous_attention_parity(w):
    from paged_kv_cache_181_gb300 import _lib

    case, st = _build(w)
    paged = case.attend(0).clone()
    case.stage(0, st)
    out = case.attend_contiguous(0, st, flags=_lib.PKV_CHECK_BOUNDS)
    torch.cuda.synchronize()
    assert _lib.check() == 0, "device error word set"
    oc = _oracle(w, case)
    full = w.batch * w.q_len * w.num_heads * w.q_len <= 2_000_000
    sample = None if full else cases.sample_rows(w, 32)
    want = cases.expected(w, oc, sample)
    got = out.float().cpu().numpy()
    mask = None if sample is None else ~np.isnan(want)
    max_abs, mean_abs = cases.compare(got, want, w.dtype, mask)
    tol_max, tol_mean = cases.TOL[w.dtype]
    assert max_abs <= tol_max and mean_abs <= tol_mean, (max_abs, mean_abs)
    assert torch.equal(out, paged), "contiguous and paged modes must give identical bits"


def test_contiguous_flag_on_a_paged_table_is_flagged_and_still_correct():
    from paged_kv_cache_181_gb300 import _lib

    w = configs.ONE_FRAME
    case, _ = _build(w)
    paged = case.attend(0).clone()
    torch.cuda.synchronize()
    assert _lib.check() == 0
    out = case.attend(0, flags=_lib.PKV_CHECK_BOUNDS | _lib.PKV_CONTIGUOUS_KV)
    torch.cuda.synchronize()
    bits = _lib.check()
    assert bits & _lib.PKV_DEVERR_BLOCK
    assert torch.equal(out, paged)


def test_gather_argument_errors():
    from paged_kv_cache_181_gb300 import _lib

    w = configs.TINY
    case, st = _build(dataclasses.replace(w, dtype="bf16"))
    W = case.meta.width
    with pytest.raises(_lib.PkvError):
        _lib.paged_kv_gather(case.k_pools[0], case.v_pools[0], case.block_table, st.k, st.v, first_block=1,
                             n_blocks=W)
    short = st.k[:, :16].contiguous()
    with pytest.raises(_lib.PkvError):
        _lib.paged_kv_gather(case.k_pools[0], case.v_pools[0], case.block_table, short, short.clone(), n_blocks=2)
    _lib.paged_kv_gather(case.k_pools[0], case.v_pools[0], case.block_table, st.k, st.v, n_blocks=0)
    assert _lib.last_launches() == 0


def test_gather_check_mode_flags_bad_block_ids():
    from paged_kv_cache_181_gb300 import _lib

    w = configs.ONE_FRAME
    case, st = _build(w)
    bad = case.block_table.clone()
    bad[0, 0] = w.pool_blocks + 5
    _lib.paged_kv_gather(case.k_pools[0], case.v_pools[0], bad, st.k, st.v, n_blocks=2,
                         flags=_lib.PKV_CHECK_BOUNDS)
    torch.cuda.synchronize()
    assert _lib.check() & _lib.PKV_DEVERR_BLOCK
