"""Fused write + attention in one launch (paged_kv_write_attn).

The pages write the chunk's K/V into the pools and then attend through the
block table (``paged_attention.py``, ``_paged_write_attn_impl``).  The fused
call does both in one launch: the attention reads the keys at the queries' own
positions from k/v while idle warps scatter k/v into the pools.  Checked here:

* after the call the pools equal the oracle's pools bit for bit (the write);
* the output is within tolerance of the float64 oracle, and bit-identical to
  paged_kv_write followed by paged_attn_varlen (same kernel arithmetic, same
  key and value bits, only their source differs);
* packed rows whose queries sit mid-sequence;
* check mode flags a token whose slot is not the one its key position implies.
"""

import dataclasses

import numpy as np
import pytest
import torch

from paged_kv_cache_181_gb300 import configs

from . import cases
from .test_gpu_parity import check_pools

pytestmark = pytest.mark.gpu

SMALL = [configs.TINY, configs.ONE_FRAME, configs.ONE_FRAME_PARTIAL, configs.GQA_ACTION, configs.MIXED_MASK]


def _fused_case(w, flags=0):
    from paged_kv_cache_181_gb300 import _lib, workload

    case = workload.build_case(w, poison=True, keep_draws=True, layers=1)  # history only in the pools
    out = case.write_attend(0, flags=flags | _lib.PKV_CHECK_BOUNDS).clone()
    torch.cuda.synchronize()
    assert _lib.check() == 0, "device error word set"
    assert _lib.last_launches() >= 1
    return case, out


@pytest.mark.parametrize("w", SMALL + [cases.EDGE[0], cases.EDGE[1], cases.EDGE[4]], ids=lambda w: w.name)
def test_fused_parity_and_pools(w):
    from paged_kv_cache_181_gb300 import _lib

    case, out = _fused_case(w)
    oc = cases.oracle_metadata(w)
    cases.oracle_pools(w, case.draws[0], oc)
    check_pools(case, oc)
    full = w.batch * w.q_len * w.num_heads * w.q_len <= 2_000_000
    sample = None if full else cases.sample_rows(w, 32)
    want = cases.expected(w, oc, sample)
    mask = None if sample is None else ~np.isnan(want)
    max_abs, mean_abs = cases.compare(out.float().cpu().numpy(), want, w.dtype, mask)
    tol_max, tol_mean = cases.TOL[w.dtype]
    assert max_abs <= tol_max and mean_abs <= tol_mean, (max_abs, mean_abs)
    # The two-call path on the now-written pools gives the same bits.
    two = case.attend(0).clone()
    torch.cuda.synchronize()
    assert torch.equal(out, two)
    assert _lib.last_launches() >= 1


@pytest.mark.parametrize("w", [configs.GQA_ACTION, configs.TINY], ids=lambda w: w.name)
def test_fused_with_forced_splits(w):
    from paged_kv_cache_181_gb300 import _lib

    case, out = _fused_case(w, flags=_lib.PKV_SPLITS(3))
    assert _lib.last_launches() == 2  # attention + combine
    oc = cases.oracle_metadata(w)
    cases.oracle_pools(w, case.draws[0], oc)
    check_pools(case, oc)
    sample = cases.sample_rows(w, 24) if w.q_len > 256 else None
    want = cases.expected(w, oc, sample)
    mask = None if sample is None else ~np.isnan(want)
    max_abs, mean_abs = cases.compare(out.float().cpu().numpy(), want, w.dtype, mask)
    tol_max, tol_mean = cases.TOL[w.dtype]
    assert max_abs <= tol_max and mean_abs <= tol_mean, (max_abs, mean_abs)


@pytest.mark.parametrize("pb", [configs.PACKED_SMALL,
                                dataclasses.replace(configs.PACKED_SMALL, name="packed-small-f32", dtype="f32",
                                                    head_dim=64, seed=34)], ids=lambda p: p.name)
def test_fused_packed_rows_mid_sequence(pb):
    from paged_kv_cache_181_gb300 import _lib, packed

    pc = packed.build_packed(pb, keep_draw=True)
    dev = pc.q.device
    # Take the query positions' keys back out of the pools (poison them) and pass them as k/v.
    ks, vs, slots = [], [], []
    for b, r in enumerate(pb.rows):
        blocks = pc.draw.row_blocks[b].numpy().astype(np.int32)
        slots.append(_lib.slot_mapping(blocks, r.kv_start_pos, r.query_len))
        ks.append(pc.draw.k_rows[b][r.kv_start_pos : r.kv_start_pos + r.query_len])
        vs.append(pc.draw.v_rows[b][r.kv_start_pos : r.kv_start_pos + r.query_len])
    slots = torch.from_numpy(np.concatenate(slots)).to(dev)
    k_new = torch.cat(ks).to(dev).contiguous()
    v_new = torch.cat(vs).to(dev).contiguous()
    pc.k_pool[slots] = float("nan")
    pc.v_pool[slots] = float("nan")
    out = _lib.paged_kv_write_attn(pc.q, k_new, v_new, slots, pc.k_pool, pc.v_pool, pc.block_table,
                                   pc.query_start_loc, pc.seq_lens, pc.max_query_len, pc.width * 16, pc.scale,
                                   segs=pc.segs, seg_start=pc.seg_start, out=pc.out, workspace=pc.workspace,
                                   flags=_lib.PKV_CHECK_BOUNDS)
    torch.cuda.synchronize()
    assert _lib.check() == 0
    op = cases.oracle_packed(pb, pc.draw)
    want = cases.expected_packed(pb, op)
    max_abs, mean_abs = cases.compare(out.float().cpu().numpy(), want, pb.dtype)
    tol_max, tol_mean = cases.TOL[pb.dtype]
    assert max_abs <= tol_max and mean_abs <= tol_mean, (max_abs, mean_abs)
    for gpu_pool, ref in ((pc.k_pool, op.k_pool), (pc.v_pool, op.v_pool)):
        got = gpu_pool.float().cpu().numpy()
        assert ((np.isnan(got) & np.isnan(ref)) | (got == ref)).all()


def test_fused_check_mode_flags_a_slot_its_key_does_not_imply():
    from paged_kv_cache_181_gb300 import _lib, workload

    w = configs.ONE_FRAME
    case = workload.build_case(w, poison=True, layers=1)
    bad = case.slots.clone()
    bad[[3, 4]] = bad[[4, 3]]  # two tokens trade slots
    _lib.paged_kv_write_attn(case.q[0], case.k_new[0], case.v_new[0], bad, case.k_pools[0], case.v_pools[0],
                             case.block_table, case.query_start_loc, case.seq_lens, case.meta.max_query_len,
                             case.meta.max_seq_len, case.scale, segs=case.segs, seg_start=case.seg_start,
                             out=case.out[0], workspace=case.workspace, flags=_lib.PKV_CHECK_BOUNDS)
    torch.cuda.synchronize()
    assert _lib.check() & _lib.PKV_DEVERR_SLOT


def test_fused_long_window_one_layer_equals_two_calls():
    # Full size: the fused launch and write-then-attend agree bit for bit, pools included;
    # sampled outputs are checked against the oracle elsewhere (test_gpu_checks).
    from paged_kv_cache_181_gb300 import _lib, workload

    w = configs.LONG_WINDOW
    a = workload.build_case(w, layers=1)
    fused = a.write_attend(0).clone()
    kp, vp = a.k_pools[0].clone(), a.v_pools[0].clone()
    a.write(0)
    two = a.attend(0)
    torch.cuda.synchronize()
    assert _lib.check() == 0
    # Bitwise: never-written slots of an unpoisoned pool may hold NaN patterns.
    assert torch.equal(kp.view(torch.int16), a.k_pools[0].view(torch.int16))
    assert torch.equal(vp.view(torch.int16), a.v_pools[0].view(torch.int16))
    assert torch.equal(fused, two)
