"""GPU parity on packed heterogeneous rows (one call, rows of different shapes).

Rows differ in query length, key length, spans and query offset; some queries
sit mid-sequence with keys after them that only a full span may reach
(``DiffusionPagedAttentionRow.kv_start_pos``; ``build_paged_piecewise_plan``).
Every row's segments come from the library's ``build_segments`` with the row's
own offset.  Compared element by element with the float64 oracle, which takes
the offsets explicitly; NaN-poisoned pools.
"""

import dataclasses

import numpy as np
import pytest
import torch

from paged_kv_cache_181_gb300 import configs

from . import cases

pytestmark = pytest.mark.gpu

SMALL = configs.PACKED_SMALL
VARIANTS = [
    SMALL,
    dataclasses.replace(SMALL, name="packed-small-f16-d64", dtype="f16", head_dim=64, num_heads=4, num_kv_heads=4,
                        seed=33),
    dataclasses.replace(SMALL, name="packed-small-f32", dtype="f32", head_dim=64, seed=34),
    # 12 heads: the CUDA-core kernel's items (128 queries) are 6 rows x 12 heads x 3 = 216, one wave of 152
    # SMs and a tail of 64 that splits, rows of every length among them.
    dataclasses.replace(SMALL, name="packed-small-f32-h12", dtype="f32", head_dim=64, num_heads=12,
                        num_kv_heads=4, seed=35),
]


def _run(pb, flags=0):
    from paged_kv_cache_181_gb300 import _lib, packed

    pc = packed.build_packed(pb, keep_draw=True)
    out = pc.attend(flags=flags | _lib.PKV_CHECK_BOUNDS)
    torch.cuda.synchronize()
    assert _lib.check() == 0, "device error word set"
    return pc, out


@pytest.mark.parametrize("pb", VARIANTS, ids=lambda p: p.name)
@pytest.mark.parametrize("splits", [0, 3])
def test_packed_rows_parity(pb, splits):
    from paged_kv_cache_181_gb300 import _lib

    pc, out = _run(pb, flags=_lib.PKV_SPLITS(splits) if splits else 0)
    if pb.dtype == "f32" and not splits:
        # With more items than SMs, the CUDA-core kernel runs its whole waves whole and splits the tail.
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        items = len(pb.rows) * pb.num_heads * -(-max(r.query_len for r in pb.rows) // cases.SIMT_ITEM_ROWS)
        got_splits, whole = _lib.last_split_plan()
        if items > sms and items % sms:
            assert got_splits > 1 and whole == items // sms * sms, (got_splits, whole)
    op = cases.oracle_packed(pb, pc.draw)
    want = cases.expected_packed(pb, op)
    max_abs, mean_abs = cases.compare(out.float().cpu().numpy(), want, pb.dtype)
    tol_max, tol_mean = cases.TOL[pb.dtype]
    assert max_abs <= tol_max and mean_abs <= tol_mean, (max_abs, mean_abs)


def test_packed_rows_equal_each_row_alone():
    # Packing must not couple rows: row b of the packed call equals a call with row b alone.
    from paged_kv_cache_181_gb300 import _lib, packed

    # One key range per CTA in both calls, so both sum in the same order.
    pc, out = _run(SMALL, flags=_lib.PKV_NO_SPLIT)
    for b, r in enumerate(SMALL.rows):
        one = dataclasses.replace(SMALL, rows=(r,))
        pc1 = packed.build_packed(one)
        # The same keys: copy row b's pool blocks into the single-row case through its table.
        pc1.k_pool.copy_(pc.k_pool)
        pc1.v_pool.copy_(pc.v_pool)
        pc1.block_table.copy_(pc.block_table[b : b + 1, : pc1.width])
        q0, q1 = int(pc.qsl_host[b]), int(pc.qsl_host[b + 1])
        pc1.q.copy_(pc.q[q0:q1])
        o1 = pc1.attend(flags=_lib.PKV_NO_SPLIT)
        torch.cuda.synchronize()
        assert torch.equal(o1, out[q0:q1]), f"row {b} differs when packed"


@pytest.mark.parametrize("pb", [configs.PACKED_MIXED, configs.PACKED_FEW_HEADS], ids=lambda p: p.name)
def test_packed_full_size_sampled_rows(pb):
    # PACKED_FEW_HEADS has 8 query-tile pairs in all, so the planner splits every item's key range
    # (split-KV + combine).
    from paged_kv_cache_181_gb300 import _lib

    pc, out = _run(pb)
    if pb is configs.PACKED_FEW_HEADS:
        splits, whole = _lib.last_split_plan()
        assert splits > 1 and whole == 0, (splits, whole)
        assert _lib.last_launches() == 2
    op = cases.oracle_packed(pb, pc.draw)
    sample = cases.sample_packed_rows(pb, 6 if len(pb.rows) > 1 else 24)
    want = cases.expected_packed(pb, op, sample)
    mask = ~np.isnan(want)
    max_abs, mean_abs = cases.compare(out.float().cpu().numpy(), want, pb.dtype, mask)
    assert max_abs <= 2e-2 and mean_abs <= 2e-3, (max_abs, mean_abs)
    assert torch.isfinite(out).all()


def test_query_offset_past_the_keys_is_flagged():
    # A row whose first segment puts its queries past its keys breaks base + Sq <= L.
    from paged_kv_cache_181_gb300 import _lib, packed

    pc = packed.build_packed(SMALL)
    bad = pc.segs.clone()
    s0 = int(pc.seg_start[1])
    bad[s0, 0] = SMALL.rows[1].seq_len  # q_start of row 1's first segment
    _lib.paged_attn_varlen(pc.q, pc.k_pool, pc.v_pool, pc.block_table, pc.query_start_loc, pc.seq_lens,
                           pc.max_query_len, pc.width * 16, pc.scale, segs=bad, seg_start=pc.seg_start,
                           out=pc.out, workspace=pc.workspace, flags=_lib.PKV_CHECK_BOUNDS)
    torch.cuda.synchronize()
    assert _lib.check() & _lib.PKV_DEVERR_SEGMENT
