"""Large pools: block ids near the top of a pool of more than 2^31 elements (64-bit addressing).

Paging only changes where keys live, so the oracle attends over a compact pool
holding the same keys (its table renumbers the blocks 0, 1, 2, ...), while the
GPU path writes and reads them at block ids around 600 000 of a 39 GB pool pair
(K and V each 600 000 blocks x 16 rows x 8 heads x 128 x bf16 = 19.7 GB: byte
offsets past 2^34).  Covers the write, both attention kernels, the fused call
and the block gather.
"""

import numpy as np
import pytest
import torch

from oracle import pagedattn as pa

from . import cases

pytestmark = pytest.mark.gpu

BS, HKV, HQ, D = 16, 8, 16, 128
POOL_BLOCKS = 600_000
ROWS = [(200, 1000, ((800, 1000),)), (37, 777, ())]  # (Sq, L, spans): a suffix query per row


def _setup():
    from paged_kv_cache_181_gb300 import _lib

    if torch.cuda.get_device_properties(0).total_memory < 80 * 2**30:
        pytest.skip("needs a large device")
    g = torch.Generator().manual_seed(77)
    dev = torch.device("cuda")
    n_blocks = [-(-L // BS) for _, L, _ in ROWS]
    W = max(n_blocks)
    # GPU block ids near the top of the pool, shuffled; the oracle's are 0..n-1 per row in order.
    top = torch.randperm(sum(n_blocks) + 50, generator=g) + (POOL_BLOCKS - sum(n_blocks) - 50)
    table = np.zeros((len(ROWS), W), dtype=np.int32)
    o_table = np.zeros((len(ROWS), W), dtype=np.int64)
    used = 0
    k_rows, v_rows = [], []
    for b, (sq, L, _) in enumerate(ROWS):
        table[b, : n_blocks[b]] = top[used : used + n_blocks[b]].numpy()
        o_table[b, : n_blocks[b]] = np.arange(used, used + n_blocks[b])
        used += n_blocks[b]
        k_rows.append(torch.randn(L, HKV, D, generator=g).to(torch.bfloat16))
        v_rows.append(torch.randn(L, HKV, D, generator=g).to(torch.bfloat16))
    tq = sum(sq for sq, _, _ in ROWS)
    q = torch.randn(tq, HQ, D, generator=g).to(torch.bfloat16)
    qsl = np.concatenate([[0], np.cumsum([sq for sq, _, _ in ROWS])]).astype(np.int32)
    seq_lens = np.array([L for _, L, _ in ROWS], dtype=np.int32)
    segs, starts = [], [0]
    o_segs = []
    for sq, L, spans in ROWS:
        row = _lib.build_segments(list(spans), L - sq, sq, L)
        segs += row
        starts.append(len(segs))
        o_segs.append(pa.build_segments(list(spans), L - sq, sq))
    k_pool = torch.empty((POOL_BLOCKS * BS, HKV, D), dtype=torch.bfloat16, device=dev)
    v_pool = torch.empty_like(k_pool)
    meta = dict(
        table=torch.from_numpy(table).to(dev), qsl=torch.from_numpy(qsl).to(dev),
        seq_lens=torch.from_numpy(seq_lens).to(dev),
        segs=torch.from_numpy(np.asarray(segs, dtype=np.int32).reshape(-1, 4)).to(dev),
        seg_start=torch.from_numpy(np.asarray(starts, dtype=np.int32)).to(dev), W=W)
    # Oracle: compact float32 pool with the same keys.
    o_kp = np.full((used * BS, HKV, D), np.nan, dtype=np.float32)
    o_vp = np.full_like(o_kp, np.nan)
    slots_hist = []
    for b, (sq, L, _) in enumerate(ROWS):
        o_slots = pa.slot_mapping(o_table[b], range(L), BS)
        pa.kv_write(o_kp, o_slots, k_rows[b].float().numpy())
        pa.kv_write(o_vp, o_slots, v_rows[b].float().numpy())
        slots_hist.append(_lib.slot_mapping(table[b, : n_blocks[b]], 0, L - sq, BS))
    want = pa.paged_attention(q.float().numpy(), o_kp, o_vp, o_table, qsl, seq_lens, D ** -0.5, BS, o_segs)
    return dict(q=q.to(dev), k_rows=k_rows, v_rows=v_rows, k_pool=k_pool, v_pool=v_pool, want=want,
                o_kp=o_kp, o_table=o_table, slots_hist=slots_hist, n_blocks=n_blocks, table_np=table, **meta)


@pytest.fixture(scope="module")
def big():
    s = _setup()
    yield s
    del s
    torch.cuda.empty_cache()


def _write_all(s):
    """Write every row's history with paged_kv_write; return the current tokens' k, v, slots."""
    from paged_kv_cache_181_gb300 import _lib

    dev = s["q"].device
    ks, vs, cur = [], [], []
    for b, (sq, L, _) in enumerate(ROWS):
        hs = torch.from_numpy(s["slots_hist"][b]).to(dev)
        _lib.paged_kv_write(s["k_rows"][b][: L - sq].to(dev), s["v_rows"][b][: L - sq].to(dev), hs, s["k_pool"],
                            s["v_pool"], flags=_lib.PKV_CHECK_BOUNDS)
        ks.append(s["k_rows"][b][L - sq :])
        vs.append(s["v_rows"][b][L - sq :])
        cur.append(_lib.slot_mapping(s["table_np"][b, : s["n_blocks"][b]], L - sq, sq, BS))
    return (torch.cat(ks).to(dev).contiguous(), torch.cat(vs).to(dev).contiguous(),
            torch.from_numpy(np.concatenate(cur)).to(dev))


def _check(out, s):
    max_abs, mean_abs = cases.compare(out.float().cpu().numpy(), s["want"], "bf16")
    assert max_abs <= 2e-2 and mean_abs <= 2e-3, (max_abs, mean_abs)


@pytest.mark.parametrize("fused", [False, True], ids=["two-call", "fused"])
def test_high_block_ids_tensor_core(big, fused):
    from paged_kv_cache_181_gb300 import _lib

    s = big
    k_new, v_new, slots = _write_all(s)
    args = (s["table"], s["qsl"], s["seq_lens"], max(sq for sq, _, _ in ROWS), s["W"] * BS, D ** -0.5)
    if fused:
        out = _lib.paged_kv_write_attn(s["q"], k_new, v_new, slots, s["k_pool"], s["v_pool"], *args, segs=s["segs"],
                                       seg_start=s["seg_start"], flags=_lib.PKV_CHECK_BOUNDS)
    else:
        _lib.paged_kv_write(k_new, v_new, slots, s["k_pool"], s["v_pool"], flags=_lib.PKV_CHECK_BOUNDS)
        out = _lib.paged_attn_varlen(s["q"], s["k_pool"], s["v_pool"], *args, segs=s["segs"], seg_start=s["seg_start"],
                                     flags=_lib.PKV_CHECK_BOUNDS)
    torch.cuda.synchronize()
    assert _lib.check() == 0
    _check(out, s)


def test_high_block_ids_cuda_core_and_gather(big):
    from paged_kv_cache_181_gb300 import _lib

    s = big
    k_new, v_new, slots = _write_all(s)
    _lib.paged_kv_write(k_new, v_new, slots, s["k_pool"], s["v_pool"])
    args = (s["table"], s["qsl"], s["seq_lens"], max(sq for sq, _, _ in ROWS), s["W"] * BS, D ** -0.5)
    out = _lib.paged_attn_varlen(s["q"], s["k_pool"], s["v_pool"], *args, segs=s["segs"], seg_start=s["seg_start"],
                                 flags=_lib.PKV_CHECK_BOUNDS | _lib.PKV_FORCE_SIMT)
    torch.cuda.synchronize()
    assert _lib.check() == 0
    _check(out, s)
    # Gather the rows' blocks out of the big pool: bit-exact against the compact oracle pool.
    stage_k = torch.empty((len(ROWS), s["W"] * BS, HKV, D), dtype=torch.bfloat16, device=out.device)
    stage_v = torch.empty_like(stage_k)
    _lib.paged_kv_gather(s["k_pool"], s["v_pool"], s["table"], stage_k, stage_v, flags=_lib.PKV_CHECK_BOUNDS)
    torch.cuda.synchronize()
    assert _lib.check() == 0
    for b, (_, L, _) in enumerate(ROWS):
        want = pa.gather_row_kv(s["o_kp"], s["o_table"][b], L, BS)
        assert np.array_equal(stage_k[b, :L].float().cpu().numpy(), want)
