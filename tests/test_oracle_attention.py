"""Pins for the oracle's paged masked attention and KV write.

Each check ties the oracle to something other than itself: a library attention
routine (torch's scaled_dot_product_attention in float64), closed forms, the
same tokens laid out contiguously, NaN-poisoned unwritten slots (the pages'
``_poison_pools`` / ``_write_prepared_chunk`` technique in test_paged_attention.py),
and the float32 twin at the pages' CPU tolerance of 1e-5.
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import pagedattn as pa

BS = 16


def make_paged(rng, kv_lens, hkv, d, num_blocks, dtype=np.float64):
    """Random contiguous K/V per row, placed into a pool through a shuffled table."""
    n_tab = [-(-L // BS) for L in kv_lens]
    width = max(n_tab)
    perm = rng.permutation(num_blocks)
    table = np.zeros((len(kv_lens), width), dtype=np.int64)
    kpool = np.full((num_blocks * BS, hkv, d), np.nan, dtype=dtype)
    vpool = np.full((num_blocks * BS, hkv, d), np.nan, dtype=dtype)
    k_rows, v_rows = [], []
    used = 0
    for b, L in enumerate(kv_lens):
        table[b, : n_tab[b]] = perm[used : used + n_tab[b]]
        used += n_tab[b]
        k = rng.standard_normal((L, hkv, d))
        v = rng.standard_normal((L, hkv, d))
        slots = pa.slot_mapping(table[b], range(L), BS)
        pa.kv_write(kpool, slots, k)
        pa.kv_write(vpool, slots, v)
        k_rows.append(k)
        v_rows.append(v)
    return kpool, vpool, table, k_rows, v_rows


def sdpa(q, k, v, mask, scale):
    """torch SDPA on one row: q [Sq,H,D], k/v [L,Hkv,D] (GQA by repeating KV heads)."""
    h, hkv = q.shape[1], k.shape[1]
    kk = torch.from_numpy(k).repeat_interleave(h // hkv, dim=1)
    vv = torch.from_numpy(v).repeat_interleave(h // hkv, dim=1)
    qt = torch.from_numpy(q).transpose(0, 1)[None]
    out = F.scaled_dot_product_attention(
        qt, kk.transpose(0, 1)[None], vv.transpose(0, 1)[None],
        attn_mask=None if mask is None else torch.from_numpy(mask)[None, None], scale=scale,
    )
    return out[0].transpose(0, 1).numpy()


def direct_mask(spans, offset, qlen, seq_len):
    m = np.zeros((qlen, seq_len), dtype=bool)
    for i in range(qlen):
        p = offset + i
        lim = p + 1
        for a, b in spans:
            if a <= p < b:
                lim = b
        m[i, :lim] = True
    return m


@pytest.mark.parametrize("hq,hkv", [(4, 4), (6, 2), (5, 1)])
def test_full_attention_matches_sdpa_and_gqa_grouping(hq, hkv):
    rng = np.random.default_rng(7)
    kv_lens, sq = [37, 20], [5, 20]
    d = 16
    kpool, vpool, table, k_rows, v_rows = make_paged(rng, kv_lens, hkv, d, 16)
    qsl = np.concatenate([[0], np.cumsum(sq)])
    q = rng.standard_normal((qsl[-1], hq, d))
    scale = 0.37
    out = pa.paged_attention(q, kpool, vpool, table, qsl, kv_lens, scale, BS)
    for b in range(2):
        want = sdpa(q[qsl[b] : qsl[b + 1]], k_rows[b], v_rows[b], None, scale)
        np.testing.assert_allclose(out[qsl[b] : qsl[b + 1]], want, rtol=1e-12, atol=1e-12)


def test_piecewise_masks_match_sdpa_with_explicit_mask():
    rng = np.random.default_rng(11)
    cases = [
        ([], 9, 23),
        ([(14, 18)], 9, 23),
        ([(5, 16), (19, 21)], 9, 23),
        ([(0, 30)], 12, 30),
        ([(16, 17), (18, 26), (27, 29)], 16, 29),
    ]
    for spans, sq, L in cases:
        kpool, vpool, table, k_rows, v_rows = make_paged(rng, [L], 2, 8, 8)
        q = rng.standard_normal((sq, 4, 8))
        off = L - sq
        segs = pa.build_segments(spans, off, sq)
        out = pa.paged_attention(q, kpool, vpool, table, [0, sq], [L], 0.5, BS, [segs])
        want = sdpa(q, k_rows[0], v_rows[0], direct_mask(spans, off, sq, L), 0.5)
        np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)


def test_single_causal_segment_is_textbook_causal():
    rng = np.random.default_rng(3)
    L = 40
    kpool, vpool, table, k_rows, v_rows = make_paged(rng, [L], 3, 8, 4)
    q = rng.standard_normal((L, 3, 8))
    segs = pa.build_segments([], 0, L)
    out = pa.paged_attention(q, kpool, vpool, table, [0, L], [L], 0.25, BS, [segs])
    qt = torch.from_numpy(q).transpose(0, 1)[None]
    want = F.scaled_dot_product_attention(
        qt, torch.from_numpy(k_rows[0]).transpose(0, 1)[None], torch.from_numpy(v_rows[0]).transpose(0, 1)[None],
        is_causal=True, scale=0.25,
    )[0].transpose(0, 1).numpy()
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)


def test_paged_equals_dense_under_two_shuffles():
    kv_lens, sq = [45, 33], [7, 33]
    outs = []
    for seed in (1, 2):
        rng = np.random.default_rng(100)
        k_rows = [rng.standard_normal((L, 2, 8)) for L in kv_lens]
        v_rows = [rng.standard_normal((L, 2, 8)) for L in kv_lens]
        q = rng.standard_normal((sum(sq), 2, 8))
        perm = np.random.default_rng(seed).permutation(12)
        table = np.zeros((2, 3), dtype=np.int64)
        kpool = np.full((12 * BS, 2, 8), np.nan)
        vpool = np.full((12 * BS, 2, 8), np.nan)
        used = 0
        for b, L in enumerate(kv_lens):
            n = -(-L // BS)
            table[b, :n] = perm[used : used + n]
            used += n
            slots = pa.slot_mapping(table[b], range(L), BS)
            pa.kv_write(kpool, slots, k_rows[b])
            pa.kv_write(vpool, slots, v_rows[b])
        qsl = [0, sq[0], sq[0] + sq[1]]
        outs.append(pa.paged_attention(q, kpool, vpool, table, qsl, kv_lens, 0.3, BS))
        # and the contiguous layout: identity table over a pool that holds the row in order
        for b, L in enumerate(kv_lens):
            dense = pa.segment_attention(q[qsl[b] : qsl[b + 1], 0], k_rows[b][:, 0], v_rows[b][:, 0], 0.3, False)
            np.testing.assert_array_equal(outs[-1][qsl[b] : qsl[b + 1], 0], dense)
    np.testing.assert_array_equal(outs[0], outs[1])


def test_zero_query_gives_mean_of_visible_values():
    rng = np.random.default_rng(5)
    L, sq = 29, 11
    kpool, vpool, table, k_rows, v_rows = make_paged(rng, [L], 1, 4, 4)
    q = np.zeros((sq, 1, 4))
    spans = [(20, 24)]
    off = L - sq
    segs = pa.build_segments(spans, off, sq)
    out = pa.paged_attention(q, kpool, vpool, table, [0, sq], [L], 0.9, BS, [segs])
    v = v_rows[0][:, 0]
    for i in range(sq):
        p = off + i
        lim = 24 if 20 <= p < 24 else p + 1
        np.testing.assert_allclose(out[i, 0], v[:lim].mean(axis=0), rtol=1e-13, atol=1e-13)


def test_single_key_returns_its_value():
    rng = np.random.default_rng(9)
    kpool, vpool, table, k_rows, v_rows = make_paged(rng, [1], 2, 8, 3)
    q = rng.standard_normal((1, 4, 8)) * 10
    out = pa.paged_attention(q, kpool, vpool, table, [0, 1], [1], 0.125, BS)
    for h in range(4):
        np.testing.assert_array_equal(out[0, h], v_rows[0][0, h // 2])


def test_scale_matters():
    rng = np.random.default_rng(13)
    kpool, vpool, table, k_rows, v_rows = make_paged(rng, [20], 1, 8, 2)
    q = rng.standard_normal((4, 1, 8))
    a = pa.paged_attention(q, kpool, vpool, table, [0, 4], [20], 0.1, BS)
    b = pa.paged_attention(q, kpool, vpool, table, [0, 4], [20], 1.0, BS)
    assert np.abs(a - b).max() > 1e-3
    np.testing.assert_allclose(b, sdpa(q, k_rows[0], v_rows[0], None, 1.0), rtol=1e-12, atol=1e-12)


def test_nan_poisoned_unwritten_slots_are_never_read():
    # Partial last block (kv 37 = 2 blocks + 5) and padding entries that point at a NaN block.
    rng = np.random.default_rng(21)
    kv_lens = [37, 16]
    kpool, vpool, table, _, _ = make_paged(rng, kv_lens, 2, 8, 10)
    poison = 9
    assert poison not in table[0, :3] and poison not in table[1, :1]
    table = np.concatenate([table, np.full((2, 4), poison)], axis=1)
    table[1, 1:] = poison
    q = rng.standard_normal((8, 2, 8))
    out = pa.paged_attention(q, kpool, vpool, table, [0, 4, 8], kv_lens, 0.3, BS)
    assert np.isfinite(out).all()


def test_sampled_rows_equal_full_evaluation():
    rng = np.random.default_rng(17)
    L, sq = 50, 30
    kpool, vpool, table, _, _ = make_paged(rng, [L], 2, 8, 4)
    q = rng.standard_normal((sq, 4, 8))
    segs = pa.build_segments([(25, 33), (40, 44)], L - sq, sq)
    full = pa.paged_attention(q, kpool, vpool, table, [0, sq], [L], 0.3, BS, [segs])
    sample = {(0, 1): np.array([0, 7, 12, 13, 29]), (0, 3): np.array([5])}
    part = pa.paged_attention(q, kpool, vpool, table, [0, sq], [L], 0.3, BS, [segs], sample=sample)
    for (b, h), rows in sample.items():
        # Same arithmetic; BLAS may block a different row count differently.
        np.testing.assert_allclose(part[rows, h], full[rows, h], rtol=1e-13, atol=1e-14)
    assert np.isnan(part[:, 0]).all()


def test_float32_twin_within_cpu_tolerance():
    rng = np.random.default_rng(23)
    kpool, vpool, table, _, _ = make_paged(rng, [300, 128], 2, 64, 40)
    q = rng.standard_normal((100, 4, 64))
    qsl = [0, 60, 100]
    segs = [pa.build_segments([(250, 270)], 240, 60), []]
    a = pa.paged_attention(q, kpool, vpool, table, qsl, [300, 128], 0.125, BS, segs)
    b = pa.paged_attention(q, kpool.astype(np.float32), vpool.astype(np.float32), table, qsl, [300, 128],
                           0.125, BS, segs, dtype=np.float32)
    assert b.dtype == np.float32
    np.testing.assert_allclose(b, a, rtol=1e-5, atol=1e-5)


def test_kv_write_is_a_bit_copy_and_skips_negative_slots():
    pool = np.full((64, 2, 4), np.nan, dtype=np.float32)
    src = np.random.default_rng(0).standard_normal((5, 2, 4)).astype(np.float32)
    slots = np.array([3, 17, -1, 40, 63])
    pa.kv_write(pool, slots, src)
    for t, s in enumerate(slots):
        if s >= 0:
            assert pool[s].tobytes() == src[t].tobytes()
    assert np.isnan(pool[[0, 1, 2, 4, 62]]).all()
    with pytest.raises(IndexError):
        pa.kv_write(pool, np.array([64]), src[:1])


def test_write_then_read_through_the_table_round_trips():
    # After the write, cache[table[p // 16], p % 16] is the token written at position p.
    rng = np.random.default_rng(31)
    blocks = rng.permutation(20)[:6]
    src = rng.standard_normal((70, 1, 2))
    pool = np.full((20 * BS, 1, 2), np.nan)
    first = 19  # chunk starting mid-block
    slots = pa.slot_mapping(blocks, range(first, first + 70), BS)
    pa.kv_write(pool, slots, src)
    cache = pool.reshape(20, BS, 1, 2)
    for t in range(70):
        p = first + t
        assert (cache[blocks[p // BS], p % BS] == src[t]).all()


def test_slot_mapping_ragged_chunk_starts_mid_block():
    # A 24-token chunk after a 24-token history starts 8 slots into the
    # history's tail block (test_paged_attention.py,
    # test_a_ragged_scratch_chunk_is_physically_continuous_with_its_history).
    blocks = [11, 5, 9, 2]
    slots = pa.slot_mapping(blocks, range(24, 48), BS)
    assert slots[0] == 5 * 16 + 8
    assert slots[7] == 5 * 16 + 15 and slots[8] == 9 * 16


def test_attention_flops_count_visible_pairs():
    # Brute force over the direct mask.
    for spans, sq, L in [([], 7, 20), ([(15, 18)], 7, 20), ([(0, 3), (5, 9)], 10, 10)]:
        segs = pa.build_segments(spans, L - sq, sq)
        pairs = direct_mask(spans, L - sq, sq, L).sum()
        assert pa.attention_flops([0, sq], [L], [segs], 3, 8) == 4 * 8 * 3 * pairs
    # No segments: every key is visible.
    assert pa.attention_flops([0, 5], [9], None, 2, 4) == 4 * 4 * 2 * 45


def test_rows_whose_query_is_not_a_suffix_match_sdpa():
    # Packed rows carry their own query offset (kv_start_pos); keys after the query exist
    # but only a full span reaching past the query makes them visible.
    rng = np.random.default_rng(13)
    cases = [
        ([], 3, 5, 21),              # causal only: keys after the query stay hidden
        ([(3, 8)], 3, 5, 21),        # full over exactly the query
        ([(2, 19)], 3, 5, 21),       # a full span reaching past the query
        ([(0, 4), (6, 12)], 2, 9, 30),
        ([(10, 12)], 0, 16, 16),     # suffix case for comparison
    ]
    for spans, off, sq, L in cases:
        kpool, vpool, table, k_rows, v_rows = make_paged(rng, [L], 2, 8, 8)
        q = rng.standard_normal((sq, 4, 8))
        segs = pa.build_segments(spans, off, sq)
        out = pa.paged_attention(q, kpool, vpool, table, [0, sq], [L], 0.5, BS, [segs], query_offsets=[off])
        want = sdpa(q, k_rows[0], v_rows[0], direct_mask(spans, off, sq, L), 0.5)
        np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)
        pairs = direct_mask(spans, off, sq, L).sum()
        assert pa.attention_flops([0, sq], [L], [segs], 4, 8, query_offsets=[off]) == 4 * 8 * 4 * pairs


def test_query_offset_outside_the_sequence_is_refused():
    rng = np.random.default_rng(14)
    kpool, vpool, table, _, _ = make_paged(rng, [10], 1, 4, 4)
    q = rng.standard_normal((4, 1, 4))
    with pytest.raises(ValueError):
        pa.paged_attention(q, kpool, vpool, table, [0, 4], [10], 1.0, BS, None, query_offsets=[7])
