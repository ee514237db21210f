"""Pins for the oracle's visible-window selection and fixed-width block table.

Checked against worked numbers from the pages (tests/golden/workload_geometry.json)
and against the window's definition by positions -- the sink ``[0, S)`` plus the
last ``W`` positions -- as the pages' slot-by-slot tests state it
(test_paged_attention.py, ``_window_positions`` and
``test_the_shipped_geometry_reads_exactly_the_window_on_every_tick``).
"""

import json
import os

import pytest

from oracle import window as ow
from paged_kv_cache_181_gb300 import configs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
BS = 16


def load():
    with open(os.path.join(GOLDEN, "workload_geometry.json")) as f:
        return json.load(f)


def read_positions(row_blocks, blocks, video_len):
    """Positions the listed blocks hold, in listed order, cut at video_len."""
    where = {b: i for i, b in enumerate(row_blocks) if b != ow.NULL_BLOCK}
    out = []
    for b in blocks:
        out.extend(where[b] * BS + o for o in range(BS))
    return out[:video_len]


def test_frame_geometry():
    g = load()["frame"]
    assert (480 // 16) * (832 // 16) == g["tokens_per_frame"]
    assert g["tokens_per_frame"] % BS == g["mod_block"]
    assert ow.ceil_div(g["tokens_per_frame"], BS) == g["blocks_per_frame"]


def test_width_of_the_shipped_sink_and_window():
    g = load()["sink9_window9"]
    assert (g["sink_tokens"] + g["window_tokens"]) // BS == g["sum_blocks"]
    assert ow.max_video_blocks(g["chunk"], BS, g["sink_tokens"], g["window_tokens"]) == g["max_video_blocks"]


@pytest.mark.parametrize(
    "chunk,sink_chunks,window_chunks,per_tick,ticks",
    [(1560, 9, 9, 3, 12), (24, 1, 2, 1, 10), (24, 0, 2, 1, 10), (24, 1, 3, 1, 10), (16, 0, 2, 1, 6), (40, 2, 2, 1, 12)],
)
def test_rollout_reads_exactly_the_window(chunk, sink_chunks, window_chunks, per_tick, ticks):
    sink, window = sink_chunks * chunk, window_chunks * chunk
    width = ow.max_video_blocks(chunk, BS, sink, window)
    row_blocks = list(range(1000, 1000 + 100000))  # block i holds logical block i
    kv_lens = []
    filled = False
    for tick in range(ticks):
        end = (tick + 1) * per_tick * chunk
        blocks, video_len = ow.visible_video_blocks(row_blocks, end, sink, window, BS)
        assert len(blocks) <= width, f"tick {tick}: {len(blocks)} blocks > width {width}"
        read = read_positions(row_blocks, blocks, video_len)
        assert len(set(read)) == len(read) and max(read) < end
        kept = ow.window_positions(end, sink, window)
        assert kept <= set(read), f"tick {tick}: window tokens not read"
        # Whole blocks are read: each of the two boundaries adds at most bs-1 tokens.
        assert video_len <= min(end, sink + window + 2 * (BS - 1))
        extra = set(read) - kept
        assert all(p // BS in {q // BS for q in kept} for p in extra)
        kv_lens.append(video_len)
        filled = filled or end > sink + window
    assert filled


def test_ragged_window_bound():
    g = load()["ragged24"]
    assert g["sink_tokens"] + g["window_tokens"] == g["max_video_tokens"]
    assert g["max_video_tokens"] % BS != 0
    assert ow.max_video_blocks(g["chunk"], BS, g["sink_tokens"], g["window_tokens"]) == g["max_video_blocks"]
    assert g["max_video_tokens"] + 2 * (BS - 1) == g["kv_len_bound"]


def test_evicted_blocks_are_skipped_by_position():
    # Blocks wholly outside the window evicted (null): the listed blocks do not change.
    chunk, sink, window = 24, 24, 48
    end = 8 * chunk
    full = list(range(50, 50 + 40))
    blocks, video_len = ow.visible_video_blocks(full, end, sink, window, BS)
    evicted = list(full)
    for i in range(len(evicted)):
        if i * BS >= sink and (i + 1) * BS <= end - window:
            evicted[i] = ow.NULL_BLOCK
    assert ow.visible_video_blocks(evicted, end, sink, window, BS) == (blocks, video_len)
    # A reset keeps only the sink: window blocks that are no longer resident are skipped, not read.
    reset = list(full)
    for i in range(ow.ceil_div(sink, BS), (end - chunk) // BS):
        reset[i] = ow.NULL_BLOCK
    b2, l2 = ow.visible_video_blocks(reset, end, sink, window, BS)
    assert all(b != ow.NULL_BLOCK for b in b2)
    assert l2 < video_len


def test_action_after_partial_video_block_is_refused():
    blocks, video_len = ow.visible_video_blocks([3, 4], 24, 0, 48, BS)
    assert video_len == 24
    with pytest.raises(ValueError):
        ow.block_table_row(blocks, video_len, [7], 3, BS, 5)


def test_block_table_pads_with_block_zero_and_adds_action_length():
    row, kv_len = ow.block_table_row([5, 6], 32, [9], 3, BS, 4)
    assert row == [5, 6, 9, 0] and kv_len == 35
    row, kv_len = ow.block_table_row([5, 6], 30, [], 0, BS, 3)
    assert row == [5, 6, 0] and kv_len == 30
    with pytest.raises(ValueError):
        ow.block_table_row([1, 2, 3], 48, [], 0, BS, 2)


def test_fixed_width_example_from_the_pages():
    # 16-token chunks, window 2 chunks, no sink: width = window / bs + 1
    # (test_paged_attention.py, test_block_table_padded_to_fixed_width).
    assert ow.table_width(16, BS, 0, 32, 0) == 32 // 16 + 1


def test_workload_geometry_golden():
    g = {w["name"]: w for w in load()["workloads"]}
    for name, wl in configs.ALL.items():
        want = g[name]
        assert wl.end_tokens == want["end"]
        n_video = ow.ceil_div(wl.end_tokens, BS)
        row_blocks = list(range(1, n_video + 1))
        blocks, video_len = ow.visible_video_blocks(row_blocks, wl.end_tokens, wl.sink_tokens, wl.window_tokens, BS)
        action = list(range(5000, 5000 + ow.ceil_div(wl.action_len, BS)))
        width = ow.table_width(wl.chunk_tokens, BS, wl.sink_tokens, wl.window_tokens, wl.action_len)
        row, kv_len = ow.block_table_row(blocks, video_len, action, wl.action_len, BS, width)
        assert kv_len == want["kv_len"], name
        assert width == want["width"], name
        if "n_listed" in want:
            assert len(blocks) + len(action) == want["n_listed"], name
        if "first_listed_block_index" in want:
            assert row[0] == row_blocks[want["first_listed_block_index"]]
