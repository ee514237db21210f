"""Oracle: the visible window (sink + recent tokens) and the fixed-width block table.

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.

Sources (page title, then the function on that page), all on
``paged_attention.py`` (vllm_omni/experimental/ar_diffusion/kv_cache) unless
stated:

* ``ARDiffusionPagedForwardContext.sink_tokens`` / ``window_tokens`` -- the sink
  is ``sink_chunks * chunk_size`` leading tokens; the recent window is the
  rest of ``max_video_tokens`` and includes the current chunk.
* ``max_video_blocks`` (docstring) -- the sink's blocks are its tokens rounded
  up; the recent range starts on a chunk boundary, so it starts at most
  ``bs - gcd(chunk, bs)`` tokens past a block edge and may need that much more
  room.  (``visible_window_blocks`` itself is not on the pages; this is the
  plain reading of that docstring.)
* ``video_block_table`` -- blocks are chosen by the positions they hold: the
  sink's blocks and the blocks from the recent window's start onward; a block
  lying wholly between the two is skipped; an evicted (null) block is skipped;
  only the last listed block may be partly written; ``video_len`` counts the
  written slots of the listed blocks.
* ``build_block_table`` -- action blocks follow the video blocks and are
  refused after a partly written video block; the table is padded with block
  0 to ``max_video_blocks + max(1, ceil(action_len / bs))`` entries; the key
  length is ``video_len + action_len``.

Model of the row's storage used here: ``row_blocks[i]`` is the physical block
holding logical block ``i`` of the row (positions ``i*bs .. i*bs+bs-1``), or
``NULL_BLOCK`` when it has been evicted.  The current chunk's own blocks are
the entries from ``history // bs`` on, so a chunk that starts mid-block shares
its first block with the history's tail, as ``ensure_video_slots`` arranges.
"""

from __future__ import annotations

import math
from typing import Sequence

NULL_BLOCK = -1


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def max_video_blocks(chunk_tokens: int, block_size: int, sink_tokens: int, window_tokens: int) -> int:
    """Most blocks the visible window can span (fixes the table width)."""
    sink_blocks = ceil_div(sink_tokens, block_size)
    slack = block_size - math.gcd(chunk_tokens, block_size)
    recent_blocks = ceil_div(window_tokens + slack, block_size)
    return sink_blocks + recent_blocks


def table_width(chunk_tokens: int, block_size: int, sink_tokens: int, window_tokens: int, action_len: int) -> int:
    """Fixed table width: the window's blocks plus at least one action-capacity block."""
    action_capacity = max(1, ceil_div(action_len, block_size))
    return max_video_blocks(chunk_tokens, block_size, sink_tokens, window_tokens) + action_capacity


def visible_video_blocks(
    row_blocks: Sequence[int],
    end_tokens: int,
    sink_tokens: int,
    window_tokens: int,
    block_size: int,
) -> tuple[list[int], int]:
    """Blocks attention reads, in token order, and how many of their slots hold tokens.

    ``end_tokens`` is the position one past the current chunk's last token.
    """
    sink_end = sink_tokens
    recent_start = end_tokens - window_tokens
    n_blocks = ceil_div(end_tokens, block_size)
    if len(row_blocks) < n_blocks:
        raise ValueError("row_blocks must cover every position before end_tokens")
    blocks: list[int] = []
    video_len = 0
    for index in range(n_blocks):
        first = index * block_size
        block = int(row_blocks[index])
        if block == NULL_BLOCK:
            continue
        if first >= sink_end and first + block_size <= recent_start:
            continue  # wholly between the sink and the recent window
        if video_len % block_size:
            raise RuntimeError("the window would read past a partly written block")
        blocks.append(block)
        video_len += min(block_size, end_tokens - first)
    return blocks, video_len


def block_table_row(
    video_blocks: Sequence[int],
    video_len: int,
    action_blocks: Sequence[int],
    action_len: int,
    block_size: int,
    width: int,
) -> tuple[list[int], int]:
    """Padded block-table row and the row's key length ``video_len + action_len``."""
    if action_len > 0 and video_len % block_size:
        raise ValueError("cannot place action tokens after a partly written video block")
    ids = list(video_blocks) + (list(action_blocks[: ceil_div(action_len, block_size)]) if action_len > 0 else [])
    if not ids:
        raise RuntimeError("paged attention needs at least one key block")
    if len(ids) > width:
        raise ValueError(f"{len(ids)} blocks do not fit a table of width {width}")
    return ids + [0] * (width - len(ids)), video_len + action_len


def window_positions(end_tokens: int, sink_tokens: int, window_tokens: int) -> set[int]:
    """Positions the window must keep: the sink ``[0, S)`` and the last ``W`` positions."""
    start = max(end_tokens - window_tokens, 0)
    return set(range(min(sink_tokens, end_tokens))) | set(range(start, end_tokens))
