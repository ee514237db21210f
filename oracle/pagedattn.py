"""Oracle: KV write, segment construction and paged masked attention (plain NumPy).

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.

Sources (page title, then the function on that page):

* ``paged_attention.py`` (vllm_omni/experimental/ar_diffusion/kv_cache):
  ``_paged_write_attn_impl`` (the pool write ``pool[slots] = x``),
  ``_reference_paged_attention`` (gather through the block table, then
  softmax(Q K^T * scale) V with float32 statistics), ``ar_diffusion_paged_attention``
  (non-causal paged attention over ``query_start_loc`` / ``seq_lens``).
* ``piecewise_attn.py`` (vllm_omni/diffusion/attention/backends/utils):
  the module docstring (bottom-right causal convention), ``build_segments``,
  ``piecewise_attn`` (one attention call per segment, query anchored at
  ``Skv - Sq``), ``build_paged_piecewise_plan`` (span / query-range validation).
* ``paged_attention_adapter.py`` (vllm_omni/diffusion/diffusion_kv):
  ``DiffusionPagedAttentionLayerAdapter.__init__`` (``num_heads`` divisible by
  ``num_kv_heads``).

Arithmetic is float64 unless ``dtype=np.float32`` is asked for; the float32
twin exists only so the CPU baseline can be timed at the GPU's accumulation
precision.  Probabilities are NOT rounded to the value dtype before P.V (the
pages' CPU reference casts them; the GPU tolerance covers that rounding).
"""

from __future__ import annotations

import math
from typing import NamedTuple, Sequence

import numpy as np

CAUSAL = "causal"
FULL = "full"


# ----------------------------------------------------------------------------
# KV write (paged_attention.py, _paged_write_attn_impl)
# ----------------------------------------------------------------------------


def slot_mapping(block_ids: Sequence[int], positions: Sequence[int], block_size: int) -> np.ndarray:
    """Slot of each position: the position's block, times the block size, plus its offset.

    ``block_ids[i]`` is the physical block holding logical block ``i`` (positions
    ``i*block_size .. i*block_size+block_size-1``).  This is the addressing the
    pages' CPU reference uses to read the cache (``block_table[i, pos // bs]``
    and ``pos % bs`` in ``_reference_paged_attention``), and the ragged-chunk test
    fixes its first slot at ``tail_block * 16 + 8`` for a chunk that starts 8
    slots into the history's tail block.
    """
    out = np.empty(len(positions), dtype=np.int64)
    for t, pos in enumerate(positions):
        pos = int(pos)
        out[t] = int(block_ids[pos // block_size]) * block_size + pos % block_size
    return out


def kv_write(pool: np.ndarray, slots: np.ndarray, src: np.ndarray) -> None:
    """``pool[slot[t]] = src[t]`` for every token ``t`` (a bit copy, in place).

    ``pool`` is the flat ``[num_blocks * block_size, H_kv, D]`` pool and ``src``
    is ``[T, H_kv, D]`` in the pool's dtype.  A negative slot means "skip this
    token" (a convention of this library; the pages never pass one).
    """
    if src.shape[0] != slots.shape[0]:
        raise ValueError("one slot per source token")
    for t in range(src.shape[0]):
        s = int(slots[t])
        if s < 0:
            continue
        if s >= pool.shape[0]:
            raise IndexError(f"slot {s} outside a pool of {pool.shape[0]} slots")
        pool[s] = src[t]


# ----------------------------------------------------------------------------
# Segments (piecewise_attn.py, build_segments / build_paged_piecewise_plan)
# ----------------------------------------------------------------------------


class Segment(NamedTuple):
    q_start: int
    q_end: int
    kv_end: int
    mode: str  # CAUSAL or FULL


def validate_spans(spans: Sequence[tuple[int, int]], query_offset: int, query_len: int, seq_len: int) -> None:
    """Raise ValueError unless the spans and query range are well formed.

    Spans must be sorted, non-overlapping and satisfy ``0 <= start < end <= seq_len``;
    the query range must satisfy ``0 <= offset``, ``len > 0`` and
    ``offset + len <= seq_len`` (``build_paged_piecewise_plan``).
    """
    previous_end = 0
    for start, end in spans:
        if start < previous_end or not (0 <= start < end <= seq_len):
            raise ValueError("spans must be sorted, non-overlapping, and within the sequence")
        previous_end = end
    if query_offset < 0 or query_len <= 0 or query_offset + query_len > seq_len:
        raise ValueError("query range must be within the sequence")


def build_segments(spans: Sequence[tuple[int, int]], query_offset: int, query_len: int) -> list[Segment]:
    """Cover the query range ``[off, off+len)`` with causal and full segments.

    Walk the spans in order with a cursor starting at the query's first
    position.  Each span is clipped to the query range and dropped if nothing
    is left.  A gap before the clipped span becomes a causal segment whose key
    range ends where the gap ends; the clipped span itself becomes a full
    segment whose key range ends at the span's UNclipped end.  Whatever follows
    the last span is a causal tail.  (``build_segments``.)
    """
    q_lo = query_offset
    q_hi = query_offset + query_len
    out: list[Segment] = []
    cursor = q_lo
    for a, b in spans:
        lo = max(a, q_lo)
        hi = min(b, q_hi)
        if lo >= hi:
            continue
        if cursor < lo:
            out.append(Segment(cursor, lo, lo, CAUSAL))
        out.append(Segment(lo, hi, b, FULL))
        cursor = hi
    if cursor < q_hi:
        out.append(Segment(cursor, q_hi, q_hi, CAUSAL))
    return out


# ----------------------------------------------------------------------------
# Attention
# ----------------------------------------------------------------------------


def segment_attention(
    q: np.ndarray,
    k: np.ndarray,
    v: np.ndarray,
    scale: float,
    causal: bool,
    *,
    rows: np.ndarray | None = None,
    segment_rows: int | None = None,
    dtype=np.float64,
) -> np.ndarray:
    """One attention call ``attn(Q[s:e], K[:kv_end], V[:kv_end], causal)`` for one head.

    ``q`` is ``[n, D]`` and ``k``/``v`` are ``[kv_end, D]``.  With ``causal`` the
    mask is anchored at the bottom-right corner (``piecewise_attn.py`` module
    docstring): row ``r`` of an ``S``-row block over ``K`` keys sees key ``j``
    exactly when ``j <= r + (K - S)``.  ``rows`` gives each row's index ``r``
    inside its segment of ``segment_rows`` rows when only some rows are
    evaluated (default: all of them, ``r = 0..n-1``, ``S = n``).

    Softmax over the visible keys; a row that sees no key returns zeros (this
    cannot happen under the bottom-right convention with ``S <= K``).
    """
    n = q.shape[0]
    n_keys = k.shape[0]
    if rows is None:
        rows = np.arange(n)
        segment_rows = n
    rows = np.asarray(rows)
    kd = k.astype(dtype)
    vd = v.astype(dtype)
    out = np.zeros((n, vd.shape[1]), dtype=dtype)
    if n_keys == 0:
        return out
    shift = n_keys - int(segment_rows)
    j = np.arange(n_keys)[None, :]
    # Rows are independent; evaluate them a few at a time to bound memory.
    step = max(1, (1 << 22) // n_keys)
    for r0 in range(0, n, step):
        r1 = min(n, r0 + step)
        scores = (q[r0:r1].astype(dtype) @ kd.T) * dtype(scale)  # [rows, K]
        if causal:
            visible = j <= (rows[r0:r1, None] + shift)
        else:
            visible = np.ones_like(scores, dtype=bool)
        scores = np.where(visible, scores, -np.inf)
        any_visible = visible.any(axis=1)
        m = np.where(any_visible, scores.max(axis=1), 0.0).astype(dtype)
        p = np.where(visible, np.exp(scores - m[:, None]), 0.0).astype(dtype)
        denom = p.sum(axis=1)
        num = p @ vd
        safe = np.where(any_visible, denom, 1.0)
        out[r0:r1] = np.where(any_visible[:, None], num / safe[:, None], 0.0)
    return out


def gather_row_kv(cache_rows: np.ndarray, table_row: Sequence[int], kv_len: int, block_size: int) -> np.ndarray:
    """Contiguous ``[kv_len, H_kv, D]`` keys (or values) of one batch row.

    Key ``j`` lives in physical block ``table_row[j // bs]`` at offset ``j % bs``
    (``_reference_paged_attention``).  ``cache_rows`` is the flat pool
    ``[num_blocks * bs, H_kv, D]``; only the first ``ceil(kv_len / bs)`` table
    entries are touched, so table padding is never read.
    """
    idx = np.empty(kv_len, dtype=np.int64)
    for j in range(kv_len):
        idx[j] = int(table_row[j // block_size]) * block_size + j % block_size
    return cache_rows[idx]


def kv_head_of(h: int, num_heads: int, num_kv_heads: int) -> int:
    """KV head read by query head ``h``: contiguous groups of ``num_heads / num_kv_heads``.

    The pages only require divisibility (``paged_attention_adapter.py``,
    ``DiffusionPagedAttentionLayerAdapter.__init__``); contiguous grouping is
    the reading this library takes.
    """
    if num_kv_heads <= 0 or num_heads % num_kv_heads:
        raise ValueError("num_heads must be a positive multiple of num_kv_heads")
    return h // (num_heads // num_kv_heads)


def paged_attention(
    query: np.ndarray,
    key_pool: np.ndarray,
    value_pool: np.ndarray,
    block_table: np.ndarray,
    query_start_loc: Sequence[int],
    seq_lens: Sequence[int],
    scale: float,
    block_size: int,
    segments: Sequence[Sequence[Segment]] | None = None,
    *,
    dtype=np.float64,
    sample: dict | None = None,
    query_offsets: Sequence[int] | None = None,
) -> np.ndarray:
    """Paged varlen attention with an optional piecewise causal/full mask per batch row.

    ``query`` is ``[Tq, Hq, D]`` packed by ``query_start_loc``; the pools are
    ``[num_blocks * bs, H_kv, D]``; ``block_table`` is ``[B, W]``.  For row ``b``
    with ``Sq`` queries and ``L = seq_lens[b]`` keys, the keys are gathered
    through the block table.  Local query ``i`` sits at global position
    ``query_offsets[b] + i``; by default the query is the suffix of the key
    sequence, ``query_offsets[b] = L - Sq`` (``piecewise_attn`` anchors the
    query at ``Skv - Sq``).  Another offset is a packed row whose write span
    starts at ``kv_start_pos`` (``DiffusionPagedAttentionRow``, with
    ``build_paged_piecewise_plan`` taking one query offset per row); its
    segments must come from ``build_segments`` with that offset.

    ``segments[b]`` (global coordinates, from ``build_segments``) splits row b's
    queries into causal and full pieces, each attended exactly as
    ``piecewise_attn`` dispatches it.  ``segments=None`` or an empty entry
    means the pages' default ``causal=False`` attention over all ``L`` keys.

    ``sample`` (optional) maps ``(b, h)`` to an array of local query indices;
    only those outputs are computed (the others stay NaN).  The result is
    ``[Tq, Hq, D]`` float64 (or ``dtype``).
    """
    tq, hq, d = query.shape
    hkv = key_pool.shape[1]
    out = np.full((tq, hq, d), np.nan, dtype=dtype)
    n_rows = len(seq_lens)
    for b in range(n_rows):
        q0, q1 = int(query_start_loc[b]), int(query_start_loc[b + 1])
        sq, kv_len = q1 - q0, int(seq_lens[b])
        if sq == 0:
            continue
        if sq > kv_len:
            raise ValueError("the query must be a suffix of the key sequence (Sq <= seq_len)")
        k_all = gather_row_kv(key_pool, block_table[b], kv_len, block_size)
        v_all = gather_row_kv(value_pool, block_table[b], kv_len, block_size)
        offset = kv_len - sq if query_offsets is None else int(query_offsets[b])
        if offset < 0 or offset + sq > kv_len:
            raise ValueError("the row's query range must lie within its key sequence")
        row_segs = list(segments[b]) if segments is not None and segments[b] else [
            Segment(offset, kv_len, kv_len, FULL)
        ]
        for h in range(hq):
            g = kv_head_of(h, hq, hkv)
            wanted = None if sample is None else set(int(i) for i in sample.get((b, h), ()))
            if wanted is not None and not wanted:
                continue
            for seg in row_segs:
                s_lo, s_hi = seg.q_start - offset, seg.q_end - offset
                if not (0 <= s_lo <= s_hi <= sq):
                    raise ValueError("segment outside the row's query range")
                kv_end = min(int(seg.kv_end), kv_len)
                local = np.arange(s_lo, s_hi)
                if wanted is not None:
                    local = np.array([i for i in local if i in wanted], dtype=np.int64)
                    if local.size == 0:
                        continue
                res = segment_attention(
                    query[q0 + local, h],
                    k_all[:kv_end, g],
                    v_all[:kv_end, g],
                    scale,
                    seg.mode == CAUSAL,
                    rows=local - s_lo,
                    segment_rows=s_hi - s_lo,
                    dtype=dtype,
                )
                out[q0 + local, h] = res
    return out


def attention_flops(query_start_loc: Sequence[int], seq_lens: Sequence[int], segments, num_heads: int, head_dim: int,
                    query_offsets: Sequence[int] | None = None) -> int:
    """Algorithmic FLOPs: ``4 * D * Hq * (visible (query, key) pairs)``, summed over rows.

    Two multiply-adds per visible pair and head dimension: one for ``Q K^T``,
    one for ``P V``.
    """
    pairs = 0
    for b in range(len(seq_lens)):
        sq = int(query_start_loc[b + 1]) - int(query_start_loc[b])
        kv_len = int(seq_lens[b])
        offset = kv_len - sq if query_offsets is None else int(query_offsets[b])
        row_segs = list(segments[b]) if segments is not None and segments[b] else [
            Segment(offset, kv_len, kv_len, FULL)
        ]
        for seg in row_segs:
            n = seg.q_end - seg.q_start
            kv_end = min(seg.kv_end, kv_len)
            if seg.mode == FULL:
                pairs += n * kv_end
            else:
                shift = kv_end - n
                for r in range(n):
                    pairs += max(0, min(kv_end, r + shift + 1))
    return 4 * head_dim * num_heads * pairs


def default_scale(head_dim: int) -> float:
    """``head_dim ** -0.5``, the scale every call on the pages passes."""
    return 1.0 / math.sqrt(head_dim)
