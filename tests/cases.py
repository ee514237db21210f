"""Oracle side of a workload: metadata, pools and expected outputs from oracle/ only.

Uses the shared seeded draws (paged_kv_cache_181_gb300.synth) and nothing of
the CUDA path.  Pools are float32 (bf16/f16 values are exact in float32) and
poisoned with NaN, so any read of a slot that was never written shows up.
"""

from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np
import torch

from oracle import pagedattn as pa
from oracle import window as ow
from paged_kv_cache_181_gb300 import configs, synth
from paged_kv_cache_181_gb300.configs import Workload


@dataclass
class OracleCase:
    table: np.ndarray
    seq_lens: np.ndarray
    qsl: np.ndarray
    slots: np.ndarray
    segments: list | None
    width: int
    k_pool: np.ndarray | None = None
    v_pool: np.ndarray | None = None
    q: np.ndarray | None = None


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float32).numpy()


def oracle_metadata(w: Workload) -> OracleCase:
    row_blocks, action_blocks = synth.allocation(w)
    bs = w.block_size
    width = ow.table_width(w.chunk_tokens, bs, w.sink_tokens, w.window_tokens, w.action_len)
    table = np.zeros((w.batch, width), dtype=np.int64)
    seq_lens = np.zeros(w.batch, dtype=np.int64)
    qsl = np.arange(w.batch + 1, dtype=np.int64) * w.q_len
    slots, segments = [], ([] if w.spans else None)
    for b in range(w.batch):
        rb = [int(x) for x in row_blocks[b]]
        ab = [int(x) for x in action_blocks[b]]
        blocks, video_len = ow.visible_video_blocks(rb, w.end_tokens, w.sink_tokens, w.window_tokens, bs)
        row, kv_len = ow.block_table_row(blocks, video_len, ab, w.action_len, bs, width)
        table[b] = row
        seq_lens[b] = kv_len
        slots.append(pa.slot_mapping(rb, range(w.history_tokens, w.end_tokens), bs))
        if w.action_len:
            slots.append(pa.slot_mapping(ab, range(w.action_len), bs))
        if segments is not None:
            pa.validate_spans(list(w.spans), kv_len - w.q_len, w.q_len, kv_len)
            segments.append(pa.build_segments(list(w.spans), kv_len - w.q_len, w.q_len))
    return OracleCase(table, seq_lens, qsl, np.concatenate(slots), segments, width)


def oracle_pools(w: Workload, d: synth.Draw, oc: OracleCase) -> None:
    """Write history and the current chunk into NaN-poisoned float32 pools."""
    row_blocks, _ = synth.allocation(w)
    n_slots = w.pool_blocks * w.block_size
    kp = np.full((n_slots, w.num_kv_heads, w.head_dim), np.nan, dtype=np.float32)
    vp = np.full_like(kp, np.nan)
    for b in range(w.batch):
        hs = pa.slot_mapping([int(x) for x in row_blocks[b]], range(w.history_tokens), w.block_size)
        pa.kv_write(kp, hs, to_np(d.k_hist[b]))
        pa.kv_write(vp, hs, to_np(d.v_hist[b]))
    pa.kv_write(kp, oc.slots, to_np(d.k_cur))
    pa.kv_write(vp, oc.slots, to_np(d.v_cur))
    oc.k_pool, oc.v_pool, oc.q = kp, vp, to_np(d.q)


def expected(w: Workload, oc: OracleCase, sample=None, scale=None, dtype=np.float64) -> np.ndarray:
    """Oracle outputs in float64 (or the float32 twin, within 1e-5 of it, for whole layers)."""
    scale = w.head_dim ** -0.5 if scale is None else scale
    return pa.paged_attention(oc.q, oc.k_pool, oc.v_pool, oc.table, oc.qsl, oc.seq_lens, scale,
                              w.block_size, oc.segments, sample=sample, dtype=dtype)


def sample_rows(w: Workload, per_head: int, seed: int = 0) -> dict:
    """Sampled local query rows per (row, head): first and last rows, the tail tile, and random ones."""
    rng = np.random.default_rng(seed)
    out = {}
    for b in range(w.batch):
        for h in range(w.num_heads):
            fixed = {0, w.q_len - 1, max(0, w.q_len - 24), w.query_tokens - 1, min(w.q_len - 1, w.query_tokens)}
            extra = rng.choice(w.q_len, size=min(per_head, w.q_len), replace=False)
            out[(b, h)] = np.array(sorted(fixed | set(int(x) for x in extra)), dtype=np.int64)
    return out


def compare(got: np.ndarray, want: np.ndarray, dtype: str, mask=None) -> tuple[float, float]:
    """(max-abs, mean-abs) error over the compared entries; NaN anywhere in got fails."""
    if mask is not None:
        got, want = got[mask], want[mask]
    assert np.isfinite(got).all(), "non-finite output"
    err = np.abs(got.astype(np.float64) - want)
    return float(err.max()), float(err.mean())


TOL = {"f32": (1e-4, 1e-4), "bf16": (2e-2, 2e-3), "f16": (2e-2, 2e-3)}

# Queries per CTA of the CUDA-core kernel: the unit its split planner counts items in.
SIMT_ITEM_ROWS = 128


# Small workloads covering edge cases: D=64, GQA 3, ragged tails, fp16, a single query, a single key,
# causal-only masks, batch 1 with an exact 256-query tile boundary.
EDGE = [
    # D=64 bf16, GQA 3, ragged query tail, window + sink, action tokens
    dataclasses.replace(configs.GQA_ACTION, name="edge-d64", num_heads=6, num_kv_heads=2, head_dim=64,
                        chunk_tokens=200, window_chunks=2, sink_chunks=1, history_tokens=600, query_tokens=200,
                        action_len=20, spans=((408, 608),), pool_blocks=512, seed=21),
    # fp16, a single query token over a partial block
    dataclasses.replace(configs.ONE_FRAME, name="edge-f16-1tok", dtype="f16", num_heads=4, num_kv_heads=4,
                        chunk_tokens=1, window_chunks=40, sink_chunks=0, history_tokens=36, query_tokens=1,
                        pool_blocks=64, seed=22),
    # one key in total
    dataclasses.replace(configs.TINY, name="edge-one-key", chunk_tokens=1, window_chunks=1, history_tokens=0,
                        query_tokens=1, seed=23),
    # fp32, MHA, causal-only mask via a span that misses the query
    dataclasses.replace(configs.TINY, name="edge-f32-causal", history_tokens=40, query_tokens=40, chunk_tokens=40,
                        window_chunks=2, spans=((0, 8),), pool_blocks=64, seed=24),
    # bf16, batch 1, query tile boundary (exactly 256 queries)
    dataclasses.replace(configs.ONE_FRAME, name="edge-b1-256", batch=1, num_heads=2, num_kv_heads=1,
                        chunk_tokens=256, window_chunks=3, sink_chunks=0, history_tokens=512, query_tokens=256,
                        pool_blocks=128, seed=25),
    # fp32 at the CUDA-core kernel's row boundary: 64 queries per row run its 64-row CTAs, 65 its 128-row ones
    dataclasses.replace(configs.TINY, name="edge-f32-q64", chunk_tokens=64, window_chunks=2, history_tokens=64,
                        query_tokens=64, seed=26),
    dataclasses.replace(configs.TINY, name="edge-f32-q65", chunk_tokens=65, window_chunks=2, history_tokens=65,
                        query_tokens=65, seed=27),
]


# ---------------------------------------------------------------- packed heterogeneous rows


@dataclass
class OraclePacked:
    table: np.ndarray
    seq_lens: np.ndarray
    qsl: np.ndarray
    offsets: np.ndarray
    segments: list
    k_pool: np.ndarray
    v_pool: np.ndarray
    q: np.ndarray


def oracle_packed(pb, d: synth.PackedDraw) -> OraclePacked:
    """Metadata and NaN-poisoned float32 pools of a packed batch, from oracle/ only."""
    bs = pb.block_size
    width = max(-(-r.seq_len // bs) for r in pb.rows)
    table = np.zeros((len(pb.rows), width), dtype=np.int64)
    kp = np.full((pb.pool_blocks * bs, pb.num_kv_heads, pb.head_dim), np.nan, dtype=np.float32)
    vp = np.full_like(kp, np.nan)
    segments = []
    for b, r in enumerate(pb.rows):
        blocks = [int(x) for x in d.row_blocks[b]]
        table[b, : len(blocks)] = blocks
        slots = pa.slot_mapping(blocks, range(r.seq_len), bs)
        pa.kv_write(kp, slots, to_np(d.k_rows[b]))
        pa.kv_write(vp, slots, to_np(d.v_rows[b]))
        pa.validate_spans(list(r.spans), r.kv_start_pos, r.query_len, r.seq_len)
        segments.append(pa.build_segments(list(r.spans), r.kv_start_pos, r.query_len))
    seq_lens = np.array([r.seq_len for r in pb.rows], dtype=np.int64)
    qsl = np.concatenate([[0], np.cumsum([r.query_len for r in pb.rows])]).astype(np.int64)
    offsets = np.array([r.kv_start_pos for r in pb.rows], dtype=np.int64)
    return OraclePacked(table, seq_lens, qsl, offsets, segments, kp, vp, to_np(d.q))


def expected_packed(pb, op: OraclePacked, sample=None) -> np.ndarray:
    return pa.paged_attention(op.q, op.k_pool, op.v_pool, op.table, op.qsl, op.seq_lens, pb.head_dim ** -0.5,
                              pb.block_size, op.segments, sample=sample, query_offsets=op.offsets)


def sample_packed_rows(pb, per_head: int, seed: int = 0) -> dict:
    """Sampled local queries per (row, head): first, last, and random ones."""
    rng = np.random.default_rng(seed)
    out = {}
    for b, r in enumerate(pb.rows):
        for h in range(pb.num_heads):
            extra = rng.choice(r.query_len, size=min(per_head, r.query_len), replace=False)
            out[(b, h)] = np.array(sorted({0, r.query_len - 1} | set(int(x) for x in extra)), dtype=np.int64)
    return out
