"""Workload shapes: chunk-wise paged self-attention as AR video diffusion runs it.

Only sizes live here -- no arithmetic of the method.  The geometry follows the
vllm-omni pages: 832x480 frames give (480/16)*(832/16) = 1560 tokens per frame
(``test_paged_attention.py``, ``test_the_checkpoints_own_default_resolution_can_build_a_cache``),
16-token pool blocks, CFG positive/negative branches as two batch rows, and a
DiT with 40 attention layers that share one set of per-forward metadata
(``paged_attention.py``, ``ARDiffusionPagedLayerInputs``).
"""

from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str            # "f32" | "bf16"
    batch: int            # rows = CFG branches
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    chunk_tokens: int     # tokens per chunk (the eviction unit)
    window_chunks: int    # recent window in chunks, the current chunk included
    sink_chunks: int
    history_tokens: int   # committed tokens before the current chunk
    query_tokens: int     # video tokens of the current chunk (per row)
    action_len: int       # action tokens per row, placed in scratch blocks
    pool_blocks: int      # blocks per layer pool
    sigma: float          # q/k/v ~ N(0, sigma)
    seed: int
    layers: int = 1
    spans: tuple = ()     # full-attention spans (global key coordinates), same for every row
    notes: str = ""

    @property
    def sink_tokens(self) -> int:
        return self.sink_chunks * self.chunk_tokens

    @property
    def window_tokens(self) -> int:
        return self.window_chunks * self.chunk_tokens

    @property
    def end_tokens(self) -> int:
        return self.history_tokens + self.query_tokens

    @property
    def q_len(self) -> int:
        return self.query_tokens + self.action_len


TINY = Workload(
    name="tiny-f32", dtype="f32", batch=2, num_heads=4, num_kv_heads=4, head_dim=64, block_size=16,
    chunk_tokens=16, window_chunks=2, sink_chunks=0, history_tokens=32, query_tokens=16, action_len=0,
    pool_blocks=64, sigma=1.0, seed=0,
    notes="32 history + 16-token chunk, window 2 chunks: keys = last 32 tokens",
)

ONE_FRAME = Workload(
    name="one-frame-bf16", dtype="bf16", batch=2, num_heads=12, num_kv_heads=12, head_dim=128, block_size=16,
    chunk_tokens=1560, window_chunks=3, sink_chunks=1, history_tokens=5 * 1560, query_tokens=1560, action_len=0,
    pool_blocks=4096, sigma=1.0, seed=2,
    notes="history 5 frames (7800 = 8 mod 16): chunk starts 8 slots into the history's tail block",
)

ONE_FRAME_PARTIAL = Workload(
    name="one-frame-partial-bf16", dtype="bf16", batch=2, num_heads=12, num_kv_heads=12, head_dim=128,
    block_size=16, chunk_tokens=1560, window_chunks=3, sink_chunks=1, history_tokens=4 * 1560,
    query_tokens=1560, action_len=0, pool_blocks=4096, sigma=1.0, seed=6,
    notes="history 4 frames: the window ends 8 slots into its last block",
)

GQA_ACTION = Workload(
    name="gqa-action-bf16", dtype="bf16", batch=2, num_heads=40, num_kv_heads=8, head_dim=128, block_size=16,
    chunk_tokens=3120, window_chunks=4, sink_chunks=1, history_tokens=6 * 3120, query_tokens=3120, action_len=32,
    pool_blocks=16384, sigma=0.5, seed=3, spans=((12480, 15600),),
    notes="two-frame chunk; 32 action tokens in scratch blocks, attended causally after the video span",
)

MIXED_MASK = Workload(
    name="mixed-mask-bf16", dtype="bf16", batch=2, num_heads=24, num_kv_heads=24, head_dim=128, block_size=16,
    chunk_tokens=4096, window_chunks=2, sink_chunks=0, history_tokens=4096, query_tokens=4096, action_len=0,
    pool_blocks=32768, sigma=1.0, seed=4, spans=((4096, 5120), (6144, 7168)),
    notes="query = last 4096 of 8192 keys; full spans [4096,5120) and [6144,7168), causal elsewhere",
)

LONG_WINDOW = Workload(
    name="long-window-40L-bf16", dtype="bf16", batch=2, num_heads=40, num_kv_heads=40, head_dim=128,
    block_size=16, chunk_tokens=1560, window_chunks=16, sink_chunks=1, history_tokens=16 * 1560,
    query_tokens=1560, action_len=0, pool_blocks=2 * 1700, sigma=1.0, seed=5, layers=40,
    notes="kv_len 26520 (last block half written); 1700 blocks per branch per layer pool",
)

# The long window's shapes with fp32 inputs, one layer: the CUDA-core kernel at full size.
LONG_WINDOW_F32 = Workload(
    name="long-window-f32-1L", dtype="f32", batch=2, num_heads=40, num_kv_heads=40, head_dim=128,
    block_size=16, chunk_tokens=1560, window_chunks=16, sink_chunks=1, history_tokens=16 * 1560,
    query_tokens=1560, action_len=0, pool_blocks=2 * 1700, sigma=1.0, seed=7, layers=1,
    notes="the long-window geometry in fp32 (one layer)",
)

ALL = {w.name: w for w in (TINY, ONE_FRAME, ONE_FRAME_PARTIAL, GQA_ACTION, MIXED_MASK, LONG_WINDOW)}

# Measured by the benchmark beside the workloads above (same geometry, another input dtype).
VARIANTS = {w.name: w for w in (LONG_WINDOW_F32,)}


# ---------------------------------------------------------------- packed heterogeneous rows
#
# One attention call over rows that differ in query length, key length, spans and
# query offset (paged_attention_adapter.py, DiffusionPagedAttentionRow: query_len,
# seq_len, kv_start_pos; piecewise_attn.py, build_paged_piecewise_plan: one span list
# and one query offset per packed row).  Every row's keys [0, seq_len) are written
# into its own shuffled blocks of one shared pool.


@dataclass(frozen=True)
class PackedRow:
    query_len: int
    seq_len: int
    kv_start_pos: int     # global key position of the row's first query token
    spans: tuple = ()     # full-attention spans of this row (global key coordinates)


@dataclass(frozen=True)
class PackedBatch:
    name: str
    dtype: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    pool_blocks: int
    sigma: float
    seed: int
    rows: tuple
    notes: str = ""


PACKED_SMALL = PackedBatch(
    name="packed-small-bf16", dtype="bf16", num_heads=6, num_kv_heads=2, head_dim=128, block_size=16,
    pool_blocks=256, sigma=1.0, seed=31,
    rows=(
        PackedRow(40, 40, 0, ((0, 40),)),                  # a first chunk, full inside itself
        PackedRow(200, 900, 700, ((700, 900),)),           # a later chunk, suffix
        PackedRow(130, 600, 200, ((200, 330),)),           # re-run mid-sequence: 270 keys after the query
        PackedRow(1, 333, 332, ()),                        # one query token, causal
        PackedRow(300, 300, 0, ()),                        # causal over everything
        PackedRow(264, 777, 500, ((520, 600), (650, 700))),  # causal/full/causal/full/causal, not a suffix
    ),
    notes="6 rows: suffix and mid-sequence queries, 1..300 queries, 40..900 keys, GQA 3",
)

PACKED_MIXED = PackedBatch(
    name="packed-mixed-bf16", dtype="bf16", num_heads=40, num_kv_heads=40, head_dim=128, block_size=16,
    pool_blocks=4900, sigma=1.0, seed=32,
    rows=(
        PackedRow(1560, 1560, 0, ((0, 1560),)),                  # a new video's first frame
        PackedRow(1560, 26520, 24960, ((24960, 26520),)),        # a long window (sink + 16 frames)
        PackedRow(1568, 12488, 10920, ((10920, 12480),)),        # frame + 8 action tokens (causal tail)
        PackedRow(1560, 14040, 6240, ((6240, 7800),)),           # a frame re-run mid-sequence
        PackedRow(512, 4096, 3584, ()),                          # causal-only row
        PackedRow(24, 18000, 17976, ()),                         # a short ragged tail
    ),
    notes="6 heterogeneous rows of the 832x480 model (40 heads, D=128): first frame, long window, "
          "actions, mid-sequence re-run, causal, ragged tail",
)

# Few CTAs over a long window: one branch, 8 heads, a 256-token chunk attending 26520 keys -- 8 query-tile
# pairs for 152 SMs unless the key range is split (split-KV + combine).
PACKED_FEW_HEADS = PackedBatch(
    name="few-heads-long-window-bf16", dtype="bf16", num_heads=8, num_kv_heads=8, head_dim=128, block_size=16,
    pool_blocks=1700, sigma=1.0, seed=35,
    rows=(PackedRow(256, 26520, 26264, ((26264, 26520),)),),
    notes="1 row x 8 heads x 256 queries over 26520 keys: needs split-KV to fill the GPU",
)

PACKED = {p.name: p for p in (PACKED_SMALL, PACKED_MIXED, PACKED_FEW_HEADS)}
