"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds random draws only -- no arithmetic of the method.

* Block allocation (one per workload, shared by every layer, as the layers of
  one forward share one block table): a CPU ``torch.Generator`` seeded
  ``seed * 1000 + 999`` draws a random permutation of blocks
  ``1 .. pool_blocks-1``; each row in turn takes ``ceil(end / bs)`` blocks for
  its video positions, then ``ceil(action_len / bs)`` scratch blocks for its
  action tokens.  Block 0 is never handed out: it is the table's padding
  entry, so a test can poison it.
* Layer data: a ``torch.Generator`` on the requested device seeded
  ``seed * 1000 + layer`` draws, in order, Q ``[B * q_len, Hq, D]``, history K
  and V ``[B, history, Hkv, D]``, and the current chunk's K and V
  ``[B * q_len, Hkv, D]`` (each row's video tokens, then its action tokens),
  all ~ N(0, sigma).

Values are drawn in float32 and rounded to the workload dtype
(round-to-nearest-even), so the oracle can upcast the exact same numbers.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

from .configs import Workload

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@dataclass
class Draw:
    workload: Workload
    layer: int
    row_blocks: list        # per row: int64 tensor, physical block of each logical video block
    action_blocks: list     # per row: int64 tensor, scratch blocks for action tokens
    q: torch.Tensor         # [B*q_len, Hq, D]
    k_hist: torch.Tensor    # [B, history, Hkv, D]
    v_hist: torch.Tensor
    k_cur: torch.Tensor     # [B*q_len, Hkv, D]
    v_cur: torch.Tensor


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def seed_of(w: Workload, layer: int) -> int:
    return w.seed * 1000 + layer


def allocation(w: Workload):
    """(row_blocks, action_blocks): per row, int64 tensors of physical block ids."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed * 1000 + 999)
    bs = w.block_size
    n_video = _ceil_div(w.end_tokens, bs)
    n_action = _ceil_div(w.action_len, bs)
    per_row = n_video + n_action
    if w.batch * per_row > w.pool_blocks - 1:
        raise ValueError(f"{w.name}: pool of {w.pool_blocks} blocks cannot hold {w.batch} rows of {per_row}")
    perm = torch.randperm(w.pool_blocks - 1, generator=g) + 1
    row_blocks, action_blocks = [], []
    for b in range(w.batch):
        base = b * per_row
        row_blocks.append(perm[base : base + n_video].clone())
        action_blocks.append(perm[base + n_video : base + per_row].clone())
    return row_blocks, action_blocks


def draw(w: Workload, layer: int = 0, device="cpu") -> Draw:
    """Draw one layer's inputs for workload ``w`` on ``device``."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed_of(w, layer))
    dt = TORCH_DTYPE[w.dtype]
    row_blocks, action_blocks = allocation(w)

    def normal(*shape):
        x = torch.randn(*shape, generator=g, device=dev, dtype=torch.float32)
        if w.sigma != 1.0:
            x.mul_(w.sigma)
        return x.to(dt)

    tq = w.batch * w.q_len
    q = normal(tq, w.num_heads, w.head_dim)
    k_hist = normal(w.batch, w.history_tokens, w.num_kv_heads, w.head_dim)
    v_hist = normal(w.batch, w.history_tokens, w.num_kv_heads, w.head_dim)
    k_cur = normal(tq, w.num_kv_heads, w.head_dim)
    v_cur = normal(tq, w.num_kv_heads, w.head_dim)
    return Draw(w, layer, row_blocks, action_blocks, q, k_hist, v_hist, k_cur, v_cur)


# ---------------------------------------------------------------- packed heterogeneous rows


@dataclass
class PackedDraw:
    batch: object            # configs.PackedBatch
    row_blocks: list         # per row: int64 tensor, physical block of each logical block
    q: torch.Tensor          # [sum query_len, Hq, D]
    k_rows: list             # per row: [seq_len, Hkv, D]
    v_rows: list


def packed_allocation(pb):
    """Per row, ``ceil(seq_len / bs)`` blocks from one permutation of blocks 1..pool_blocks-1
    (CPU generator seeded ``seed * 1000 + 999``); block 0 stays the padding entry."""
    g = torch.Generator(device="cpu")
    g.manual_seed(pb.seed * 1000 + 999)
    need = [_ceil_div(r.seq_len, pb.block_size) for r in pb.rows]
    if sum(need) > pb.pool_blocks - 1:
        raise ValueError(f"{pb.name}: pool of {pb.pool_blocks} blocks cannot hold {sum(need)} blocks")
    perm = torch.randperm(pb.pool_blocks - 1, generator=g) + 1
    out, used = [], 0
    for n in need:
        out.append(perm[used : used + n].clone())
        used += n
    return out


def packed_draw(pb, device="cpu") -> PackedDraw:
    """Q for every row's queries, then each row's K and V for all of its positions
    (generator seeded ``seed * 1000``), ~ N(0, sigma), rounded to the batch dtype."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(pb.seed * 1000)
    dt = TORCH_DTYPE[pb.dtype]

    def normal(*shape):
        x = torch.randn(*shape, generator=g, device=dev, dtype=torch.float32)
        if pb.sigma != 1.0:
            x.mul_(pb.sigma)
        return x.to(dt)

    tq = sum(r.query_len for r in pb.rows)
    q = normal(tq, pb.num_heads, pb.head_dim)
    k_rows, v_rows = [], []
    for r in pb.rows:
        k_rows.append(normal(r.seq_len, pb.num_kv_heads, pb.head_dim))
        v_rows.append(normal(r.seq_len, pb.num_kv_heads, pb.head_dim))
    return PackedDraw(pb, packed_allocation(pb), q, k_rows, v_rows)
