"""One attention call over packed heterogeneous rows, assembled through the C ABI.

Rows differ in query length, key length, spans and query offset
(``paged_attention_adapter.py``, ``DiffusionPagedAttentionRow``;
``piecewise_attn.py``, ``build_paged_piecewise_plan``).  Every row's keys are
written into its own blocks of one shared pool with the library's slot mapping
and write kernel; the segments come from the library's ``build_segments`` with
each row's own query offset, which is how the kernel learns where the row's
queries sit.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import _lib, synth
from .configs import PackedBatch


@dataclass
class PackedCase:
    pb: PackedBatch
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    q: torch.Tensor
    out: torch.Tensor
    block_table: torch.Tensor
    query_start_loc: torch.Tensor
    seq_lens: torch.Tensor
    segs: torch.Tensor
    seg_start: torch.Tensor
    segments: list            # host copy: per row, (q_start, q_end, kv_end, mode)
    qsl_host: np.ndarray
    seq_lens_host: np.ndarray
    width: int
    max_query_len: int
    workspace: torch.Tensor | None
    scale: float
    draw: synth.PackedDraw | None = None

    def attend(self, flags: int = 0, stream=None) -> torch.Tensor:
        return _lib.paged_attn_varlen(
            self.q, self.k_pool, self.v_pool, self.block_table, self.query_start_loc, self.seq_lens,
            self.max_query_len, self.width * self.pb.block_size, self.scale, segs=self.segs,
            seg_start=self.seg_start, out=self.out, workspace=self.workspace, flags=flags, stream=stream)


def build_packed(pb: PackedBatch, device="cuda", poison: bool = True, keep_draw: bool = False) -> PackedCase:
    dev = torch.device(device)
    bs = pb.block_size
    d = synth.packed_draw(pb, "cpu")
    dt = synth.TORCH_DTYPE[pb.dtype]
    n_rows = len(pb.rows)
    width = max(-(-r.seq_len // bs) for r in pb.rows)
    table = np.zeros((n_rows, width), dtype=np.int32)
    seq_lens = np.array([r.seq_len for r in pb.rows], dtype=np.int32)
    qsl = np.concatenate([[0], np.cumsum([r.query_len for r in pb.rows])]).astype(np.int32)
    k_pool = torch.empty((pb.pool_blocks * bs, pb.num_kv_heads, pb.head_dim), dtype=dt, device=dev)
    v_pool = torch.empty_like(k_pool)
    if poison:
        k_pool.fill_(float("nan"))
        v_pool.fill_(float("nan"))
    segments, flat, starts = [], [], [0]
    for b, r in enumerate(pb.rows):
        blocks = d.row_blocks[b].numpy().astype(np.int32)
        table[b, : blocks.size] = blocks
        slots = torch.from_numpy(_lib.slot_mapping(blocks, 0, r.seq_len, bs)).to(dev)
        _lib.paged_kv_write(d.k_rows[b].to(dev), d.v_rows[b].to(dev), slots, k_pool, v_pool)
        row = _lib.build_segments(list(r.spans), r.kv_start_pos, r.query_len, r.seq_len)
        segments.append(row)
        flat += row
        starts.append(len(flat))
    segs = torch.from_numpy(np.asarray(flat, dtype=np.int32).reshape(-1, 4)).to(dev)
    seg_start = torch.from_numpy(np.asarray(starts, dtype=np.int32)).to(dev)
    q = d.q.to(dev)
    max_q = int(max(r.query_len for r in pb.rows))
    nbytes = _lib.workspace_size(int(qsl[-1]), pb.num_heads, pb.head_dim, n_rows, max_q, width * bs)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev) if nbytes else None
    torch.cuda.synchronize(dev)
    return PackedCase(pb, k_pool, v_pool, q, torch.empty_like(q), torch.from_numpy(table).to(dev),
                      torch.from_numpy(qsl).to(dev), torch.from_numpy(seq_lens).to(dev), segs, seg_start, segments,
                      qsl, seq_lens, width, max_q, ws, pb.head_dim ** -0.5, d if keep_draw else None)
