"""Assemble one forward of a workload on the GPU through the library's C ABI.

This is what a caller of the library does once per forward and per layer:

* host metadata, once per forward (``paged_attention.py``, ``prepare`` /
  ``build_block_table``): visible window -> padded block-table rows and
  ``seq_lens``; ``query_start_loc``; slot mapping of the current chunk (video
  tokens after the history, action tokens in their scratch blocks); segments
  from the full-attention spans.  All of it is computed by the library's host
  functions and copied to the device once, through pinned memory;
* per layer (``_paged_write_attn_impl``): write the chunk's K/V into the
  layer's pools, then attend through the block table.

The history of every layer is written into its pools at set-up time with the
same write kernel, as earlier forwards would have written it.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from . import _lib, synth
from .configs import Workload


@dataclass
class Metadata:
    """Per-forward metadata shared by every layer."""

    width: int
    table: np.ndarray          # [B, W] int32 (host)
    seq_lens: np.ndarray       # [B] int32
    query_start_loc: np.ndarray  # [B+1] int32
    slots: np.ndarray          # [Tq] int64: current chunk (video then action per row)
    history_slots: list        # per row: int64 slots of positions [0, history)
    segments: list | None      # per row: list of (q_start, q_end, kv_end, mode), or None (no mask)
    max_query_len: int
    max_seq_len: int


def build_metadata(w: Workload, row_blocks, action_blocks) -> Metadata:
    bs = w.block_size
    width = _lib.table_width(w.chunk_tokens, w.sink_tokens, w.window_tokens, w.action_len, bs)
    table = np.zeros((w.batch, width), dtype=np.int32)
    seq_lens = np.zeros(w.batch, dtype=np.int32)
    qsl = np.zeros(w.batch + 1, dtype=np.int32)
    slots, hist_slots, segments = [], [], ([] if w.spans else None)
    for b in range(w.batch):
        rb = row_blocks[b].numpy().astype(np.int32)
        ab = action_blocks[b].numpy().astype(np.int32)
        vis, video_len = _lib.visible_window(rb, w.end_tokens, w.sink_tokens, w.window_tokens, bs)
        row, kv_len = _lib.block_table_row(vis, video_len, ab, w.action_len, width, bs)
        table[b] = row
        seq_lens[b] = kv_len
        qsl[b + 1] = qsl[b] + w.q_len
        slots.append(_lib.slot_mapping(rb, w.history_tokens, w.query_tokens, bs))
        if w.action_len:
            slots.append(_lib.slot_mapping(ab, 0, w.action_len, bs))
        hist_slots.append(_lib.slot_mapping(rb, 0, w.history_tokens, bs))
        if segments is not None:
            segments.append(_lib.build_segments(list(w.spans), kv_len - w.q_len, w.q_len, kv_len))
    return Metadata(width, table, seq_lens, qsl, np.concatenate(slots), hist_slots, segments, w.q_len, width * bs)


def _pinned_to(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory().to(device, non_blocking=True)


@dataclass
class Staging:
    k: torch.Tensor            # [B, W*16, Hkv, D]
    v: torch.Tensor
    table: torch.Tensor        # [B, W] int32, consecutive blocks of the staged rows
    first_block: int           # first table entry a probe of the same chunk must re-gather
    used_blocks: int           # table entries covering the longest row


@dataclass
class Case:
    w: Workload
    meta: Metadata
    layers: int
    k_pools: list
    v_pools: list
    q: list
    k_new: list
    v_new: list
    out: list
    slots: torch.Tensor
    block_table: torch.Tensor
    query_start_loc: torch.Tensor
    seq_lens: torch.Tensor
    segs: torch.Tensor | None
    seg_start: torch.Tensor | None
    workspace: torch.Tensor | None
    scale: float
    draws: list = field(default_factory=list)  # host copies of the layers' draws (when kept)

    def write(self, layer: int, flags: int = 0, stream=None) -> None:
        _lib.paged_kv_write(self.k_new[layer], self.v_new[layer], self.slots, self.k_pools[layer],
                            self.v_pools[layer], flags=flags, stream=stream)

    def attend(self, layer: int, flags: int = 0, stream=None) -> torch.Tensor:
        return _lib.paged_attn_varlen(
            self.q[layer], self.k_pools[layer], self.v_pools[layer], self.block_table, self.query_start_loc,
            self.seq_lens, self.meta.max_query_len, self.meta.max_seq_len, self.scale, segs=self.segs,
            seg_start=self.seg_start, out=self.out[layer], workspace=self.workspace, flags=flags, stream=stream)

    # ------------------------------------------------------------ contiguous K/V (staged window)

    def make_staging(self) -> "Staging":
        """Caller-owned contiguous buffers for one layer's visible window (``paged_attention.py``, the
        history staging pairs): ``[B, W*16, Hkv, D]`` for K and V, and the table that reads them as
        consecutive blocks (row ``b`` entry ``i`` = ``b*W + i``)."""
        w, W = self.w, self.meta.width
        dev = self.k_pools[0].device
        shape = (w.batch, W * w.block_size, w.num_kv_heads, w.head_dim)
        sk = torch.empty(shape, dtype=self.k_pools[0].dtype, device=dev)
        sv = torch.empty_like(sk)
        table = (torch.arange(w.batch, dtype=torch.int32, device=dev)[:, None] * W
                 + torch.arange(W, dtype=torch.int32, device=dev)[None, :]).contiguous()
        # Every block the current chunk's write can touch starts at the block of the first query
        # token's kv position; the blocks before it hold history only.
        first = int(min((int(L) - self.meta.max_query_len) // w.block_size for L in self.meta.seq_lens))
        used = int(-(-int(self.meta.seq_lens.max()) // w.block_size))
        return Staging(sk, sv, table, max(0, first), used)

    def stage(self, layer: int, st: "Staging", reuse_history: bool = False, flags: int = 0, stream=None) -> None:
        """Gather the layer's visible blocks into ``st``; with ``reuse_history`` only from the chunk's first block."""
        first = st.first_block if reuse_history else 0
        _lib.paged_kv_gather(self.k_pools[layer], self.v_pools[layer], self.block_table, st.k, st.v,
                             first_block=first, n_blocks=st.used_blocks - first, flags=flags, stream=stream)

    def attend_contiguous(self, layer: int, st: "Staging", flags: int = 0, stream=None) -> torch.Tensor:
        """The same attention on the staged contiguous K/V (one TMA box per key tile)."""
        w = self.w
        kf = st.k.view(-1, w.num_kv_heads, w.head_dim)
        vf = st.v.view(-1, w.num_kv_heads, w.head_dim)
        return _lib.paged_attn_varlen(
            self.q[layer], kf, vf, st.table, self.query_start_loc, self.seq_lens, self.meta.max_query_len,
            self.meta.max_seq_len, self.scale, segs=self.segs, seg_start=self.seg_start, out=self.out[layer],
            workspace=self.workspace, flags=flags | _lib.PKV_CONTIGUOUS_KV, stream=stream)

    def write_attend(self, layer: int, flags: int = 0, stream=None) -> torch.Tensor:
        """The layer's write and attention in one launch (attention reads the chunk from k/v)."""
        return _lib.paged_kv_write_attn(
            self.q[layer], self.k_new[layer], self.v_new[layer], self.slots, self.k_pools[layer], self.v_pools[layer],
            self.block_table, self.query_start_loc, self.seq_lens, self.meta.max_query_len, self.meta.max_seq_len,
            self.scale, segs=self.segs, seg_start=self.seg_start, out=self.out[layer], workspace=self.workspace,
            flags=flags, stream=stream)

    def step(self, flags: int = 0, stream=None, fused: bool = False) -> None:
        """One forward: for every layer, write the chunk's K/V, then attend (``fused``: one launch)."""
        for layer in range(self.layers):
            if fused:
                self.write_attend(layer, flags, stream)
            else:
                self.write(layer, flags, stream)
                self.attend(layer, flags, stream)


def build_case(w: Workload, device="cuda", layers: int | None = None, poison: bool = False,
               keep_draws: bool = False, data_device=None, workspace: bool = True) -> Case:
    """Allocate pools, draw inputs, write every layer's history; metadata on the device.

    ``poison`` fills the pools with NaN first, so a read of any slot that was
    never written turns the output NaN.  ``data_device`` is where the random
    draws are made (default: the CPU for single-layer cases, else ``device``).
    """
    dev = torch.device(device)
    n_layers = w.layers if layers is None else layers
    if data_device is None:
        data_device = "cpu" if n_layers == 1 else dev
    row_blocks, action_blocks = synth.allocation(w)
    meta = build_metadata(w, row_blocks, action_blocks)
    dt = synth.TORCH_DTYPE[w.dtype]
    n_slots = w.pool_blocks * w.block_size
    slots = _pinned_to(meta.slots, dev)
    table = _pinned_to(meta.table, dev)
    qsl = _pinned_to(meta.query_start_loc, dev)
    seq_lens = _pinned_to(meta.seq_lens, dev)
    segs = seg_start = None
    if meta.segments is not None:
        flat = [s for row in meta.segments for s in row]
        starts = np.concatenate([[0], np.cumsum([len(r) for r in meta.segments])]).astype(np.int32)
        segs = _pinned_to(np.asarray(flat, dtype=np.int32).reshape(-1, 4), dev)
        seg_start = _pinned_to(starts, dev)
    hist_slots = [_pinned_to(s, dev) for s in meta.history_slots]
    k_pools, v_pools, qs, ks, vs, outs, draws = [], [], [], [], [], [], []
    for layer in range(n_layers):
        d = synth.draw(w, layer, device=data_device)
        kp = torch.empty((n_slots, w.num_kv_heads, w.head_dim), dtype=dt, device=dev)
        vp = torch.empty_like(kp)
        if poison:
            kp.fill_(float("nan"))
            vp.fill_(float("nan"))
        for b in range(w.batch):
            if w.history_tokens:
                _lib.paged_kv_write(d.k_hist[b].to(dev), d.v_hist[b].to(dev), hist_slots[b], kp, vp)
        k_pools.append(kp)
        v_pools.append(vp)
        qs.append(d.q.to(dev))
        ks.append(d.k_cur.to(dev))
        vs.append(d.v_cur.to(dev))
        outs.append(torch.empty_like(qs[-1]))
        if keep_draws:
            draws.append(d)
        del d
    ws = None
    if workspace:
        tq = w.batch * w.q_len
        nbytes = _lib.workspace_size(tq, w.num_heads, w.head_dim, w.batch, meta.max_query_len, meta.max_seq_len)
        if nbytes:
            ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize(dev)
    return Case(w, meta, n_layers, k_pools, v_pools, qs, ks, vs, outs, slots, table, qsl, seq_lens, segs, seg_start,
                ws, w.head_dim ** -0.5, draws)
