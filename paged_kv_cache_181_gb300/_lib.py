"""ctypes binding of libpagedkv (argument marshalling only).

Every function here converts Python/torch arguments to the C ABI declared in
include/pagedkv.h and raises on a non-OK status with the library's message.
No step of the method runs in Python: the host metadata runs in the library's
C++ and every device step in its CUDA kernels.  When the shared library is
missing, importing this module raises -- there is no fallback.
"""

from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedkv.so")

PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA, PKV_ERR_DEVICE_CHECK, PKV_ERR_CAPACITY = range(6)
PKV_F32, PKV_BF16, PKV_F16 = 0, 1, 2
PKV_CHECK_BOUNDS = 0x1
PKV_FORCE_SIMT = 0x2
PKV_NO_SPLIT = 0x4
PKV_CONTIGUOUS_KV = 0x8
PKV_SEG_CAUSAL, PKV_SEG_FULL = 0, 1
PKV_DEVERR_SLOT, PKV_DEVERR_BLOCK, PKV_DEVERR_SEQLEN, PKV_DEVERR_QUERY, PKV_DEVERR_SEGMENT = 1, 2, 4, 8, 16
PKV_DEVERR_TIMEOUT = 32

EXPORTS = (
    "pkv_last_error", "pkv_version", "build_segments", "pkv_slot_mapping", "pkv_table_width",
    "pkv_visible_window", "pkv_block_table_row", "paged_kv_write", "paged_attn_workspace_size",
    "paged_attn_varlen", "pkv_check", "pkv_sm_count", "pkv_last_launches", "paged_attn_varlen_noalloc",
    "paged_kv_gather", "paged_kv_write_attn", "pkv_selftest_wait", "pkv_last_split_plan",
)


def PKV_SPLITS(n: int) -> int:
    return (int(n) & 0xFF) << 8


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"[pkv status {status}] {message}")
        self.status = status


class pkv_segment(C.Structure):
    _fields_ = [("q_start", C.c_int32), ("q_end", C.c_int32), ("kv_end", C.c_int32), ("mode", C.c_int32)]


def _load() -> C.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python -m paged_kv_cache_181_gb300.build` "
            "(or __graft_entry__.build()) first"
        )
    lib = C.CDLL(LIB_PATH)
    i32p, i64p, vp = C.POINTER(C.c_int32), C.POINTER(C.c_int64), C.c_void_p
    sig = {
        "pkv_last_error": (C.c_char_p, []),
        "pkv_version": (C.c_char_p, []),
        "build_segments": (C.c_int, [i32p, C.c_int, C.c_int32, C.c_int32, C.c_int32, C.POINTER(pkv_segment), C.c_int,
                                     C.POINTER(C.c_int)]),
        "pkv_slot_mapping": (C.c_int, [i32p, C.c_int64, C.c_int64, C.c_int64, C.c_int, i64p]),
        "pkv_table_width": (C.c_int64, [C.c_int64, C.c_int64, C.c_int64, C.c_int64, C.c_int]),
        "pkv_visible_window": (C.c_int, [i32p, C.c_int64, C.c_int64, C.c_int64, C.c_int64, C.c_int, i32p, C.c_int64,
                                         i64p, i64p]),
        "pkv_block_table_row": (C.c_int, [i32p, C.c_int64, C.c_int64, i32p, C.c_int64, C.c_int, C.c_int64, i32p,
                                          i64p]),
        "paged_kv_write": (C.c_int, [vp, vp, vp, C.c_int64, vp, vp, C.c_int64, C.c_int, C.c_int, C.c_int, C.c_uint32,
                                     vp]),
        "paged_kv_write_attn": (C.c_int, [vp, vp, vp, vp, C.c_int64, C.c_int, vp, vp, C.c_int64, C.c_int, C.c_int,
                                          C.c_int, C.c_int, vp, C.c_int, C.c_int, vp, vp, C.c_int, C.c_int, C.c_float,
                                          vp, vp, vp, vp, C.c_size_t, C.c_uint32, vp]),
        "pkv_selftest_wait": (C.c_int, [C.c_uint64, vp]),
        "paged_kv_gather": (C.c_int, [vp, vp, C.c_int64, vp, C.c_int, C.c_int, C.c_int, C.c_int, vp, vp, C.c_int64,
                                      C.c_int, C.c_int, C.c_int, C.c_uint32, vp]),
        "paged_attn_workspace_size": (C.c_size_t, [C.c_int64, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int]),
        "paged_attn_varlen": (C.c_int, [vp, C.c_int64, C.c_int, vp, vp, C.c_int64, C.c_int, C.c_int, C.c_int, C.c_int,
                                        vp, C.c_int, C.c_int, vp, vp, C.c_int, C.c_int, C.c_float, vp, vp, vp, vp,
                                        C.c_size_t, C.c_uint32, vp]),
        "pkv_check": (C.c_int, [vp, C.POINTER(C.c_uint32)]),
        "pkv_sm_count": (C.c_int, []),
        "pkv_last_launches": (C.c_int, []),
        "pkv_last_split_plan": (None, [C.POINTER(C.c_int), C.POINTER(C.c_int64)]),
        "paged_attn_varlen_noalloc": (C.c_int, [vp, C.c_int64, C.c_int, vp, vp, C.c_int64, C.c_int, C.c_int, C.c_int,
                                                C.c_int, vp, C.c_int, C.c_int, vp, vp, C.c_int, C.c_int, C.c_float, vp,
                                                vp, vp, C.c_uint32, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def last_error() -> str:
    return lib.pkv_last_error().decode()


def _ok(status: int) -> None:
    if status != PKV_OK:
        raise PkvError(status, last_error())


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p(arr: np.ndarray, ctype):
    return arr.ctypes.data_as(C.POINTER(ctype))


# ---------------------------------------------------------------- host metadata


def build_segments(spans, query_offset: int, query_len: int, seq_len: int) -> list[tuple[int, int, int, int]]:
    """Segments (q_start, q_end, kv_end, mode) of one row; mode 0 causal, 1 full."""
    sp = _i32(np.asarray(spans, dtype=np.int64).reshape(-1, 2)) if len(spans) else np.zeros((0, 2), np.int32)
    cap = 2 * len(spans) + 1
    out = (pkv_segment * cap)()
    n = C.c_int(0)
    _ok(lib.build_segments(_p(sp, C.c_int32), len(spans), int(query_offset), int(query_len), int(seq_len), out, cap,
                           C.byref(n)))
    return [(out[i].q_start, out[i].q_end, out[i].kv_end, out[i].mode) for i in range(n.value)]


def slot_mapping(blocks, first_position: int, n_tokens: int, block_size: int = 16) -> np.ndarray:
    b = _i32(blocks)
    out = np.empty(int(n_tokens), dtype=np.int64)
    _ok(lib.pkv_slot_mapping(_p(b, C.c_int32), b.size, int(first_position), int(n_tokens), int(block_size),
                             _p(out, C.c_int64)))
    return out


def table_width(chunk_tokens: int, sink_tokens: int, window_tokens: int, action_len: int, block_size: int = 16) -> int:
    w = lib.pkv_table_width(int(chunk_tokens), int(sink_tokens), int(window_tokens), int(action_len), int(block_size))
    if w < 0:
        raise PkvError(PKV_ERR_INVALID_ARG, last_error())
    return int(w)


def visible_window(row_blocks, end_tokens: int, sink_tokens: int, window_tokens: int, block_size: int = 16):
    """(visible block ids, video_len) of one row."""
    rb = _i32(row_blocks)
    cap = max(1, rb.size)
    out = np.empty(cap, dtype=np.int32)
    n = C.c_int64(0)
    vl = C.c_int64(0)
    _ok(lib.pkv_visible_window(_p(rb, C.c_int32), rb.size, int(end_tokens), int(sink_tokens), int(window_tokens),
                               int(block_size), _p(out, C.c_int32), cap, C.byref(n), C.byref(vl)))
    return out[: n.value].copy(), int(vl.value)


def block_table_row(video_blocks, video_len: int, action_blocks, action_len: int, width: int, block_size: int = 16):
    """(padded int32 row, kv_len)."""
    vb = _i32(video_blocks)
    ab = _i32(action_blocks) if len(action_blocks) else np.zeros(1, np.int32)
    out = np.empty(int(width), dtype=np.int32)
    kv = C.c_int64(0)
    _ok(lib.pkv_block_table_row(_p(vb, C.c_int32), vb.size, int(video_len), _p(ab, C.c_int32), int(action_len),
                                int(block_size), int(width), _p(out, C.c_int32), C.byref(kv)))
    return out, int(kv.value)


# ---------------------------------------------------------------- device ops


def _torch():
    import torch

    return torch


def dtype_code(t) -> int:
    torch = _torch()
    return {torch.float32: PKV_F32, torch.bfloat16: PKV_BF16, torch.float16: PKV_F16}[t.dtype]


def _stream(stream) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _dptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _require(fn: str, *tensors) -> None:
    """Every tensor (None skipped) contiguous and on the current CUDA device.

    The library takes raw device pointers: a host tensor's address would reach the kernels, and a
    tensor of another device would be launched on this device's stream.
    """
    torch = _torch()
    dev = None
    for t in tensors:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{fn}: tensors must be on a CUDA device (got {t.device})")
        if not t.is_contiguous():
            raise ValueError(f"{fn}: tensors must be contiguous")
        if dev is None:
            dev = t.device
            if dev.index is not None and dev.index != torch.cuda.current_device():
                raise ValueError(f"{fn}: tensors are on {dev}, the current device is cuda:{torch.cuda.current_device()}")
        elif t.device != dev:
            raise ValueError(f"{fn}: tensors must be on one device")


def _require_metadata(fn: str, *tensors) -> None:
    torch = _torch()
    for t in tensors:
        if t is not None and t.dtype != torch.int32:
            raise ValueError(f"{fn}: metadata must be int32")


def _check_attn_shapes(fn: str, q, key_pool, value_pool, block_table, query_start_loc, seq_lens, segs, seg_start,
                       out, block_size: int) -> None:
    """Shapes the C call cannot see: it takes one size per dimension (Tq/Hq/D from q, Hkv and the block
    count from key_pool, B/W from block_table), so every other tensor must agree with them, or a kernel
    would read or write past an allocation that no device-side check knows the size of."""
    if q.dim() != 3 or key_pool.dim() != 3:
        raise ValueError(f"{fn}: q must be [Tq, Hq, D] and the pools [num_blocks * {block_size}, Hkv, D]")
    if tuple(value_pool.shape) != tuple(key_pool.shape):
        raise ValueError(f"{fn}: value_pool shape {tuple(value_pool.shape)} differs from key_pool "
                         f"{tuple(key_pool.shape)}")
    if key_pool.shape[2] != q.shape[2]:
        raise ValueError(f"{fn}: the pools' head dim {key_pool.shape[2]} differs from q's {q.shape[2]}")
    if key_pool.shape[0] % block_size:
        raise ValueError(f"{fn}: the pools' {key_pool.shape[0]} slots are not a whole number of {block_size}-slot "
                         f"blocks")
    if out is not None and tuple(out.shape) != tuple(q.shape):
        raise ValueError(f"{fn}: out shape {tuple(out.shape)} differs from q {tuple(q.shape)}")
    if block_table.dim() != 2:
        raise ValueError(f"{fn}: block_table must be [B, W]")
    B = block_table.shape[0]
    if query_start_loc.numel() != B + 1 or seq_lens.numel() != B:
        raise ValueError(f"{fn}: query_start_loc must hold B+1 = {B + 1} and seq_lens B = {B} entries "
                         f"(got {query_start_loc.numel()} and {seq_lens.numel()})")
    if (segs is None) != (seg_start is None):
        raise ValueError(f"{fn}: segs and seg_start go together")
    if segs is not None:
        if segs.dim() != 2 or segs.shape[1] != 4:
            raise ValueError(f"{fn}: segs must be [n, 4] (q_start, q_end, kv_end, mode)")
        if seg_start.numel() != B + 1:
            raise ValueError(f"{fn}: seg_start must hold B+1 = {B + 1} entries (got {seg_start.numel()})")


def paged_kv_write(k, v, slot_mapping, key_pool, value_pool, *, flags: int = 0, stream=None) -> None:
    """key_pool[slot[t]] = k[t]; value_pool[slot[t]] = v[t] (pools ``[num_slots, Hkv, D]``)."""
    T, hkv, d = k.shape
    if v.shape != k.shape or key_pool.shape != value_pool.shape or key_pool.shape[1:] != k.shape[1:]:
        raise ValueError("paged_kv_write: shape mismatch")
    if slot_mapping.numel() != T:
        raise ValueError("paged_kv_write: slot_mapping must hold one slot per token")
    _require("paged_kv_write", k, v, slot_mapping, key_pool, value_pool)
    if k.dtype != key_pool.dtype or v.dtype != value_pool.dtype or k.dtype != v.dtype:
        raise ValueError("paged_kv_write: sources and pools must share one dtype")
    if slot_mapping.dtype != _torch().int64 or slot_mapping.numel() != T:
        raise ValueError("paged_kv_write: slot_mapping must be int64 [T]")
    _ok(lib.paged_kv_write(_dptr(k), _dptr(v), _dptr(slot_mapping), T, _dptr(key_pool), _dptr(value_pool),
                           key_pool.shape[0], hkv, d, dtype_code(k), flags, _stream(stream)))


def paged_kv_gather(key_pool, value_pool, block_table, stage_k, stage_v, *, first_block: int = 0,
                    n_blocks: int | None = None, flags: int = 0, block_size: int = 16, stream=None) -> None:
    """Copy table blocks [first_block, first_block + n_blocks) of every row into ``stage_k/v [B, rows, Hkv, D]``."""
    torch = _torch()
    B, W = block_table.shape
    if n_blocks is None:
        n_blocks = W - first_block
    _require("paged_kv_gather", key_pool, value_pool, block_table, stage_k, stage_v)
    if block_table.dtype != torch.int32:
        raise ValueError("paged_kv_gather: block_table must be int32")
    if stage_k.shape != stage_v.shape or stage_k.shape[0] != B or stage_k.shape[2:] != key_pool.shape[1:]:
        raise ValueError("paged_kv_gather: staging buffers must be [B, rows, Hkv, D]")
    if len({key_pool.dtype, value_pool.dtype, stage_k.dtype, stage_v.dtype}) != 1:
        raise ValueError("paged_kv_gather: pools and staging buffers must share one dtype")
    hkv, d = key_pool.shape[1:]
    _ok(lib.paged_kv_gather(_dptr(key_pool), _dptr(value_pool), key_pool.shape[0] // block_size, _dptr(block_table),
                            B, W, int(first_block), int(n_blocks), _dptr(stage_k), _dptr(stage_v), stage_k.shape[1],
                            hkv, d, dtype_code(key_pool), flags, _stream(stream)))


def workspace_size(Tq: int, Hq: int, D: int, B: int, max_query_len: int, max_seq_len: int) -> int:
    return int(lib.paged_attn_workspace_size(int(Tq), int(Hq), int(D), int(B), int(max_query_len), int(max_seq_len)))


def paged_attn_varlen(q, key_pool, value_pool, block_table, query_start_loc, seq_lens, max_query_len: int,
                      max_seq_len: int, softmax_scale: float, *, segs=None, seg_start=None, out=None,
                      workspace=None, flags: int = 0, block_size: int = 16, stream=None):
    """Paged varlen attention; pools are ``[num_blocks * 16, Hkv, D]``; returns ``out``."""
    torch = _torch()
    _check_attn_shapes("paged_attn_varlen", q, key_pool, value_pool, block_table, query_start_loc, seq_lens, segs,
                       seg_start, out, block_size)
    Tq, hq, d = q.shape
    hkv = key_pool.shape[1]
    if out is None:
        out = torch.empty_like(q)
    _require("paged_attn_varlen", q, key_pool, value_pool, block_table, query_start_loc, seq_lens, segs, seg_start,
             out, workspace)
    if key_pool.dtype != q.dtype or value_pool.dtype != q.dtype or out.dtype != q.dtype:
        raise ValueError("paged_attn_varlen: q, pools and out must share one dtype")
    _require_metadata("paged_attn_varlen", block_table, query_start_loc, seq_lens, segs, seg_start)
    B, W = block_table.shape
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _ok(lib.paged_attn_varlen(_dptr(q), Tq, hq, _dptr(key_pool), _dptr(value_pool), key_pool.shape[0] // block_size,
                              block_size, hkv, d, dtype_code(q), _dptr(block_table), B, W, _dptr(query_start_loc),
                              _dptr(seq_lens), int(max_query_len), int(max_seq_len), float(softmax_scale),
                              _dptr(segs), _dptr(seg_start), _dptr(out), _dptr(workspace), ws, flags,
                              _stream(stream)))
    return out


def paged_kv_write_attn(q, k, v, slot_mapping, key_pool, value_pool, block_table, query_start_loc, seq_lens,
                        max_query_len: int, max_seq_len: int, softmax_scale: float, *, segs=None, seg_start=None,
                        out=None, workspace=None, flags: int = 0, block_size: int = 16, stream=None):
    """paged_kv_write + paged_attn_varlen in one launch (see include/pagedkv.h); returns ``out``."""
    torch = _torch()
    _check_attn_shapes("paged_kv_write_attn", q, key_pool, value_pool, block_table, query_start_loc, seq_lens, segs,
                       seg_start, out, block_size)
    Tq, hq, d = q.shape
    hkv = key_pool.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if k.shape != (Tq, hkv, d) or v.shape != k.shape:
        raise ValueError("paged_kv_write_attn: k and v must be [Tq, Hkv, D]")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != Tq:
        raise ValueError("paged_kv_write_attn: slot_mapping must be int64 [Tq]")
    _require("paged_kv_write_attn", q, k, v, slot_mapping, key_pool, value_pool, block_table, query_start_loc, seq_lens,
             segs, seg_start, out, workspace)
    _require_metadata("paged_kv_write_attn", block_table, query_start_loc, seq_lens, segs, seg_start)
    if len({q.dtype, k.dtype, v.dtype, key_pool.dtype, value_pool.dtype, out.dtype}) != 1:
        raise ValueError("paged_kv_write_attn: q, k, v, pools and out must share one dtype")
    B, W = block_table.shape
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _ok(lib.paged_kv_write_attn(_dptr(q), _dptr(k), _dptr(v), _dptr(slot_mapping), Tq, hq, _dptr(key_pool),
                                _dptr(value_pool), key_pool.shape[0] // block_size, block_size, hkv, d, dtype_code(q),
                                _dptr(block_table), B, W, _dptr(query_start_loc), _dptr(seq_lens),
                                int(max_query_len), int(max_seq_len), float(softmax_scale), _dptr(segs),
                                _dptr(seg_start), _dptr(out), _dptr(workspace), ws, flags, _stream(stream)))
    return out


def paged_attn_varlen_noalloc(q, key_pool, value_pool, block_table, query_start_loc, seq_lens, max_query_len: int,
                              max_seq_len: int, softmax_scale: float, *, segs=None, seg_start=None, out=None,
                              flags: int = 0, block_size: int = 16, stream=None):
    """paged_attn_varlen without a workspace: split partials go to the library's fixed scratch array.

    For callers that cannot allocate device memory; see include/pagedkv.h.
    """
    torch = _torch()
    _check_attn_shapes("paged_attn_varlen_noalloc", q, key_pool, value_pool, block_table, query_start_loc, seq_lens,
                       segs, seg_start, out, block_size)
    Tq, hq, d = q.shape
    hkv = key_pool.shape[1]
    if out is None:
        out = torch.empty_like(q)
    _require("paged_attn_varlen_noalloc", q, key_pool, value_pool, block_table, query_start_loc, seq_lens, segs,
             seg_start, out)
    if key_pool.dtype != q.dtype or value_pool.dtype != q.dtype or out.dtype != q.dtype:
        raise ValueError("paged_attn_varlen_noalloc: q, pools and out must share one dtype")
    _require_metadata("paged_attn_varlen_noalloc", block_table, query_start_loc, seq_lens, segs, seg_start)
    B, W = block_table.shape
    _ok(lib.paged_attn_varlen_noalloc(_dptr(q), Tq, hq, _dptr(key_pool), _dptr(value_pool),
                                      key_pool.shape[0] // block_size, block_size, hkv, d, dtype_code(q),
                                      _dptr(block_table), B, W, _dptr(query_start_loc), _dptr(seq_lens),
                                      int(max_query_len), int(max_seq_len), float(softmax_scale), _dptr(segs),
                                      _dptr(seg_start), _dptr(out), flags, _stream(stream)))
    return out


def check(stream=None) -> int:
    """Synchronise, read and clear the device error word; returns its bits (0: clean).

    Raises PkvError only when the call itself fails (no device, a CUDA error on the stream)."""
    bits = C.c_uint32(0)
    st = lib.pkv_check(_stream(stream), C.byref(bits))
    if st not in (PKV_OK, PKV_ERR_DEVICE_CHECK):
        _ok(st)
    return int(bits.value)


def selftest_wait(limit_ns: int, stream=None) -> None:
    """Launch the bounded-wait self-test (see include/pagedkv.h); read the result with check()."""
    _ok(lib.pkv_selftest_wait(int(limit_ns), _stream(stream)))


def last_launches() -> int:
    """Kernels launched by the last device call on this thread."""
    return int(lib.pkv_last_launches())


def last_split_plan() -> tuple[int, int]:
    """(splits per split item, items run whole before them) of the last attention call on this thread."""
    s, w = C.c_int(), C.c_int64()
    lib.pkv_last_split_plan(C.byref(s), C.byref(w))
    return int(s.value), int(w.value)


def sm_count() -> int:
    return int(lib.pkv_sm_count())
