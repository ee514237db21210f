"""The C ABI library on the host: it loads, exports every declared symbol, and its
host metadata functions agree bit-exactly with the oracle.  No GPU needed."""

import os
import random
import re

import numpy as np
import pytest

from oracle import pagedattn as pa
from oracle import window as ow

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_181_gb300 import build

    if not os.path.exists(build.LIB):
        build.build()
    from paged_kv_cache_181_gb300 import _lib

    return _lib


def declared_symbols():
    text = open(HEADER).read()
    return set(re.findall(r"PKV_API\s+[\w\s\*]+?\b(\w+)\s*\(", text))


def test_library_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert len(names) >= 12
    for name in names:
        assert hasattr(lib.lib, name), name
    assert set(lib.EXPORTS) == names


def test_version_and_error_strings(lib):
    assert b"pagedkv" in lib.lib.pkv_version()
    assert lib.last_error() == ""


def test_device_calls_fail_cleanly_without_gpu(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("has a GPU")
    assert lib.sm_count() == -1
    # Host-side validation happens before any CUDA call.
    import ctypes as C

    st = lib.lib.paged_attn_varlen(None, 1, 3, None, None, 1, 16, 2, 64, 1, None, 1, 1, None, None, 1, 16, 1.0,
                                   None, None, None, None, 0, 0, None)
    assert st == lib.PKV_ERR_INVALID_ARG and "multiple" in lib.last_error()
    st = lib.lib.paged_attn_varlen(None, 1, 4, None, None, 1, 32, 2, 64, 1, None, 1, 1, None, None, 1, 16, 1.0,
                                   None, None, None, None, 0, 0, None)
    assert st == lib.PKV_ERR_UNSUPPORTED and "block_size" in lib.last_error()
    st = lib.lib.paged_attn_varlen(None, 1, 4, None, None, 1, 16, 2, 96, 1, None, 1, 1, None, None, 1, 16, 1.0,
                                   None, None, None, None, 0, 0, None)
    assert st == lib.PKV_ERR_UNSUPPORTED
    st = lib.lib.paged_attn_varlen(None, 1, 4, None, None, 1, 16, 2, 64, 1, None, 1, 1, None, None, 1, 32, 1.0,
                                   None, None, None, None, 0, 0, None)
    assert st == lib.PKV_ERR_INVALID_ARG and "max_seq_len" in lib.last_error()
    st = lib.lib.paged_kv_write(None, None, None, 4, None, None, 10, 3, 3, 1, 0, None)
    assert st == lib.PKV_ERR_INVALID_ARG
    st = lib.lib.paged_kv_write(None, None, None, 0, None, None, 10, 3, 3, 1, 0, None)
    assert st == lib.PKV_OK  # T == 0 is a no-op
    assert lib.lib.paged_attn_workspace_size(100, 4, 64, 2, 50, 100) > 0
    bits = C.c_uint32(7)
    assert lib.lib.pkv_check(None, C.byref(bits)) == lib.PKV_ERR_CUDA


def _oracle_segments(spans, off, qlen):
    return [(s.q_start, s.q_end, s.kv_end, 0 if s.mode == pa.CAUSAL else 1) for s in pa.build_segments(spans, off, qlen)]


def test_build_segments_bit_exact_with_oracle(lib):
    rng = random.Random(5)
    n = 0
    for _ in range(4000):
        seq_len = rng.randint(1, 40)
        k = rng.randint(0, 4)
        cuts = sorted(rng.sample(range(seq_len + 1), min(seq_len + 1, 2 * k)))
        spans = [(cuts[i], cuts[i + 1]) for i in range(0, len(cuts) - 1, 2) if cuts[i] < cuts[i + 1]]
        off = rng.randint(0, seq_len - 1)
        qlen = rng.randint(1, seq_len - off)
        assert lib.build_segments(spans, off, qlen, seq_len) == _oracle_segments(spans, off, qlen)
        n += 1
    assert n == 4000


def test_build_segments_golden_and_errors(lib):
    assert lib.build_segments([(4096, 5120), (6144, 7168)], 4096, 4096, 8192) == [
        (4096, 5120, 5120, 1), (5120, 6144, 6144, 0), (6144, 7168, 7168, 1), (7168, 8192, 8192, 0)]
    for spans, off, qlen, L in [([(3, 5), (4, 6)], 0, 8, 8), ([(5, 6), (1, 2)], 0, 8, 8), ([(3, 3)], 0, 8, 8),
                                ([(3, 9)], 0, 8, 8), ([(-1, 2)], 0, 8, 8), ([], -1, 4, 8), ([], 0, 0, 8),
                                ([], 6, 4, 8)]:
        with pytest.raises(lib.PkvError) as e:
            lib.build_segments(spans, off, qlen, L)
        assert e.value.status == lib.PKV_ERR_INVALID_ARG
        with pytest.raises(ValueError):
            pa.validate_spans(spans, off, qlen, L)


def test_build_segments_capacity(lib):
    import ctypes as C

    out = (lib.pkv_segment * 1)()
    n = C.c_int(0)
    sp = np.array([[2, 3], [5, 6]], dtype=np.int32)
    st = lib.lib.build_segments(sp.ctypes.data_as(C.POINTER(C.c_int32)), 2, 0, 8, 8, out, 1, C.byref(n))
    assert st == lib.PKV_ERR_CAPACITY


def test_slot_mapping_bit_exact_with_oracle(lib):
    rng = np.random.default_rng(3)
    for _ in range(200):
        nb = int(rng.integers(1, 30))
        blocks = rng.permutation(1000)[:nb]
        first = int(rng.integers(0, nb * 16))
        n = int(rng.integers(0, nb * 16 - first + 1))
        got = lib.slot_mapping(blocks, first, n)
        want = pa.slot_mapping(blocks, range(first, first + n), 16)
        assert np.array_equal(got, want)
    with pytest.raises(lib.PkvError):
        lib.slot_mapping([1, 2], 20, 20)


@pytest.mark.parametrize("chunk,sink_chunks,window_chunks,action", [(1560, 9, 9, 0), (24, 1, 2, 3), (16, 0, 2, 0),
                                                                     (40, 2, 3, 17), (3120, 1, 4, 32), (1560, 1, 16, 0)])
def test_window_and_table_bit_exact_with_oracle(lib, chunk, sink_chunks, window_chunks, action):
    sink, window = sink_chunks * chunk, window_chunks * chunk
    width = lib.table_width(chunk, sink, window, action)
    assert width == ow.table_width(chunk, 16, sink, window, action)
    rng = np.random.default_rng(chunk)
    for tick in range(1, 14):
        end = tick * chunk
        nb = ow.ceil_div(end, 16)
        row = rng.permutation(100000)[:nb].astype(np.int32) + 1
        if tick % 3 == 0:  # evict a few blocks between the sink and the window
            for i in range(nb):
                if i * 16 >= sink and (i + 1) * 16 <= end - window and rng.random() < 0.5:
                    row[i] = -1
        got_blocks, got_len = lib.visible_window(row, end, sink, window)
        want_blocks, want_len = ow.visible_video_blocks(list(row), end, sink, window, 16)
        assert list(got_blocks) == want_blocks and got_len == want_len
        act = rng.permutation(1000)[: ow.ceil_div(action, 16)].astype(np.int32) + 200000
        try:
            want_row, want_kv = ow.block_table_row(want_blocks, want_len, list(act), action, 16, width)
        except ValueError:
            with pytest.raises(lib.PkvError) as e:
                lib.block_table_row(got_blocks, got_len, act, action, width)
            assert e.value.status == lib.PKV_ERR_INVALID_ARG
            continue
        got_row, got_kv = lib.block_table_row(got_blocks, got_len, act, action, width)
        assert list(got_row) == want_row and got_kv == want_kv


def test_table_errors(lib):
    with pytest.raises(lib.PkvError):
        lib.block_table_row([], 0, [], 0, 3)
    with pytest.raises(lib.PkvError) as e:
        lib.block_table_row([1, 2, 3], 48, [], 0, 2)
    assert e.value.status == lib.PKV_ERR_CAPACITY
    with pytest.raises(lib.PkvError):
        lib.table_width(0, 1, 1, 0)
    with pytest.raises(lib.PkvError):
        lib.visible_window([1], 40, 0, 40)  # too few row blocks


def test_empty_attention_calls_are_no_ops(lib):
    # Empty sizes return before any pointer is read or any CUDA call is made (also without a GPU).
    for tq, b, max_q in ((0, 1, 1), (4, 0, 1), (4, 1, 0)):
        st = lib.lib.paged_attn_varlen(None, tq, 4, None, None, 1, 16, 2, 64, 1, None, b, 1, None, None, max_q, 16,
                                       1.0, None, None, None, None, 0, 0, None)
        assert st == lib.PKV_OK, (tq, b, max_q, lib.last_error())
        assert lib.last_launches() == 0
        st = lib.lib.paged_kv_write_attn(None, None, None, None, tq, 4, None, None, 1, 16, 2, 64, 1, None, b, 1,
                                         None, None, max_q, 16, 1.0, None, None, None, None, 0, 0, None)
        assert st == lib.PKV_OK, (tq, b, max_q, lib.last_error())
        assert lib.last_launches() == 0


def test_wrappers_refuse_host_tensors(lib):
    # The library takes raw device pointers: the binding must stop a host tensor before the C call.
    import torch

    k = torch.zeros(4, 2, 64, dtype=torch.bfloat16)
    slots = torch.arange(4, dtype=torch.int64)
    pool = torch.zeros(64, 2, 64, dtype=torch.bfloat16)
    q = torch.zeros(4, 4, 64, dtype=torch.bfloat16)
    qsl = torch.tensor([0, 4], dtype=torch.int32)
    seq = torch.tensor([4], dtype=torch.int32)
    table = torch.zeros(1, 4, dtype=torch.int32)
    calls = [
        lambda: lib.paged_kv_write(k, k, slots, pool, pool),
        lambda: lib.paged_kv_gather(pool, pool, table, torch.zeros(1, 64, 2, 64, dtype=torch.bfloat16),
                                    torch.zeros(1, 64, 2, 64, dtype=torch.bfloat16)),
        lambda: lib.paged_attn_varlen(q, pool, pool, table, qsl, seq, 4, 64, 0.125),
        lambda: lib.paged_attn_varlen_noalloc(q, pool, pool, table, qsl, seq, 4, 64, 0.125),
        lambda: lib.paged_kv_write_attn(q, k, k, slots, pool, pool, table, qsl, seq, 4, 64, 0.125),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="CUDA device"):
            call()


def test_attention_wrappers_refuse_mismatched_shapes(lib):
    # The C call takes one size per dimension (D from q, Hkv and the block count from key_pool, B from the
    # table): a tensor that disagrees with them would send a kernel past its allocation, so the binding stops
    # it before the C call (and before it looks at the device).
    import torch

    bf = torch.bfloat16
    q = torch.zeros(4, 4, 64, dtype=bf)
    pool = torch.zeros(64, 2, 64, dtype=bf)
    k = torch.zeros(4, 2, 64, dtype=bf)
    slots = torch.arange(4, dtype=torch.int64)
    qsl = torch.tensor([0, 4], dtype=torch.int32)
    seq = torch.tensor([4], dtype=torch.int32)
    table = torch.zeros(1, 4, dtype=torch.int32)
    segs = torch.zeros(1, 4, dtype=torch.int32)
    seg_start = torch.tensor([0, 1], dtype=torch.int32)
    good = dict(q=q, kp=pool, vp=pool, table=table, qsl=qsl, seq=seq, segs=segs, seg_start=seg_start, out=None)
    bad = [
        ("value_pool shape", dict(vp=torch.zeros(48, 2, 64, dtype=bf))),
        ("head dim", dict(kp=torch.zeros(64, 2, 128, dtype=bf), vp=torch.zeros(64, 2, 128, dtype=bf))),
        ("whole number", dict(kp=torch.zeros(60, 2, 64, dtype=bf), vp=torch.zeros(60, 2, 64, dtype=bf))),
        ("out shape", dict(out=torch.zeros(3, 4, 64, dtype=bf))),
        ("B\\+1", dict(qsl=torch.tensor([0, 2, 4], dtype=torch.int32))),
        ("B\\+1", dict(seq=torch.tensor([4, 4], dtype=torch.int32))),
        ("seg_start", dict(seg_start=torch.tensor([0, 1, 1], dtype=torch.int32))),
        ("segs must be", dict(segs=torch.zeros(4, dtype=torch.int32))),
        ("go together", dict(seg_start=None)),
        ("q must be", dict(q=torch.zeros(4, 256, dtype=bf))),
    ]
    for what, change in bad:
        a = good | change
        calls = [
            lambda: lib.paged_attn_varlen(a["q"], a["kp"], a["vp"], a["table"], a["qsl"], a["seq"], 4, 64, 0.125,
                                          segs=a["segs"], seg_start=a["seg_start"], out=a["out"]),
            lambda: lib.paged_attn_varlen_noalloc(a["q"], a["kp"], a["vp"], a["table"], a["qsl"], a["seq"], 4, 64,
                                                  0.125, segs=a["segs"], seg_start=a["seg_start"], out=a["out"]),
            lambda: lib.paged_kv_write_attn(a["q"], k, k, slots, a["kp"], a["vp"], a["table"], a["qsl"], a["seq"], 4,
                                            64, 0.125, segs=a["segs"], seg_start=a["seg_start"], out=a["out"]),
        ]
        for call in calls:
            with pytest.raises(ValueError, match=what):
                call()
    # The same call with consistent shapes gets as far as the device check.
    with pytest.raises(ValueError, match="CUDA device"):
        lib.paged_attn_varlen(q, pool, pool, table, qsl, seq, 4, 64, 0.125, segs=segs, seg_start=seg_start)
    with pytest.raises(ValueError, match="one slot per token"):
        lib.paged_kv_write(k, k, torch.arange(3, dtype=torch.int64), pool, pool)
