"""The library's per-forward host metadata for every workload equals the oracle's, bit for bit."""

import dataclasses

import numpy as np
import pytest

from paged_kv_cache_181_gb300 import configs, synth

from . import cases

SMOKE = dataclasses.replace(
    configs.GQA_ACTION, name="smoke-gqa-bf16", num_heads=10, num_kv_heads=2, chunk_tokens=160, window_chunks=2,
    sink_chunks=1, history_tokens=480, query_tokens=160, action_len=16, spans=((320, 480),), pool_blocks=256)


@pytest.mark.parametrize("w", list(configs.ALL.values()) + cases.EDGE + [SMOKE], ids=lambda w: w.name)
def test_metadata_matches_oracle(w):
    from paged_kv_cache_181_gb300 import build

    import os

    if not os.path.exists(build.LIB):
        build.build()
    from paged_kv_cache_181_gb300 import workload
    from oracle import pagedattn as pa

    rb, ab = synth.allocation(w)
    meta = workload.build_metadata(w, rb, ab)
    oc = cases.oracle_metadata(w)
    assert meta.width == oc.width
    assert np.array_equal(meta.table, oc.table)
    assert np.array_equal(meta.seq_lens, oc.seq_lens)
    assert np.array_equal(meta.query_start_loc, oc.qsl)
    assert np.array_equal(meta.slots, oc.slots)
    assert len(np.unique(meta.slots)) == meta.slots.size  # distinct write targets
    for b in range(w.batch):
        want = pa.slot_mapping([int(x) for x in rb[b]], range(w.history_tokens), w.block_size)
        assert np.array_equal(meta.history_slots[b], want)
    if oc.segments is None:
        assert meta.segments is None
    else:
        want = [[(s.q_start, s.q_end, s.kv_end, 0 if s.mode == "causal" else 1) for s in row] for row in oc.segments]
        assert meta.segments == want
    assert meta.max_seq_len >= int(meta.seq_lens.max())
    # block 0 (padding) is never handed out, so poisoning it is safe
    for b in range(w.batch):
        n = -(-int(meta.seq_lens[b]) // w.block_size)
        assert 0 not in set(meta.table[b, :n].tolist())


@pytest.mark.parametrize("w", list(configs.ALL.values()), ids=lambda w: w.name)
def test_bench_flop_count_matches_oracle(w):
    # The bench's algorithmic FLOPs (4 * D * Hq * visible pairs, from the library's segments) equal the
    # oracle's count over its own metadata: the roofline's numerator does not rest on the bench's arithmetic.
    import os
    import sys

    from paged_kv_cache_181_gb300 import build

    if not os.path.exists(build.LIB):
        build.build()
    from oracle import pagedattn as pa
    from paged_kv_cache_181_gb300 import workload

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    rb, ab = synth.allocation(w)
    meta = workload.build_metadata(w, rb, ab)
    oc = cases.oracle_metadata(w)
    want = pa.attention_flops(oc.qsl, oc.seq_lens, oc.segments, w.num_heads, w.head_dim)
    assert 4 * w.head_dim * w.num_heads * bench.visible_pairs(meta) == want
