"""Host side of packed heterogeneous rows (no GPU): the library's segments with a per-row
query offset equal the oracle's, and the shapes fit their pools."""

import numpy as np
import pytest

from oracle import pagedattn as pa
from paged_kv_cache_181_gb300 import configs, synth


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_181_gb300 import _lib

    return _lib


@pytest.mark.parametrize("pb", list(configs.PACKED.values()), ids=lambda p: p.name)
def test_library_segments_with_row_offsets_match_the_oracle(lib, pb):
    for r in pb.rows:
        got = lib.build_segments(list(r.spans), r.kv_start_pos, r.query_len, r.seq_len)
        want = [(s.q_start, s.q_end, s.kv_end, 0 if s.mode == pa.CAUSAL else 1)
                for s in pa.build_segments(list(r.spans), r.kv_start_pos, r.query_len)]
        assert got == want
        # The kernel reads a row's query offset from its first segment.
        assert got[0][0] == r.kv_start_pos


@pytest.mark.parametrize("pb", list(configs.PACKED.values()), ids=lambda p: p.name)
def test_packed_allocation_is_distinct_and_never_uses_block_zero(pb):
    blocks = np.concatenate([b.numpy() for b in synth.packed_allocation(pb)])
    assert len(set(blocks.tolist())) == blocks.size
    assert blocks.min() >= 1 and blocks.max() < pb.pool_blocks


def test_bench_pair_count_matches_the_oracle_flops():
    import bench

    pb = configs.PACKED_MIXED
    segs_host = [[(s.q_start, s.q_end, s.kv_end, 0 if s.mode == pa.CAUSAL else 1)
                  for s in pa.build_segments(list(r.spans), r.kv_start_pos, r.query_len)] for r in pb.rows]
    qsl = np.concatenate([[0], np.cumsum([r.query_len for r in pb.rows])])
    L = [r.seq_len for r in pb.rows]
    offs = [r.kv_start_pos for r in pb.rows]
    segs_oracle = [pa.build_segments(list(r.spans), r.kv_start_pos, r.query_len) for r in pb.rows]
    want = pa.attention_flops(qsl, L, segs_oracle, 1, 1, query_offsets=offs) // 4
    assert bench.pairs_from_segments(qsl, L, segs_host) == want
