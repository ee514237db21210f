"""Pins for the oracle's segment construction (piecewise_attn.py, build_segments).

The segments are checked against a direct statement of the mask that does not
go through them: a query at global position ``p`` that lies in a full span
``[a, b)`` sees keys ``j < b``; every other query sees ``j <= p`` (the module
docstring of piecewise_attn.py: a full span lets ``Q[s:e]`` see ``K[:b]``, and
causal pieces are bottom-right aligned).
"""

import itertools
import json
import os
import random

import numpy as np
import pytest

from oracle import pagedattn as pa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def direct_mask(spans, offset, qlen, seq_len):
    mask = np.zeros((qlen, seq_len), dtype=bool)
    for i in range(qlen):
        p = offset + i
        lim = p + 1
        for a, b in spans:
            if a <= p < b:
                lim = b
        mask[i, : min(lim, seq_len)] = True
    return mask


def mask_from_segments(segs, offset, qlen, seq_len):
    mask = np.zeros((qlen, seq_len), dtype=bool)
    covered = np.zeros(qlen, dtype=int)
    for s in segs:
        n = s.q_end - s.q_start
        for r in range(n):
            p = s.q_start + r
            covered[p - offset] += 1
            if s.mode == pa.FULL:
                lim = s.kv_end
            else:
                lim = s.kv_end - n + r + 1  # bottom-right: row r of n rows over kv_end keys
            mask[p - offset, : min(lim, seq_len)] = True
    assert (covered == 1).all(), "segments must cover every query exactly once"
    return mask


def all_span_sets(seq_len, max_spans):
    spans = [(a, b) for a in range(seq_len) for b in range(a + 1, seq_len + 1)]
    yield ()
    for k in range(1, max_spans + 1):
        for combo in itertools.combinations(spans, k):
            ok = all(combo[i][1] <= combo[i + 1][0] for i in range(k - 1))
            if ok:
                yield combo


@pytest.mark.parametrize("seq_len", [1, 2, 5, 8])
def test_segments_match_direct_mask_exhaustive(seq_len):
    n = 0
    for spans in all_span_sets(seq_len, 2):
        for offset in range(seq_len):
            for qlen in range(1, seq_len - offset + 1):
                segs = pa.build_segments(list(spans), offset, qlen)
                got = mask_from_segments(segs, offset, qlen, seq_len)
                want = direct_mask(spans, offset, qlen, seq_len)
                assert (got == want).all(), (spans, offset, qlen, segs)
                n += 1
    assert n > 0


def test_segments_match_direct_mask_random_three_spans():
    rng = random.Random(1234)
    for _ in range(3000):
        seq_len = rng.randint(1, 24)
        cuts = sorted(rng.sample(range(seq_len + 1), min(seq_len + 1, rng.choice([2, 4, 6]))))
        spans = [(cuts[i], cuts[i + 1]) for i in range(0, len(cuts) - 1, 2) if cuts[i] < cuts[i + 1]][:3]
        offset = rng.randint(0, seq_len - 1)
        qlen = rng.randint(1, seq_len - offset)
        segs = pa.build_segments(spans, offset, qlen)
        assert (mask_from_segments(segs, offset, qlen, seq_len) == direct_mask(spans, offset, qlen, seq_len)).all()
        # Segments are ordered and contiguous over the query range.
        assert segs[0].q_start == offset and segs[-1].q_end == offset + qlen
        for s0, s1 in zip(segs, segs[1:]):
            assert s0.q_end == s1.q_start


def test_segments_worked_examples_golden():
    with open(os.path.join(GOLDEN, "segments.json")) as f:
        cases = json.load(f)["cases"]
    assert len(cases) >= 3
    for case in cases:
        segs = pa.build_segments([tuple(s) for s in case["spans"]], case["query_offset"], case["query_len"])
        got = [[s.q_start, s.q_end, s.kv_end, s.mode] for s in segs]
        assert got == case["segments"], case["name"]


def test_no_span_is_one_causal_segment():
    assert pa.build_segments([], 3, 5) == [pa.Segment(3, 8, 8, pa.CAUSAL)]


def test_span_past_query_keeps_unclipped_kv_end():
    # A span that runs past the query's end keeps its own end as kv_end, so the
    # last queries of a local shard can attend past their own boundary.
    segs = pa.build_segments([(2, 10)], 0, 6)
    assert segs == [pa.Segment(0, 2, 2, pa.CAUSAL), pa.Segment(2, 6, 10, pa.FULL)]


@pytest.mark.parametrize(
    "spans,offset,qlen,seq_len",
    [
        ([(3, 5), (4, 6)], 0, 8, 8),  # overlapping
        ([(5, 6), (1, 2)], 0, 8, 8),  # unsorted
        ([(3, 3)], 0, 8, 8),  # empty span
        ([(3, 9)], 0, 8, 8),  # past the sequence
        ([(-1, 2)], 0, 8, 8),  # negative start
        ([], -1, 4, 8),  # negative offset
        ([], 0, 0, 8),  # empty query
        ([], 6, 4, 8),  # query past the sequence
    ],
)
def test_validate_spans_rejects(spans, offset, qlen, seq_len):
    with pytest.raises(ValueError):
        pa.validate_spans(spans, offset, qlen, seq_len)


def test_validate_spans_accepts_touching_spans():
    pa.validate_spans([(0, 2), (2, 5)], 1, 4, 5)


@pytest.mark.parametrize("seq_len", [6, 8, 10])
def test_segments_match_direct_mask_exhaustive_three_spans(seq_len):
    # Every set of exactly three ordered, non-overlapping spans (touching allowed), at every query
    # offset and length: the case the random test above only samples.
    n = 0
    for spans in all_span_sets(seq_len, 3):
        if len(spans) != 3:
            continue
        for offset in range(seq_len):
            for qlen in range(1, seq_len - offset + 1):
                segs = pa.build_segments(list(spans), offset, qlen)
                got = mask_from_segments(segs, offset, qlen, seq_len)
                want = direct_mask(spans, offset, qlen, seq_len)
                assert (got == want).all(), (spans, offset, qlen, segs)
                n += 1
    assert n > 0
