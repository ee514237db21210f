"""CUDA-graph capture of a forward (fixed shapes, new contents each replay).

Every device call of the library is asynchronous on the caller's stream, allocates nothing and
never synchronises, so a whole forward -- every layer's fused write + attention, or the two-call
form, with or without split-KV -- can be captured once and replayed.  A replay must give the same
bits as the eager calls, also after the inputs' contents change in place.
"""

import pytest
import torch

from paged_kv_cache_181_gb300 import configs

pytestmark = pytest.mark.gpu


def _capture(case, fused, flags):
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):  # warm-up outside the capture (first-call attribute setup)
        case.step(fused=fused, flags=flags)
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        case.step(fused=fused, flags=flags)
    return graph


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "two-call"])
@pytest.mark.parametrize("splits", [0, 2])
def test_graph_replay_matches_eager(fused, splits):
    from paged_kv_cache_181_gb300 import _lib, workload

    w = configs.GQA_ACTION
    case = workload.build_case(w, layers=2, poison=True)
    flags = _lib.PKV_SPLITS(splits) if splits else 0
    case.step(fused=fused, flags=flags)
    torch.cuda.synchronize()
    eager = [o.clone() for o in case.out]
    graph = _capture(case, fused, flags)
    for o in case.out:
        o.zero_()
    graph.replay()
    torch.cuda.synchronize()
    for got, want in zip(case.out, eager):
        assert torch.equal(got, want)
    # New contents in the same buffers: the replay follows them.
    for q in case.q:
        q.mul_(0.5)
    graph.replay()
    torch.cuda.synchronize()
    replayed = [o.clone() for o in case.out]
    case.step(fused=fused, flags=flags)
    torch.cuda.synchronize()
    for got, want in zip(replayed, case.out):
        assert torch.equal(got, want)
    assert not any(torch.equal(a, b) for a, b in zip(replayed, eager))
    assert _lib.check() == 0
