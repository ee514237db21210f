"""Host: the key-range split the library plans, read through paged_attn_workspace_size (no GPU needed).

The workspace a call may use is max(8, planned splits) x Tq x Hq x (D + 1) x 4 bytes, the planned splits
being the larger of the two kernels' plans (256-query items for the tensor-core kernel, 128-query items for
the CUDA-core one), so the planned split count shows in it.  Without a device the planner assumes GB300's 152
SMs.  The expected counts are the ones the GPU sweeps measured best for these workloads (and the rule's
boundaries): whole waves of items run unsplit and only a last, partly filled wave is split.
"""

import pytest

from paged_kv_cache_181_gb300 import _lib


def planned(tq, hq, d, b, max_q, max_kv):
    n = _lib.workspace_size(tq, hq, d, b, max_q, max_kv)
    per_split = tq * hq * (d + 1) * 4
    assert n % per_split == 0
    return n // per_split


@pytest.fixture(autouse=True)
def _no_device():
    if _lib.sm_count() > 0:
        pytest.skip("a device is present: the planner uses its SM count")


@pytest.mark.parametrize("name, sizes, splits", [
    # 560 items = 3 waves + 104: the tail splits 4 ways, below the 8-split floor of the workspace
    ("long window", (3120, 40, 128, 2, 1560, 26528), 8),
    # 768 items = 5 waves + 8: the 8 tail items split 13 ways (65 key tiles: 5 per split)
    ("mixed mask", (8192, 24, 128, 2, 4096, 8208), 13),
    # 8 items, fewer than the SMs: every item splits 16 ways
    ("few heads", (256, 8, 128, 1, 256, 26528), 16),
    # 168 items = 1 wave + 16: the tail splits 9 ways; the CUDA-core kernel's 312 items = 2 waves + 8, whose
    # tail splits 14 ways, set the workspace
    ("one frame", (3120, 12, 128, 2, 1560, 6272), 14),
])
def test_planned_splits_of_the_workloads(name, sizes, splits):
    assert planned(*sizes) == splits


def test_whole_waves_are_not_split():
    # 152 items of 256 queries over 26.5k keys: exactly one wave, nothing to balance
    assert planned(256, 152, 128, 1, 256, 26528) == 8


def test_one_item_past_a_wave_splits_it_finely():
    # 153 items: the lone tail item splits 16 ways (13 key tiles each) instead of taking a whole wave
    assert planned(256, 153, 128, 1, 256, 26528) == 16


def test_short_keys_are_not_split():
    # 3 key tiles per item: a split would hold fewer than 4 tiles
    assert planned(256, 153, 128, 1, 256, 384) == 8


def test_empty_sizes():
    assert _lib.workspace_size(0, 8, 128, 1, 1, 1) == 0
