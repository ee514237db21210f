"""GPU: the KV write on row widths and slot patterns the workloads do not cover, bit for bit against the oracle.

The write kernel cuts rows into 2 KB chunks (128 16-byte vectors) and walks the flat list of (row, chunk)
pairs; these cases put rows of 1, 3 and 127 vectors (one partial chunk), exactly one and exactly two chunks,
and 2.5 chunks through it, with negative (skipped) slots scattered among the tokens and the slots in random
order over the pool (paged_attention.py, _paged_write_attn_impl: pool[slots] = x).
"""

import numpy as np
import pytest
import torch

from oracle import pagedattn as pa

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16).cpu().numpy() if t.dtype != torch.float32 else t.view(torch.int32).cpu().numpy()


@pytest.mark.parametrize("hkv,d,dtype", [
    (1, 8, torch.bfloat16),      # 16-byte rows: one vector
    (3, 8, torch.float16),       # 48-byte rows: three vectors
    (127, 8, torch.bfloat16),    # 127 vectors: one partial chunk
    (8, 128, torch.bfloat16),    # 2 KB rows: exactly one chunk
    (32, 64, torch.float32),     # 8 KB rows: four chunks
    (20, 128, torch.bfloat16),   # 5 KB rows: two chunks and a half
])
def test_write_rows_bit_exact(hkv, d, dtype):
    from paged_kv_cache_181_gb300 import _lib

    g = torch.Generator().manual_seed(hkv * 1000 + d)
    T, n_slots = 1337, 4096
    k = torch.randn(T, hkv, d, generator=g).to(dtype)
    v = torch.randn(T, hkv, d, generator=g).to(dtype)
    slots = torch.randperm(n_slots, generator=g)[:T].to(torch.int64)
    slots[torch.randperm(T, generator=g)[:97]] = -1  # skipped tokens
    kp = torch.full((n_slots, hkv, d), float("nan"), dtype=dtype)
    vp = torch.full_like(kp, float("nan"))
    want_k, want_v = _bits(kp).copy(), _bits(vp).copy()
    pa.kv_write(want_k, slots.numpy(), _bits(k))
    pa.kv_write(want_v, slots.numpy(), _bits(v))
    kp_d, vp_d = kp.cuda(), vp.cuda()
    _lib.paged_kv_write(k.cuda(), v.cuda(), slots.cuda(), kp_d, vp_d, flags=_lib.PKV_CHECK_BOUNDS)
    torch.cuda.synchronize()
    assert _lib.check() == 0
    assert np.array_equal(_bits(kp_d), want_k)
    assert np.array_equal(_bits(vp_d), want_v)
