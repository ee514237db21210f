"""GB300-native chunk-wise paged self-attention over a block-paged KV pool.

The product is ``libpagedkv.so`` (C ABI in include/pagedkv.h): a slot-mapping
KV write, a varlen paged attention with a piecewise causal/full mask (tcgen05
tensor cores for bf16/f16, CUDA cores for fp32), a split-KV combine, and the
host metadata (segments, visible window, block table, slot mapping).  This
package is a thin ctypes binding over it.  The binding loads on first use of
an operation, and fails loudly when the library has not been built; the
workload shapes (``configs``) and seeded draws (``synth``) need no library.
"""

_API = (
    "PKV_BF16", "PKV_CHECK_BOUNDS", "PKV_F16", "PKV_F32", "PKV_FORCE_SIMT", "PKV_NO_SPLIT", "PKV_SEG_CAUSAL",
    "PKV_SEG_FULL", "PKV_SPLITS", "PkvError", "block_table_row", "build_segments", "check", "last_error",
    "paged_attn_varlen", "paged_kv_write", "slot_mapping", "sm_count", "table_width", "visible_window",
    "workspace_size",
)

__all__ = list(_API)


def __getattr__(name):
    if name in _API:
        from . import _lib

        return getattr(_lib, name)
    raise AttributeError(name)
