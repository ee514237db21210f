"""Plain CPU oracle for chunk-wise paged self-attention over a block-paged KV pool.

TEST INFRASTRUCTURE ONLY. Nothing in the product path (the CUDA library and its
Python binding) imports, links or executes anything under this directory.  Only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` use it.

The oracle is written from the text of the vllm-omni pages and shares no code
with the CUDA path:

* ``oracle.pagedattn`` -- the slot-mapping KV write, ``build_segments``, the
  block-table gather and dense masked softmax attention in float64 (with a
  float32 twin used only for timing), piecewise over causal/full segments.
* ``oracle.window``    -- the sink + recent visible-window block selection,
  the fixed table width and the padded block-table row.

Every function says which page and which function on it it follows.  Parity
pins (tests/test_oracle_*.py) tie each function to something other than itself:
brute force, closed forms, a library attention routine, and worked values from
the pages' own tests.
"""

from . import pagedattn, window  # noqa: F401
