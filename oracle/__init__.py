"""Plain, slow, CPU-only oracle for the paged KV-cache decode path.

THIS PACKAGE IS TEST INFRASTRUCTURE. Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline / reference legs of ``bench.py`` may
import it. The CUDA product path never imports, calls or links anything here,
and nothing here imports the product package: the two share no code.

What it restates, in float64 (or exact integer / byte arithmetic):

* ``paged_pool``  -- the page-table simulator with prefix sharing,
  copy-on-write and release ("Notebook 10. KV cache and serving: bytes,
  pages, and ceilings", section 5 "Page pool: prefix sharing and
  copy-on-write", and the lecture-level core's private-page allocator).
  The one addition is that copy-on-write records the (old, new) block pair a
  real cache must copy.
* ``geometry``    -- K+V bytes per token, exact payload, page-waste closed
  forms and attention FLOP counts (same notebook, sections 1, 2, 3 and 6).
* ``kv_ops``      -- block copy and slot-mapped append on host arrays
  (release page "NeuralOps v1.3.4", Architectural Breakdown 1: 16-token
  physical blocks, block table, slot mapping).
* ``attention``   -- gather K/V through a block table, then max-subtracted
  softmax attention (notebook project demo, Demo 2 ``attention``), with the
  grouped-query head mapping of notebook section 3.
* ``prefix``      -- the two-phase (chunk-first over blocks shared by a group
  of sequences, then sequence-first over each suffix) decode and its
  log-sum-exp combination (paper-search page, ChunkAttention abstract;
  notebook sections 5 and 7).
* ``quant``       -- per-row symmetric low-bit quantization of K/V rows (the
  notebook's ``fake_quantize_rows`` with the scale stored as float32), the
  quantizing append and attention over the quantized cache (section 8).
* ``multiquery``  -- several causal queries per sequence against its paged
  context: speculative verification tokens or a prefill chunk (release page
  Architectural Breakdown 2; notebook section 7).

Pins that tie these functions to the pages (not to themselves) live in
``tests/test_oracle_*.py`` and ``tests/golden/``.
"""

from . import geometry, paged_pool, kv_ops, attention, prefix, multiquery, quant  # noqa: F401
