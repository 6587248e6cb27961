"""CPU fp64 oracle for batched attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
its Python binding) imports, calls or links anything in this package.  Only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs
of ``bench.py`` may use it.

The oracle restates what the pages define, in plain numpy, in float64:

* ``oracle.metadata`` -- slot_mapping, block table -> CSR page table
  (``kv_indptr`` / ``kv_indices`` / ``last_page_len``), token table -> page
  table, and the page-size-1 view of a pool.
* ``oracle.fp8`` -- the OCP FP8 E4M3 ("fn") codec: exact decode and a
  round-to-nearest-even, saturate-to-finite encoder.
* ``oracle.attention`` -- the KV write (a scatter through slot_mapping), the
  paged attention definition (per request: gather the pages in logical order,
  bottom-right-aligned causal mask, optional sliding window, GQA by contiguous
  head groups, softmax(q k^T * scale) v with its log-sum-exp) and the merge of
  two attention states.

Every function is pinned by ``tests/test_oracle_pins.py`` against something
other than itself: the worked examples the pages print (``tests/golden/``),
closed forms, invariants the pages state, brute force on tiny inputs and the
library routine the pages' own CPU reference uses.  No function here is
"parity unpinned".

The oracle shares no code with the CUDA path; the only module both sides use
is the seeded input generator ``workloads.py``, which holds none of the
method's arithmetic.
"""

from . import attention, fp8, metadata  # noqa: F401
