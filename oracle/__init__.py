"""CPU oracle for exact ring attention — TEST INFRASTRUCTURE ONLY.

This package is the plain, slow, obviously-correct statement of what the GPU
path computes.  It exists so that tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` have something independent to compare the
CUDA path against.  Nothing in the product path (the C-ABI library or its
Python binding) may import or call it, and it imports nothing from the product
package: it shares no kernels, headers, helpers, tables or constants with the
CUDA path.  Inputs are NumPy arrays; all arithmetic is float64.

Sources (web pages on ring attention; cited by title and section):
  * "Sequence Parallelism and Ring Attention Quiz" (aiunderstanding.org),
    questions 2, 3, 6, 7, 8.
  * "06 - Sequence / Context Parallelism" (inference-engineering tutorial,
    part IX), section 4 "Ring Attention - the core algorithm", section 5
    "The variants", section 10 "Hands-on exercise".
  * "Splitting the Sequence" (Parallelism plate 8 of 11, context parallelism),
    the ring/zig-zag paragraphs, "One sequence, sixteen devices", "Terms".

Modules
  attention  - full-materialised masked softmax attention (the definition).
  ring       - the ring algorithm as the tutorial states it (initialise; for
               each step attend the held block and update (out, m, l) with
               rescaling; divide by l), shard layouts, ring schedule, work
               counts, derived ring traffic and imbalance.
  merge      - combination of partial (out, m, l) states.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
against brute force, closed forms or values printed on the pages; none is
"parity unpinned".
"""

from .attention import attention_reference, attention_bruteforce  # noqa: F401
from .merge import merge_states, finalize_state  # noqa: F401
from . import ring  # noqa: F401
