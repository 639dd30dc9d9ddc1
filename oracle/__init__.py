"""Float64 CPU oracle for paged KV attention.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` call it. It shares no code with the
CUDA library (``paged_kv_attention_gb300``) and imports nothing from it.

Every function here states, plainly and slowly, the result the method reaches:
the definition of masked softmax attention over the pages a block table names,
evaluated in float64 on the exact stored values. No blocking, no splitting, no
online softmax: those are the kernels' business, and the oracle is what they
are checked against.

Parity status: every function is pinned by ``tests/test_oracle.py`` (closed
forms, invariants, a brute-force pool scan, a torch SDPA special case and a
hand-written golden fixture); no function is "parity unpinned".
"""

from . import quant  # noqa: F401
from .attention import (  # noqa: F401
    attend,
    cascade_decode,
    default_scale,
    gather_context,
    paged_attention_decode,
    paged_attention_varlen,
    reshape_and_cache,
)
