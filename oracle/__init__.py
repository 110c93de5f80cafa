"""CPU oracle for the Grok-1 grouped-query attention core. TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct NumPy restatement of what the pages define:
RoPE on Q and K, the KV-cache append (``rope``), soft-capped, masked GQA
attention in fp64 for prefill and decode (``attention``), and the Q/K/V
projections in front of them (``projection``), and the continuous-batching
slot insertion (``slots``). It shares no code with
the CUDA library: neither imports the other. Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may use it; the
library's own code path must never call it.

Every function cites the passage of the code-reading guide it follows; the
readings taken where the pages are silent are listed in the module headers.
Parity with the original JAX implementation's bits is unpinned (the pages
print no output values); each piece is pinned instead by closed forms,
invariants, special cases and brute force in ``tests/test_oracle_*.py``.
"""
from . import attention, bf16, projection, rope, slots  # noqa: F401
