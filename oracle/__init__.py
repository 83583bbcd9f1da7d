"""Plain fp64 CPU oracle for blockwise online-softmax attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package
(`ring_attention_online_gb300`) imports this package, and this package imports
nothing from it.  Only `tests/`, `__graft_entry__.smoke()` and the CPU legs of
`bench.py` (`cpu_baseline`, `--impl reference`) may import or call it.

Modules
-------
attention  exact softmax attention (the definition), per-range partial
           triplets (m, l, O), the pairwise online-softmax merge and the final
           normalisation, jagged and split-KV decode forms.
schedule   the integer side: which KV tiles a Q tile visits (ring-order chunk
           walk, causal prune, tail), and the flattened jagged worklist.

Every function is pinned by `-m "not gpu"` tests against brute force, closed
forms, a library special case and hand-derived golden values; none is
"parity unpinned".
"""

from . import attention, schedule  # noqa: F401
