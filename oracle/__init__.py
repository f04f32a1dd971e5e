"""CPU oracle for sparse causal flash attention (SCFA). TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline / reference arm of
`bench.py` may import anything here. The product path (the C-ABI library and
its Python binding) never imports, links or executes this package, and this
package never imports the product path.

Source of every definition: the summary page "Faster Causal Attention Over
Large Sequences Through Sparse Flash Attention" (deep-paper.org, arXiv
2306.01160), sections "FlashAttention 的兴起", "动态稀疏性为何会破坏它" and
"SCFA 解决方案" (parts 1 QK-Sparse and 2 Hash-Sparse). The method is exact
attention under an irregular causal mask, so the oracle is that definition
written out plainly in float64 with an explicit mask:

  attention.py  masks, forward (O, LSE), backward (dQ, dK, dV)
  lsh.py        random-rotation argmax bucket id (exact), stable bucket sort,
                row gather / unsort
  tiles.py      per-tile min/max, live-tile test, FULL flag, CSR/CSC lists,
                work order
  pipelines.py  the QK-sparse, hash-sparse and dense problems end to end

Pins: every function is checked in `tests/test_oracle_*.py` against facts
other than itself (closed forms, brute force, library routines, invariants and
hand-worked fixtures in `tests/golden/`). No function here is parity-unpinned.
"""
