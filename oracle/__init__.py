"""CPU oracle for tree-verified speculative decoding — TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct restatement of what the verification path computes,
in float64 (NumPy) with explicit per-node / per-row loops.  It exists to check the
CUDA library, never to stand in for it: only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
It shares no code, table or helper with the CUDA path and imports nothing from it.

Modules and the passages they restate
-------------------------------------
tree       PTD (Progressive Tree Drafting) §3.1 "tree construction": the observable
           prefix set pi(v) = {v} U pi(P(v)) and the position id from |pi(v)|.
attention  PTD §3.1 (each node attends only to its ancestors) and the speculative
           decoding blog, section "why target verification can be parallel"
           (one forward scores every drafted position under a causal mask).
vocab      blog, "greedy decoding" and "acceptance probability for sampling"
           (the target's argmax, p_i(y_i)).
greedy     blog, "greedy decoding, intuitive version" + "accept a prefix and start
           the next round" (accepted prefix plus one corrected token).
philox     Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3"
           (SC'11): Philox4x32-10, the counter-based generator both sides use.
sampling   blog, "acceptance probability for sampling" (alpha = min(1, p/q)) and
           "how to correct after a rejection" ((p - q)+ normalised).
selection  TAPS §4.1-§4.2 (candidate pool from per-position top-K marginals, budgeted
           prefix-closed subtree) and TreeGraft §3.1 (cumulative path score s(v)).
kvcommit   blog, "KV cache handling": keep the accepted tokens' cache entries, drop the
           rejected candidates' (the accepted root path laid out as a plain sequence).
frontier   TreeGraft §3.1 single-drafter expansion: frontier Top_W by s(v), the top-m
           tokens of each frontier node's drafter distribution attached as children.
prune      PTD §3.1 "overhead constraints": a per-parent child cap and the sliding-window
           stepping of the root when the tree gets too deep (page truncated there).

Readings taken where the pages are silent are listed in each module's docstring.
Parity status: every function is pinned by tests under ``tests/test_oracle_*.py``
against closed forms, brute force or hand-built cases.  The absolute acceptance
*rates* on synthetic data are the only quantity left unpinned (the pages print none).
"""
from . import tree, attention, vocab, greedy, philox, sampling, selection  # noqa: F401
