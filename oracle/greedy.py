"""Greedy acceptance walk (oracle).

What it restates (speculative-decoding blog, "greedy decoding, intuitive version" and
"accept a prefix and start the next round"): drafts are accepted while they equal the
target's own choice; at the first disagreement the target's token replaces the draft and
the round ends, so a round yields the accepted drafts plus one token from the target.

Tree reading: starting at the root, the walk moves to the child whose token equals the
argmax of the current node's row (siblings carry distinct tokens, so at most one child
matches); when no child matches - or the node is a leaf - the walk stops and the
bonus token is that argmax.  A chain reduces to the linear rule above.
"""
from __future__ import annotations

from .tree import children, validate


def greedy_walk(parent, tokens, argmax):
    """Returns (accepted node list excluding the root, bonus token)."""
    validate(parent)
    kids = children(parent)
    cur = 0
    accepted = []
    while True:
        want = int(argmax[cur])
        nxt = None
        for c in kids[cur]:
            if int(tokens[c]) == want:
                nxt = c
                break
        if nxt is None:
            return accepted, want
        accepted.append(nxt)
        cur = nxt
