"""Workflow-aware prefix eviction, plain Python (test infrastructure only).

KVFlow review, "Agent Step Graph and Steps-to-Execution": an agent's
steps-to-execution is the expected number of workflow steps before it runs
again.  It follows from its predecessors' values by the join's aggregation:
a synchronisation barrier (AND: the agent waits for all predecessors) takes
``max(E_1, ..., E_k) + 1``; a conditional branch (OR: any predecessor
triggers it) takes ``min(E_1, ..., E_k) + 1``.  Applied recursively it
gives every agent's value.

KVFlow review, "Workflow-aware eviction" (the priority-assignment and
eviction algorithms of figure 2(b)): every agent with value ``step`` marks
its fixed-prompt prefix node and all ancestors: ``counter[step] += 1`` and
``priority = min(priority, step)``; a node shared by several agents keeps
the smallest (it is kept while any of them runs soon).  Nodes no agent
marks (dynamic suffixes) are evicted first.  Eviction repeatedly removes the
evictable leaf with the largest priority; a parent whose last child goes
becomes a leaf and a candidate itself.

Readings where the review is silent (also stated in the C ABI):

* Base case: the caller fixes some agents' values (e.g. 0 for agents that
  run in the current step).  An agent with no fixed value and no
  predecessor never runs (value ``None``); an AND agent with a predecessor
  that never runs never runs; an OR agent runs if any predecessor does.
  A cycle that passes through no fixed agent has no value: it is rejected.
* A node referenced by an adapter leaf (an agent is reading it right now)
  is not evictable, as in the tree's LRU eviction.
* Ties between equal priorities go to the least recently used node.
* Evicting a node leaves the counts its agents put on the ancestors: the
  agent still needs the shared prefix, which keeps its priority.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

AND, OR = 0, 1


def steps_to_execution(preds: Sequence[Sequence[int]], join: Sequence[int],
                       fixed: Sequence[Optional[int]]) -> List[Optional[int]]:
    """Steps-to-execution of every agent by recursion over its predecessors.

    ``preds[i]``: predecessor agent ids of agent ``i``; ``join[i]``: AND or
    OR; ``fixed[i]``: a given value or None.  Returns None for agents that
    never run.  Raises ValueError on a cycle through unfixed agents."""
    n = len(preds)
    memo: Dict[int, Optional[int]] = {}
    on_path = set()

    def value(i: int) -> Optional[int]:
        if fixed[i] is not None:
            return fixed[i]
        if i in memo:
            return memo[i]
        if i in on_path:
            raise ValueError(f"cycle through agent {i} with no fixed value")
        on_path.add(i)
        vals = [value(p) for p in preds[i]]
        on_path.discard(i)
        if not vals:
            out = None
        elif join[i] == AND:
            out = None if any(v is None for v in vals) else max(vals) + 1
        else:
            live = [v for v in vals if v is not None]
            out = min(live) + 1 if live else None
        memo[i] = out
        return out

    return [value(i) for i in range(n)]


class PrefixTree:
    """The cache tree as a plain dictionary model: node -> parent, with the
    per-node step counters and priority of the assignment algorithm.
    ``None`` priority means no agent marked the node."""

    def __init__(self):
        self.parent: Dict[int, Optional[int]] = {0: None}
        self.pages: Dict[int, List[int]] = {0: []}
        self.counter: Dict[int, Dict[int, int]] = {0: {}}
        self.ref: Dict[int, int] = {0: 0}
        self.last_use: Dict[int, int] = {0: 0}

    def add(self, node: int, parent: int, pages: List[int], last_use: int, ref: int = 0):
        self.parent[node] = parent
        self.pages[node] = list(pages)
        self.counter[node] = {}
        self.ref[node] = ref
        self.last_use[node] = last_use

    def priority(self, node: int) -> Optional[int]:
        c = self.counter[node]
        return min(c) if c else None

    def assign(self, node: int, step: int):
        """One agent with steps-to-execution ``step`` whose fixed prompt ends
        at ``node``: mark the node and every ancestor up to the root."""
        x = node
        while x is not None and x != 0:
            self.counter[x][step] = self.counter[x].get(step, 0) + 1
            x = self.parent[x]

    def release(self, node: int, step: int):
        x = node
        while x is not None and x != 0:
            self.counter[x][step] -= 1
            if self.counter[x][step] == 0:
                del self.counter[x][step]
            x = self.parent[x]

    def children(self, node: int) -> List[int]:
        return [c for c, p in self.parent.items() if p == node]

    def evict(self, want_pages: int) -> List[int]:
        """Remove evictable leaves, largest priority first (unmarked nodes
        before every marked one, then least recently used first), until
        ``want_pages`` pages are freed or nothing is evictable.  Returns the
        freed page ids in eviction order.  Written as a plain scan over the
        current leaves at every pick."""
        freed: List[int] = []
        inf = float("inf")
        while len(freed) < want_pages:
            cands = [x for x in self.parent if x != 0 and self.ref[x] == 0 and not self.children(x)]
            if not cands:
                break

            def key(x):
                p = self.priority(x)
                return (inf if p is None else p, -self.last_use[x])

            v = max(cands, key=key)
            freed += self.pages[v]
            for d in (self.parent, self.pages, self.counter, self.ref, self.last_use):
                del d[v]
        return freed
