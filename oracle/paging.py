"""Sharing classes of a paged base cache (test oracle, integer work).

Agents that were forked from one prefix name the same physical pages,
read-only, until one of them writes (ForkKV guide, "The Copy-on-Write
Paradigm"); the base tier of the index hands out those shared block pointers
(ForkKV guide, "Two-Tier Lookup Mechanics", item 1).  A kernel that streams
each shared page once for all of its readers needs, per logical page index,
the groups of agents that name the same physical page there.
"""
from __future__ import annotations

from typing import List, Set, Tuple

import numpy as np


def page_classes(block_table, seq_lens, P: int) -> List[Tuple[int, int, Tuple[int, ...]]]:
    """Sorted ``(logical_page, physical_page, agents)`` for every page some
    agent reads; ``agents`` is the sorted tuple of agents naming that page at
    that logical index."""
    bt = np.asarray(block_table)
    groups = {}
    for a, T in enumerate(np.asarray(seq_lens)):
        for lp in range((int(T) + P - 1) // P):
            groups.setdefault((lp, int(bt[a, lp])), []).append(a)
    return sorted((lp, ph, tuple(sorted(ag))) for (lp, ph), ag in groups.items())


def coverage(block_table, seq_lens, P: int) -> Set[Tuple[int, int, int]]:
    """Every ``(agent, logical_page, physical_page)`` a kernel must read."""
    bt = np.asarray(block_table)
    out = set()
    for a, T in enumerate(np.asarray(seq_lens)):
        for lp in range((int(T) + P - 1) // P):
            out.add((a, lp, int(bt[a, lp])))
    return out
