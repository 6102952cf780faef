"""Workflow-aware prefix eviction (KVFlow review, "Agent Step Graph and
Steps-to-Execution" and "Workflow-aware eviction").

The first half pins the oracle (oracle/kvflow.py) to what the review fixes:
its AND / OR aggregation examples, hand-worked trees, an independent
fixpoint iteration of the step values and a heap form of the eviction
algorithm.  The second half checks the host C++ index (fk_radix_* priority
calls and fk_workflow_steps) against the oracle on random workflows and
trees."""
import heapq

import numpy as np
import pytest

from oracle import kvflow as ok

AND, OR = ok.AND, ok.OR


# ------------------------------------------------------------ oracle pins --

def test_review_aggregation_examples():
    # an Expresser after two Executors with steps-to-execution 0 and 2:
    # waiting for both (barrier) gives max + 1, either one (branch) min + 1
    preds = [[], [], [0, 1]]
    fixed = [0, 2, None]
    assert ok.steps_to_execution(preds, [AND, AND, AND], fixed)[2] == 3
    assert ok.steps_to_execution(preds, [AND, AND, OR], fixed)[2] == 1


def test_chain_unreachable_and_cycles():
    # a -> b -> c, a runs now
    assert ok.steps_to_execution([[], [0], [1]], [AND] * 3, [0, None, None]) == [0, 1, 2]
    # d has no predecessor and no value: it never runs; so does an AND after it,
    # while an OR after it follows its other predecessor
    got = ok.steps_to_execution([[], [], [0, 1], [0, 1]], [AND, AND, AND, OR],
                                [0, None, None, None])
    assert got == [0, None, None, 1]
    with pytest.raises(ValueError):                       # cycle of unfixed agents
        ok.steps_to_execution([[1], [0]], [AND, AND], [None, None])
    # a loop planner -> worker -> planner is fine once the planner's value is given
    assert ok.steps_to_execution([[1], [0]], [AND, AND], [0, None]) == [0, 1]


def _random_dag(rng, n):
    order = rng.permutation(n)
    preds = [[] for _ in range(n)]
    for a in range(n):
        for b in range(a):
            if rng.random() < 0.3:
                preds[order[a]].append(int(order[b]))
    join = [int(rng.integers(0, 2)) for _ in range(n)]
    fixed = [int(rng.integers(0, 3)) if rng.random() < 0.25 else None for _ in range(n)]
    return preds, join, fixed


def _fixpoint(preds, join, fixed):
    """Kleene iteration from 'never': each round recomputes every agent from
    the previous round's values; on a DAG it settles within n rounds."""
    n = len(preds)
    val = [fixed[i] for i in range(n)]
    for _ in range(n + 1):
        new = []
        for i in range(n):
            if fixed[i] is not None:
                new.append(fixed[i])
                continue
            vs = [val[p] for p in preds[i]]
            if not vs:
                new.append(None)
            elif join[i] == AND:
                new.append(None if any(v is None for v in vs) else max(vs) + 1)
            else:
                live = [v for v in vs if v is not None]
                new.append(min(live) + 1 if live else None)
        val = new
    return val


def test_steps_match_an_independent_fixpoint_iteration():
    rng = np.random.default_rng(31)
    for _ in range(300):
        preds, join, fixed = _random_dag(rng, int(rng.integers(1, 12)))
        assert ok.steps_to_execution(preds, join, fixed) == _fixpoint(preds, join, fixed)


def _hand_tree():
    t = ok.PrefixTree()
    t.add(1, 0, [10, 11], last_use=1)     # A
    t.add(2, 1, [12], last_use=2)         # B under A
    t.add(3, 1, [13], last_use=3)         # C under A
    t.add(4, 0, [14], last_use=4)         # D, a dynamic suffix no agent marks
    return t


def test_hand_tree_priorities_and_eviction_order():
    t = _hand_tree()
    t.assign(2, 0)                          # an agent running now uses B
    t.assign(3, 5)                          # an agent five steps away uses C
    assert (t.priority(1), t.priority(2), t.priority(3), t.priority(4)) == (0, 0, 5, None)
    # D (unmarked) goes first although it is the most recently used, then C
    # (priority 5); A waits for B, its last child
    assert t.evict(1) == [14]
    assert t.evict(1) == [13]
    assert t.evict(10) == [12, 10, 11]
    assert t.evict(1) == []


def test_release_and_references():
    t = _hand_tree()
    t.assign(2, 0)
    t.assign(2, 3)
    t.release(2, 0)
    assert t.priority(2) == 3 and t.priority(1) == 3
    t.ref[3] = 1                            # an agent is reading C
    t.ref[1] = 1                            # (references count up the path)
    assert t.evict(10) == [14, 12]          # C and A stay
    # B's agent still needs the shared prefix: its count stays on A
    assert t.priority(1) == 3


def _random_tree(rng, n_nodes, n_assign):
    t = ok.PrefixTree()
    page = 0
    uses = rng.permutation(n_nodes) + 1          # distinct last-use times
    for x in range(1, n_nodes + 1):
        parent = int(rng.integers(0, x))
        k = int(rng.integers(1, 4))
        t.add(x, parent, list(range(page, page + k)), last_use=int(uses[x - 1]))
        page += k
    for _ in range(n_assign):
        t.assign(int(rng.integers(1, n_nodes + 1)), int(rng.integers(0, 6)))
    return t


def test_shared_node_keeps_its_smallest_priority():
    rng = np.random.default_rng(32)
    for _ in range(50):
        t = _random_tree(rng, int(rng.integers(1, 15)), int(rng.integers(0, 10)))
        for x in t.parent:
            if x == 0:
                continue
            kids = [t.priority(c) for c in t.children(x)]
            # every step counted at a child is counted at x too
            below = [p for p in kids if p is not None]
            if below:
                assert t.priority(x) is not None and t.priority(x) <= min(below)


def _heap_evict(t, want):
    """The review's eviction as a max-heap over the leaves: pop the largest
    priority, push a parent once it has become a leaf."""
    inf = float("inf")
    kids = {x: set() for x in t.parent}
    for x, p in t.parent.items():
        if p is not None:
            kids[p].add(x)

    def key(x):
        p = t.priority(x)
        return (-(inf if p is None else p), t.last_use[x])

    heap = [(key(x), x) for x in t.parent if x != 0 and not kids[x] and t.ref[x] == 0]
    heapq.heapify(heap)
    freed = []
    while len(freed) < want and heap:
        _, v = heapq.heappop(heap)
        freed += t.pages[v]
        p = t.parent[v]
        kids[p].discard(v)
        if p != 0 and not kids[p] and t.ref[p] == 0:
            heapq.heappush(heap, (key(p), p))
    return freed


def test_scan_eviction_equals_the_heap_form():
    rng = np.random.default_rng(33)
    for _ in range(100):
        seed = int(rng.integers(0, 2 ** 31))
        a = _random_tree(np.random.default_rng(seed), 12, 8)
        b = _random_tree(np.random.default_rng(seed), 12, 8)
        want = int(rng.integers(1, 30))
        assert a.evict(want) == _heap_evict(b, want)


# ---------------------------------------------- C++ index against the oracle --

import shared_base_kv_gb300 as fk  # noqa: E402

P = 4


class _Mirror:
    """The same tree in the library's index and in the oracle model.  Nodes
    are added as whole new spans under an existing prefix (no splits), and
    the model replays the index's logical clock: an insert marks the root,
    then every node on the parent's path, then the new node as used."""

    def __init__(self):
        self.r = fk.RadixIndex(P)
        self.t = ok.PrefixTree()
        self.clock = 0
        self.tokens = {0: []}
        self.path = {0: [0]}
        self.next_page = 0
        self.uid = 0

    def add(self, parent, k):
        toks = list(self.tokens[parent])
        for _ in range(k):
            self.uid += 1
            toks += [self.uid * 1000 + i for i in range(P)]
        pages = list(range(self.next_page, self.next_page + k))
        self.next_page += k
        node = self.r.insert(toks, pages)
        for x in self.path[parent]:
            self.clock += 1
            self.t.last_use[x] = self.clock
        self.clock += 1
        self.t.add(node, parent, pages, last_use=self.clock)
        self.tokens[node] = toks
        self.path[node] = self.path[parent] + [node]
        return node

    def attach(self, node, adapter):
        self.r.adapter_attach(node, adapter, 0)
        for x in self.path[node][1:]:
            self.t.ref[x] += 1

    def assign(self, node, step):
        self.r.priority_assign(node, step)
        self.t.assign(node, step)


def test_index_priorities_and_eviction_match_the_oracle():
    rng = np.random.default_rng(41)
    for trial in range(60):
        m = _Mirror()
        nodes = [0]
        for _ in range(int(rng.integers(1, 16))):
            nodes.append(m.add(int(rng.choice(nodes)), int(rng.integers(1, 4))))
        live = nodes[1:]
        for _ in range(int(rng.integers(0, 10))):
            m.assign(int(rng.choice(live)), int(rng.integers(0, 6)))
        for a in range(int(rng.integers(0, 3))):
            m.attach(int(rng.choice(live)), a)
        for x in live:
            assert m.r.node_priority(x) == m.t.priority(x), (trial, x)
        while True:
            want = int(rng.integers(1, 6))
            got = list(m.r.evict_workflow(want))
            exp = m.t.evict(want)
            assert got == exp, (trial, got, exp)
            if not exp:
                break
        assert m.r.stats()[1] == sum(len(p) for x, p in m.t.pages.items() if x != 0)
        m.r.close()


def test_release_clear_and_split_keep_the_counts():
    m = _Mirror()
    a = m.add(0, 3)
    b = m.add(a, 1)
    m.assign(b, 4)
    m.assign(b, 1)
    assert m.r.node_priority(a) == 1
    m.r.priority_release(b, 1)
    assert m.r.node_priority(a) == 4 and m.r.node_priority(b) == 4
    with pytest.raises(fk.FKError):
        m.r.priority_release(b, 1)                 # no such assignment left
    with pytest.raises(fk.FKError):
        m.r.priority_assign(b, -1)
    with pytest.raises(fk.FKError):
        m.r.priority_assign(0, 1)                  # the root carries no mark
    # a lookup that ends inside a's span splits it; the new prefix node
    # carries a's marks
    _, _, head = m.r.match(m.tokens[a][:P])
    assert head not in (0, a) and m.r.node_priority(head) == 4
    m.r.priority_clear()
    assert m.r.node_priority(b) is None and m.r.node_priority(head) is None
    m.r.close()


def test_workflow_steps_match_the_oracle():
    rng = np.random.default_rng(42)
    for _ in range(300):
        preds, join, fixed = _random_dag(rng, int(rng.integers(1, 14)))
        assert fk.workflow_steps(preds, join, fixed) == ok.steps_to_execution(preds, join, fixed)
    # loops broken by a fixed agent, and the errors
    assert fk.workflow_steps([[2], [0], [1]], [AND, OR, AND], [0, None, None]) == [0, 1, 2]
    with pytest.raises(fk.FKError):
        fk.workflow_steps([[1], [0]], [AND, AND], [None, None])
    with pytest.raises(fk.FKError):
        fk.workflow_steps([[5]], [AND], [None])                  # predecessor out of range
    with pytest.raises(fk.FKError):
        fk.workflow_steps([[]], [2], [None])                     # join type
    assert fk.workflow_steps([], [], []) == []
