"""Two-tier prefix index (ForkKV guide, "DualRadixTree", "Two-Tier Lookup
Mechanics", "Reference Counting and Eviction") checked on the host against a
plain dictionary model: every cached page is the entry prefix-tuple -> page
id, a prompt matches the longest run of cached page prefixes, and eviction
removes only prefixes no adapter depends on."""
import numpy as np
import pytest

import shared_base_kv_gb300 as fk

P = 4


def toks(*pages, tail=()):
    out = []
    for pg in pages:
        out += [pg * 100 + i for i in range(P)]
    return out + list(tail)


def test_empty_index_matches_nothing():
    r = fk.RadixIndex(P)
    m, pages, node = r.match(toks(1, 2))
    assert m == 0 and pages.size == 0 and node == 0
    assert r.stats() == (0, 0)


def test_insert_then_match_longest_whole_page_prefix():
    r = fk.RadixIndex(P)
    n = r.insert(toks(1, 2, 3), [10, 11, 12])
    m, pages, node = r.match(toks(1, 2, 3, 4))
    assert m == 3 and list(pages) == [10, 11, 12] and node == n
    m, pages, _ = r.match(toks(1, 2))
    assert m == 2 and list(pages) == [10, 11]
    m, pages, _ = r.match(toks(1, 9))            # diverges in the second page
    assert m == 1 and list(pages) == [10]
    # a token differing inside a page breaks the match at that page
    t = toks(1, 2, 3)
    t[P + 1] += 1
    assert r.match(t)[0] == 1


def test_partial_trailing_page_is_not_indexed():
    r = fk.RadixIndex(P)
    r.insert(toks(1, 2, tail=(7, 7)), [10, 11])
    assert r.stats() == (1, 2)
    assert r.match(toks(1, 2, tail=(7, 7)))[0] == 2
    with pytest.raises(fk.FKError):               # pages must cover exactly the uncached part
        r.insert(toks(1, 2, 3), [12, 13])


def test_branching_prefixes_share_their_common_pages():
    r = fk.RadixIndex(P)
    a = r.insert(toks(1, 2, 3, 4), [10, 11, 12, 13])
    assert r.match(toks(1, 2, 5))[0] == 2
    b = r.insert(toks(1, 2, 5), [20])
    m, pages, node = r.match(toks(1, 2, 5))
    assert (m, list(pages), node) == (3, [10, 11, 20], b)
    m, pages, node = r.match(toks(1, 2, 3, 4))
    assert (m, list(pages), node) == (4, [10, 11, 12, 13], a)   # handles survive a split
    assert r.stats()[1] == 5


def test_two_tier_cases_and_reference_counts():
    r = fk.RadixIndex(P)
    doc = toks(1, 2, 3)
    # case C: full miss; both tiers are filled
    m, _, node = r.match(doc)
    assert m == 0
    node = r.insert(doc, [10, 11, 12])
    r.adapter_attach(node, adapter=7, owner=0)
    # case A: full hit for adapter 7; case B: base only for adapter 8
    m, _, node2 = r.match(doc)
    assert m == 3 and node2 == node
    assert r.adapter_get(node, 7) == 0
    assert r.adapter_get(node, 8) == -1
    r.adapter_attach(node, adapter=8, owner=1)
    assert r.node_ref(node) == 2
    # a shorter prefix node created by a split counts the leaves below it
    _, _, head = r.match(toks(1))
    assert r.node_ref(head) == 2
    with pytest.raises(fk.FKError):
        r.adapter_attach(node, adapter=8, owner=2)
    assert r.adapter_detach(node, 7) == 0
    assert r.node_ref(node) == 1 and r.node_ref(head) == 1


def test_eviction_skips_referenced_prefixes_and_goes_lru_first():
    r = fk.RadixIndex(P)
    x = r.insert(toks(1, 2), [10, 11])
    y = r.insert(toks(3, 4), [20, 21])
    z = r.insert(toks(5), [30])
    r.adapter_attach(z, 1, 5)                     # z is in use
    r.match(toks(1, 2))                           # x used after y
    freed = r.evict(1)
    assert list(freed) == [20, 21]                # y: least recently used, unreferenced
    assert r.match(toks(3, 4))[0] == 0
    freed = r.evict(10)
    assert list(freed) == [10, 11]                # z stays: an adapter depends on it
    assert r.match(toks(5))[0] == 1
    r.adapter_detach(z, 1)
    assert list(r.evict(10)) == [30]
    assert r.stats() == (0, 0)


def test_eviction_frees_children_before_parents():
    r = fk.RadixIndex(P)
    r.insert(toks(1, 2), [10, 11])
    r.insert(toks(1, 2, 3), [12])
    r.insert(toks(1, 2, 4), [13])
    r.match(toks(1, 2, 3))
    freed = r.evict(1)
    assert list(freed) == [13]                    # a leaf; the shared [1, 2] waits for its children
    assert list(r.evict(1)) == [12]
    assert list(r.evict(1)) == [10, 11]


def test_random_operations_against_a_dictionary_model():
    rng = np.random.default_rng(11)
    r = fk.RadixIndex(P)
    model = {}          # tuple(prefix tokens) -> page id
    attached = []       # (node, adapter, prefix tuple)
    next_page = 0

    def model_match(t):
        m = 0
        while (m + 1) * P <= len(t) and tuple(t[:(m + 1) * P]) in model:
            m += 1
        return m

    for step in range(400):
        # prompts over a small page alphabet so that prefixes collide often
        n_pages = int(rng.integers(1, 7))
        t = toks(*[int(v) for v in rng.integers(0, 3, n_pages)], tail=(1,) * int(rng.integers(0, P)))
        op = rng.random()
        m, pages, node = r.match(t)
        assert m == model_match(t), step
        assert list(pages) == [model[tuple(t[:(k + 1) * P])] for k in range(m)]
        if op < 0.5:
            new = list(range(next_page, next_page + n_pages - m))
            next_page += len(new)
            node = r.insert(t, new)
            for k in range(m, n_pages):
                model[tuple(t[:(k + 1) * P])] = new[k - m]
            if rng.random() < 0.3:
                a = int(rng.integers(0, 4))
                if r.adapter_get(node, a) < 0:
                    r.adapter_attach(node, a, step)
                    attached.append((node, a, tuple(t[:n_pages * P])))
        elif op < 0.65 and attached:
            node, a, _ = attached.pop(int(rng.integers(0, len(attached))))
            r.adapter_detach(node, a)
        else:
            freed = set(int(v) for v in r.evict(int(rng.integers(1, 4))))
            gone = [k for k, v in model.items() if v in freed]
            for k in gone:
                del model[k]
            # no page an adapter depends on was evicted, and what remains
            # is prefix-closed
            for _, _, pre in attached:
                for k in range(1, len(pre) // P + 1):
                    assert pre[:k * P] in model
            for k in model:
                for j in range(1, len(k) // P):
                    assert k[:j * P] in model
        assert r.stats()[1] == len(model)


def test_bad_arguments_are_rejected():
    r = fk.RadixIndex(P)
    with pytest.raises(fk.FKError):
        r.adapter_get(12345, 1)
    with pytest.raises(fk.FKError):
        r.adapter_attach(0, 1, 1)                # the empty prefix carries no adapter
    node = r.insert(toks(1), [1])
    with pytest.raises(fk.FKError):
        r.adapter_detach(node, 3)
    with pytest.raises(fk.FKError):
        fk.RadixIndex(0)


def test_eviction_scales_to_many_prefixes():
    # 20,000 cached prefixes under 100 shared heads, then everything evicted:
    # the heap over the current leaves keeps this well under a second
    import time
    r = fk.RadixIndex(P)
    page = 0
    for h in range(100):
        r.insert(toks(10000 + h), [page])
        page += 1
        for j in range(199):
            r.insert(toks(10000 + h, 20000 + j), [page])
            page += 1
    assert r.stats() == (20000, 20000)
    t0 = time.perf_counter()
    freed = r.evict(10 ** 6, cap=10 ** 6)
    dt = time.perf_counter() - t0
    assert sorted(freed) == list(range(20000)) and r.stats() == (0, 0)
    assert dt < 2.0, dt
