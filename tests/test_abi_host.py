"""Host-side checks of the C ABI (no GPU): the library loads, exports every
symbol the header declares, rejects bad configurations, and its work-list
planner covers exactly the sharing classes the oracle derives."""
import os
import re

import numpy as np
import pytest

import oracle
import shared_base_kv_gb300 as fk
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "forkkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fk_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = declared_symbols()
    assert len(names) >= 20
    L = fk.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(fk.EXPORTS)


def test_version_and_error_string():
    assert "sm_103a" in fk.fk_version()
    cfg = fk.fk_pool_config(1, 32, 8, 96, 16, 10, 4, 16, 100, 0, 0, 10000.0, 0)
    with pytest.raises(fk.FKError) as e:
        fk.fk_pool_bytes(cfg)
    assert "head_dim" in str(e.value)


@pytest.mark.parametrize("field,value,msg", [
    ("page_size", 32, "page_size"), ("max_rank", 12, "max_rank"),
    ("n_q_heads", 30, "multiple"), ("num_pages", 0, "num_pages"),
    ("rope_base", 0.5, "rope_base")])
def test_bad_configs_are_rejected(field, value, msg):
    cfg = fk.fk_pool_config(1, 32, 8, 128, 16, 10, 4, 16, 100, 0, 0, 10000.0, 0)
    setattr(cfg, field, value)
    with pytest.raises(fk.FKError) as e:
        fk.fk_pool_bytes(cfg)
    assert msg in str(e.value)


def test_pool_bytes_accounts_for_every_region():
    cfg = fk.fk_pool_config(2, 32, 8, 128, 16, 100, 4, 16, 1000, 0, 1 << 20, 10000.0, 1)
    n = fk.fk_pool_bytes(cfg)
    page_bytes = 2 * 2 * 100 * 8 * 16 * 128 * 2               # K and V pages, 2 layers
    rc = 4 * 16 * 2 * 1024 * 2 * 2                             # 4 agents, rank 16, 2 layers
    comp = 2 * 100 * 8 * 16 * (128 + 48 + 4)
    assert n >= page_bytes + rc + comp + (1 << 20)
    assert n < (page_bytes + rc + comp + (1 << 20)) * 1.5


def test_pool_bytes_hold_the_rope_table_for_d128():
    # d = 128 pools also hold [cos, sin](t theta_i) as f16 pairs for every
    # position of the rCache capacity (rounded up to 128 tokens): 256 bytes
    # per position; d = 64 pools hold none
    def nbytes(d, max_tokens):
        return fk.fk_pool_bytes(fk.fk_pool_config(1, 8, 2, d, 16, 16, 2, 16, max_tokens, 0,
                                                  1 << 20, 10000.0, 0))
    for d in (64, 128):
        grow = nbytes(d, 4096) - nbytes(d, 4096 - 127)     # same capacity: 4096
        assert grow == 0
    # 128 more positions: the rCache arena grows by the same amount for both
    # head sizes, the table by 128 x 256 bytes for d = 128 only (regions are
    # 256-byte aligned, so the table adds exactly that)
    extra64 = nbytes(64, 4096 + 128) - nbytes(64, 4096)
    extra128 = nbytes(128, 4096 + 128) - nbytes(128, 4096)
    assert extra128 - extra64 == 128 * 256


def _plan(w, target=152):
    return fk.fk_plan_host(w.A, w.C, w.H_q, w.H_kv, w.block_table, w.seq_lens, w.ranks, target)


@pytest.mark.parametrize("name,kw", [
    ("llama8b_32k", dict(prefix=1000, A=8)),
    ("agents32_layers32", dict(prefix=200, suffix=(0, 40), A=9, n_layers=1)),
    ("qwen72b_chunk", dict(prefix=100, A=3)),
    ("compressed", dict(prefix=333, A=15)),
    ("tiny", {}),
])
def test_plan_covers_sharing_classes_exactly_once(name, kw):
    w = workloads.make_workload(name, **kw)
    items, row_agent, row_cg, pages, tile_agents = _plan(w)
    cov = oracle.coverage(w.block_table, w.seq_lens, w.P)
    classes = {(lp, ph): set(ag) for lp, ph, ag in oracle.page_classes(w.block_table, w.seq_lens, w.P)}
    G = w.H_q // w.H_kv
    for h in range(w.H_kv):
        seen = {}
        for it in items:
            if it["head"] != h:
                continue
            ags = tile_agents[it["agent_begin"]: it["agent_begin"] + it["n_agents"]]
            rows = list(zip(row_agent[it["row_begin"]: it["row_begin"] + it["n_rows"]],
                            row_cg[it["row_begin"]: it["row_begin"] + it["n_rows"]]))
            assert set(a for a, _ in rows) == set(int(a) for a in ags)
            assert it["n_rows"] <= 64 and it["n_agents"] <= 4
            assert sum(((int(w.ranks[a]) + 15) // 16) * 16 for a in ags) <= 64
            for k in range(it["n_pages"]):
                lp = it["lp_begin"] + k
                ph = int(pages[it["page_begin"] + k])
                assert set(int(a) for a in ags) <= classes[(lp, ph)]
                for a, cg in rows:
                    key = (int(a), lp, ph, int(cg))
                    seen[key] = seen.get(key, 0) + 1
        expect = {(a, lp, ph, cg) for a, lp, ph in cov for cg in range(G * w.C)}
        assert set(seen) == expect
        assert all(v == 1 for v in seen.values())


@pytest.mark.parametrize("name,kw", [
    ("llama8b_32k", dict(prefix=900, A=8)),
    ("llama8b_32k", dict(prefix=300, A=19)),                       # ragged last tile, 3 tiles
    ("agents32_layers32", dict(prefix=200, suffix=(0, 40), A=13, n_layers=1)),   # mixed ranks
])
def test_plan_slots8_covers_sharing_classes_exactly_once(name, kw):
    w = workloads.make_workload(name, **kw)
    items, row_agent, row_cg, pages, tile_agents = fk.fk_plan_host_slots8(
        w.A, w.C, w.H_q, w.H_kv, w.block_table, w.seq_lens, w.ranks, 152)
    cov = oracle.coverage(w.block_table, w.seq_lens, w.P)
    classes = {(lp, ph): set(ag) for lp, ph, ag in oracle.page_classes(w.block_table, w.seq_lens, w.P)}
    for h in range(w.H_kv):
        seen = {}
        for it in items:
            if it["head"] != h:
                continue
            slots = [int(a) for a in tile_agents[it["agent_begin"]: it["agent_begin"] + 8]]
            assert it["n_agents"] == 8 and it["n_rows"] == 32
            for half in (slots[:4], slots[4:]):
                real = [a for a in half if a >= 0]
                assert sum(((int(w.ranks[a]) + 15) // 16) * 16 for a in real) <= 64
            rows = list(zip(row_agent[it["row_begin"]: it["row_begin"] + 32],
                            row_cg[it["row_begin"]: it["row_begin"] + 32]))
            for r, (a, cg) in enumerate(rows):            # slot s owns rows 4 s .. 4 s + 3
                assert int(a) == slots[r // 4]
                if a >= 0:
                    assert int(cg) == r % 4
            for k in range(it["n_pages"]):
                lp = it["lp_begin"] + k
                ph = int(pages[it["page_begin"] + k])
                assert set(a for a in slots if a >= 0) <= classes[(lp, ph)]
                for a, cg in rows:
                    if a >= 0:
                        key = (int(a), lp, ph, int(cg))
                        seen[key] = seen.get(key, 0) + 1
        expect = {(a, lp, ph, cg) for a, lp, ph in cov for cg in range(4)}
        assert set(seen) == expect
        assert all(v == 1 for v in seen.values())


def test_plan_slots8_reads_each_shared_page_once_per_head():
    # eight agents over one prefix fill one tile: every (page, head) is in
    # exactly one item's page run
    w = workloads.make_workload("llama8b_32k", prefix=4096, A=8)
    items, *_ = fk.fk_plan_host_slots8(w.A, w.C, w.H_q, w.H_kv, w.block_table, w.seq_lens,
                                       w.ranks, 152)
    per_head = {}
    for it in items:
        per_head[it["head"]] = per_head.get(it["head"], 0) + it["n_pages"]
    assert set(per_head.values()) == {4096 // 16}
    with pytest.raises(fk.FKError):                      # only four rows per agent
        w2 = workloads.make_workload("qwen72b_chunk", prefix=64, A=2)
        fk.fk_plan_host_slots8(w2.A, w2.C, w2.H_q, w2.H_kv, w2.block_table, w2.seq_lens,
                               w2.ranks, 152)


def test_plan_balances_pieces():
    w = workloads.make_workload("llama8b_32k")
    items, *_ = _plan(w, 152)
    pages_per_head = {}
    for it in items:
        pages_per_head[it["head"]] = pages_per_head.get(it["head"], 0) + it["n_pages"]
    # every head covers all 2048 pages twice (two 4-agent row tiles)
    assert set(pages_per_head.values()) == {2 * 2048}
    assert len(items) <= 152 + 16
    # pieces are cut at whole 128-key tiles of their segment
    assert all(it["lp_begin"] % 8 == 0 for it in items)
    tiles = [(it["n_pages"] + 7) // 8 for it in items]
    assert sum(tiles) == 16 * 256


def _prefix_tiles(w):
    """Agent tiles (call-local agent indices in slot order) of the items
    that cover the shared prefix."""
    items, row_agent, row_cg, pages, tile_agents = _plan(w)
    tiles = set()
    for it in items:
        if it["lp_begin"] == 0:
            tiles.add(tuple(int(a) for a in tile_agents[it["agent_begin"]: it["agent_begin"] + it["n_agents"]]))
    return tiles


def test_plan_packs_decode_tiles_largest_rank_first():
    # eight agents over one prefix, ranks 32 16 64 16 32 64 16 16: packed
    # largest first into the first tile with room, four tiles (cutting in
    # call order would close one at every rank-64 agent: five tiles)
    w = workloads.make_workload("llama8b_32k", prefix=512, A=8)
    w.ranks = np.array([32, 16, 64, 16, 32, 64, 16, 16], dtype=np.int32)
    assert _prefix_tiles(w) == {(2,), (5,), (0, 4), (1, 3, 6, 7)}


def test_plan_balances_tile_halves():
    # one tile of ranks 32, 16, 16: the rank-32 agent takes the second half
    # (slot 2) so that both compute warpgroups hold 32 ranks
    w = workloads.make_workload("llama8b_32k", prefix=512, A=3)
    w.ranks = np.array([32, 16, 16], dtype=np.int32)
    assert _prefix_tiles(w) == {(1, 2, 0)}


def test_plan_keeps_call_order_for_equal_ranks():
    w = workloads.make_workload("llama8b_32k", prefix=512, A=8)
    w.ranks = np.full(8, 16, dtype=np.int32)
    assert _prefix_tiles(w) == {(0, 1, 2, 3), (4, 5, 6, 7)}


def test_plan_rejects_bad_tables():
    w = workloads.make_workload("tiny")
    bt = w.block_table.copy()
    bt[1, 3] = -1
    with pytest.raises(fk.FKError):
        fk.fk_plan_host(w.A, w.C, w.H_q, w.H_kv, bt, w.seq_lens, w.ranks, 16)
    seq = w.seq_lens.copy()
    seq[0] = 0
    with pytest.raises(fk.FKError):
        fk.fk_plan_host(w.A, w.C, w.H_q, w.H_kv, w.block_table, seq, w.ranks, 16)


def _chunk_plan_checks(A, C, H_q, H_kv, seq, n_ctas, seed):
    """The chunk kernel's work list against a brute-force account of what it
    must cover (integer work: exact)."""
    rng = np.random.default_rng(seed)
    P = 16
    max_pages = max((s + P - 1) // P for s in seq) + 2
    bt = np.full((A, max_pages), -1, np.int32)
    nxt = 0
    for a in range(A):
        n = (seq[a] + P - 1) // P
        bt[a, :n] = rng.permutation(1000)[:n] + nxt
        nxt += 1000
    its, cta, pages, ptr, slots = fk.fk_plan_chunk_host(A, C, H_q, H_kv, bt, np.array(seq, np.int32),
                                                        n_ctas)
    G, R = H_q // H_kv, (H_q // H_kv) * C
    nb = (R + 127) // 128
    # every (agent, head, row block) covers its logical pages exactly once, in order
    cover = {}
    for it in its:
        assert it["n_agents"] == 1 and it["lp_begin"] % 8 == 0
        assert it["row_begin"] % 128 == 0 and it["n_rows"] == min(128, R - it["row_begin"])
        key = (it["agent_begin"], it["head"], it["row_begin"] // 128)
        got = list(pages[it["page_begin"]: it["page_begin"] + it["n_pages"]])
        assert got == list(bt[it["agent_begin"], it["lp_begin"]: it["lp_begin"] + it["n_pages"]])
        cover.setdefault(key, []).append((it["lp_begin"], it["n_pages"]))
    assert len(cover) == A * H_kv * nb
    for (a, h, b), runs in cover.items():
        runs.sort()
        pos = 0
        for lp, n in runs:
            assert lp == pos
            pos += n
        assert pos == (seq[a] + P - 1) // P
    # CTAs: consecutive item ranges, each within the tile quota
    tiles = [(it["n_pages"] + 7) // 8 for it in its]
    quota = -(-sum(tiles) // n_ctas)
    assert cta[0] == 0 and cta[-1] == len(its) and len(cta) - 1 <= n_ctas
    assert all(cta[i] < cta[i + 1] for i in range(len(cta) - 1))
    for i in range(len(cta) - 1):
        assert sum(tiles[cta[i]: cta[i + 1]]) <= quota
    # partial slots: one per (item, row), distinct, and every output row
    # (a, c, hq) lists exactly the slots of the items holding it
    want = {}
    for it in its:
        for r in range(it["n_rows"]):
            ridx = it["row_begin"] + r
            row = (it["agent_begin"] * C + ridx // G) * H_q + it["head"] * G + ridx % G
            want.setdefault(row, []).append(it["partial_begin"] + r)
    assert len(ptr) == A * C * H_q + 1 and ptr[0] == 0
    for row in range(A * C * H_q):
        assert sorted(slots[ptr[row]: ptr[row + 1]]) == sorted(want[row])
    all_slots = [s for v in want.values() for s in v]
    assert len(set(all_slots)) == len(all_slots) == slots.size


def test_chunk_plan_covers_every_row_block_and_page_once():
    # Qwen-72B-like: 8 query heads x 32 chunk tokens = 256 rows, 2 row blocks
    _chunk_plan_checks(A=5, C=32, H_q=64, H_kv=8, seq=[1000, 33, 4128, 129, 2048], n_ctas=152,
                       seed=3)
    # rows not a multiple of 128 (G*C = 192) and few CTAs
    _chunk_plan_checks(A=3, C=24, H_q=64, H_kv=8, seq=[300, 24, 900], n_ctas=7, seed=4)
    # more CTAs than tiles
    _chunk_plan_checks(A=1, C=32, H_q=32, H_kv=8, seq=[40], n_ctas=152, seed=5)


def test_chunk_plan_rejects_bad_shapes():
    bt = np.zeros((1, 4), np.int32)
    with pytest.raises(fk.FKError):
        fk.fk_plan_chunk_host(1, 32, 64, 8, bt, np.array([16], np.int32), 8)    # seq < C
    with pytest.raises(fk.FKError):
        fk.fk_plan_chunk_host(1, 32, 60, 8, bt, np.array([40], np.int32), 8)    # H_q % H_kv
    bt[0, 1] = -1
    with pytest.raises(fk.FKError):
        fk.fk_plan_chunk_host(1, 32, 64, 8, bt, np.array([40], np.int32), 8)    # page missing
