"""Pool bookkeeping and byte-exact data movement through the C ABI: base and
residual appends, copy-on-write forks, reference counts, error paths, and
the GPU encoder of the compressed pool against the oracle's codes."""
import numpy as np
import pytest
import torch

import oracle
import shared_base_kv_gb300 as fk
import workloads
from _gpu_util import as_u16, decode_base, decode_lk, decode_lv, pool_u16
from shared_base_kv_gb300 import harness

pytestmark = pytest.mark.gpu

L, HQ, H, D = 2, 8, 2, 128


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _pool(num_pages=12, compressed=False, agents=4, max_rank=64, max_tokens=200):
    return fk.Pool(n_layers=L, n_q_heads=HQ, n_kv_heads=H, head_dim=D, num_pages=num_pages,
                   max_agents=agents, max_rank=max_rank, max_tokens=max_tokens,
                   compressed=compressed)


def _bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(torch.bfloat16).cuda()


def _read_tokens(pool, layer, row, T):
    """[T, H, D] bf16 bits of keys and values read back through a row."""
    ku, vu = pool_u16(pool, fk.FK_REGION_KB), pool_u16(pool, fk.FK_REGION_VB)
    NP = pool.cfg.num_pages
    k = np.zeros((T, H, D), np.uint16)
    v = np.zeros((T, H, D), np.uint16)
    for t in range(T):
        for h in range(H):
            page, r = row[t // 16], t % 16
            k[t, h] = decode_base(ku, L, NP, H, D, layer, page, h, False)[r]
            v[t, h] = decode_base(vu, L, NP, H, D, layer, page, h, True)[r]
    return k, v


def test_base_append_round_trip_and_zero_fill():
    pool = _pool()
    row = np.full(8, -1, np.int32)
    kb, vb = _bf16((45, H, D), 1), _bf16((45, H, D), 2)
    for lo, hi in ((0, 7), (7, 16), (16, 40), (40, 45)):       # chunks crossing pages
        fk.fk_base_append(pool.h, 1, row, lo, kb[lo:hi].contiguous(), vb[lo:hi].contiguous())
    torch.cuda.synchronize()
    assert (row[:3] >= 0).all() and (row[3:] == -1).all()
    k, v = _read_tokens(pool, 1, row, 48)
    assert np.array_equal(k[:45], as_u16(kb)) and np.array_equal(v[:45], as_u16(vb))
    assert not k[45:].any() and not v[45:].any()            # rest of the last page zeroed
    k0, _ = _read_tokens(pool, 0, row, 45)                  # layer 0 untouched
    assert not k0.any()
    assert [fk.fk_page_refcount(pool.h, int(p)) for p in row[:3]] == [1, 1, 1]


def test_fork_shares_pages_and_copy_on_write():
    pool = _pool()
    parent = np.full(4, -1, np.int32)
    kb, vb = _bf16((20, H, D), 3), _bf16((20, H, D), 4)
    for layer in range(L):
        fk.fk_base_append(pool.h, layer, parent, 0, kb, vb)
    child = fk.fk_fork(pool.h, parent)
    assert np.array_equal(child, parent)
    assert fk.fk_page_refcount(pool.h, int(parent[0])) == 2
    assert fk.fk_page_refcount(pool.h, int(parent[1])) == 2
    kc, vc = _bf16((5, H, D), 5), _bf16((5, H, D), 6)
    for layer in range(L):
        fk.fk_base_append(pool.h, layer, child, 20, kc, vc)
    torch.cuda.synchronize()
    assert child[0] == parent[0]                     # full shared page untouched
    assert child[1] != parent[1]                     # partial page copied on write
    assert fk.fk_page_refcount(pool.h, int(parent[0])) == 2
    assert fk.fk_page_refcount(pool.h, int(parent[1])) == 1
    assert fk.fk_page_refcount(pool.h, int(child[1])) == 1
    for layer in range(L):
        kp, vp = _read_tokens(pool, layer, parent, 20)
        assert np.array_equal(kp, as_u16(kb)) and np.array_equal(vp, as_u16(vb))
        kk, vv = _read_tokens(pool, layer, child, 25)
        assert np.array_equal(kk[:20], as_u16(kb)) and np.array_equal(kk[20:], as_u16(kc))
        assert np.array_equal(vv[:20], as_u16(vb)) and np.array_equal(vv[20:], as_u16(vc))


def test_page_errors_leave_state_unchanged():
    pool = _pool(num_pages=4)
    ids = fk.fk_pages_alloc(pool.h, 3)
    with pytest.raises(fk.FKError) as e:
        fk.fk_pages_alloc(pool.h, 2)
    assert e.value.code == fk.FK_ERR_OUT_OF_PAGES
    last = fk.fk_pages_alloc(pool.h, 1)
    fk.fk_pages_release(pool.h, ids)
    with pytest.raises(fk.FKError) as e:
        fk.fk_pages_release(pool.h, [int(ids[0]), int(last[0]), int(last[0])])
    assert e.value.code == fk.FK_ERR_INVALID_ARG
    assert fk.fk_page_refcount(pool.h, int(last[0])) == 1       # nothing released
    with pytest.raises(fk.FKError):
        fk.fk_pages_release(pool.h, [99])
    row = np.full(2, -1, np.int32)
    fk.fk_pages_release(pool.h, last)
    kb = _bf16((40, H, D), 7)
    with pytest.raises(fk.FKError):                              # past max_pages
        fk.fk_base_append(pool.h, 0, row, 0, kb, kb)


def test_residual_append_round_trip():
    pool = _pool()
    for agent, r in ((0, 8), (1, 16), (2, 40), (3, 64)):
        Bk, Bv = _bf16((L, r, H * D), 10 + r), _bf16((L, r, H * D), 20 + r)
        fk.fk_agent_register(pool.h, agent, r, 2.0, Bk, Bv)
        lk, lv = _bf16((130, r), 30 + r), _bf16((130, r), 40 + r)
        fk.fk_residual_append(pool.h, 1, agent, 0, lk[:77].contiguous(), lv[:77].contiguous())
        fk.fk_residual_append(pool.h, 1, agent, 77, lk[77:].contiguous(), lv[77:].contiguous())
        torch.cuda.synchronize()
        off, layer_bytes, rp = fk.fk_agent_rcache(pool.h, agent)
        assert rp == (r + 15) // 16 * 16
        mem = pool.mem.cpu().numpy()
        base = off + 1 * layer_bytes
        got_k = decode_lk(mem[base: base + layer_bytes // 2], rp, 136)
        got_v = decode_lv(mem[base + layer_bytes // 2: base + layer_bytes], rp, 136)
        assert np.array_equal(got_k[:130, :r], as_u16(lk))
        assert np.array_equal(got_v[:130, :r], as_u16(lv))
        assert not got_k[:, r:].any() and not got_v[:, r:].any()   # rank padding is zero
        assert not got_k[130:].any()                               # never-appended rows


def test_agent_errors():
    pool = _pool(agents=2, max_rank=16)
    B = _bf16((L, 16, H * D), 1)
    fk.fk_agent_register(pool.h, 0, 16, 1.0, B, B)
    with pytest.raises(fk.FKError):
        fk.fk_agent_register(pool.h, 0, 16, 1.0, B, B)           # id taken
    with pytest.raises(fk.FKError):
        fk.fk_agent_register(pool.h, 1, 12, 1.0, B, B)           # not a multiple of 8
    with pytest.raises(fk.FKError):
        fk.fk_residual_append(pool.h, 0, 1, 0, B[0], B[0])       # unregistered agent
    with pytest.raises(fk.FKError):
        fk.fk_residual_append(pool.h, 0, 0, 190, _bf16((20, 16), 2), _bf16((20, 16), 3))
    fk.fk_agent_release(pool.h, 0)
    fk.fk_agent_register(pool.h, 0, 16, 1.0, B, B)


def test_attention_argument_errors():
    w = workloads.make_workload("tiny")
    dw = harness.DeviceWorkload(w)
    q = dw.queries(0)
    out = torch.empty_like(q)
    ag = np.arange(w.A, dtype=np.int32)
    bad = dw.block_table.copy()
    bad[0, 0] = 10 ** 6
    with pytest.raises(fk.FKError):
        fk.fk_residual_attention(dw.pool.h, 0, q, ag, bad, w.seq_lens, False, False, out)
    with pytest.raises(fk.FKError):
        fk.fk_residual_attention(dw.pool.h, 0, q, np.array([0, 0, 1, 2], np.int32),
                                 dw.block_table, w.seq_lens, False, False, out)
    with pytest.raises(fk.FKError):                      # no compressed copy
        fk.fk_residual_attention(dw.pool.h, 0, q, ag, dw.block_table, w.seq_lens, False, True, out)
    with pytest.raises(fk.FKError):                      # layer out of range
        fk.fk_residual_attention(dw.pool.h, 1, q, ag, dw.block_table, w.seq_lens, False, False, out)
    dw.check()


def _near_tie_ok(codes_gpu, codes_ref, z_ref):
    """Codes may differ only where fp64 z sits within 1e-4 of a boundary,
    and then only to the adjacent level."""
    diff = codes_gpu != codes_ref
    if not diff.any():
        return True, 0
    b = oracle.LLOYD_MAX_BOUNDARIES
    dist = np.min(np.abs(z_ref[..., None] - b), axis=-1)
    ok = (dist[diff] < 1e-4).all() and (np.abs(codes_gpu[diff].astype(int) - codes_ref[diff]) == 1).all()
    return bool(ok), int(diff.sum())


def test_gpu_encoder_matches_oracle_codes():
    w = workloads.make_workload("compressed", prefix=333, A=3)
    dw = harness.DeviceWorkload(w, compressed="gpu")
    ld = w.layer(0)
    kq_ref, ks_ref, vc_ref, vn_ref = oracle.encode_pages(ld.pages_k, ld.pages_v, w.slot_fill)
    pool = dw.pool
    NP = pool.cfg.num_pages
    kq = pool.region(fk.FK_REGION_KQ).cpu().numpy().view(np.int8).reshape(1, NP, w.H_kv, 16, w.d)
    vc = pool.region(fk.FK_REGION_VC).cpu().numpy().reshape(1, NP, w.H_kv, 16, 3 * w.d // 8)
    vn = pool.region(fk.FK_REGION_VN).cpu().numpy().view(np.float32).reshape(1, NP, w.H_kv, 16)
    ks = pool.region(fk.FK_REGION_KS).cpu().numpy().view(np.float32)[0]
    assert ks == ks_ref                                   # fp32 max|K| / 127, same rounding
    pk = ld.pages_k.to(torch.float64).numpy()
    pv = ld.pages_v.to(torch.float64).numpy()
    n_ties = 0
    for slot in range(w.n_slots):
        page = int(dw.slot_page[slot])
        fill = int(w.slot_fill[slot])
        gk = kq[0, page].transpose(1, 0, 2)[:fill]         # [rows, H, d]
        rk = kq_ref[slot, :fill]
        dk = gk != rk
        if dk.any():   # only where K/scale sits on a .5 tie in fp32
            x = pk[slot, :fill][dk] / float(ks_ref)
            assert (np.abs(np.abs(x - np.floor(x)) - 0.5) < 1e-5).all()
        codes_g = oracle.unpack_planes(vc[0, page].transpose(1, 0, 2)[:fill], w.d)
        v = pv[slot, :fill]
        z = oracle.fwht(v) / np.linalg.norm(v, axis=-1, keepdims=True)
        ok, nt = _near_tie_ok(codes_g, vc_ref[slot, :fill], z)
        assert ok
        n_ties += nt
        assert np.allclose(vn[0, page].T[:fill], vn_ref[slot, :fill], rtol=2e-6)
    print("near-tie code differences:", n_ties)


def test_load_compressed_round_trip():
    pool = _pool(compressed=True)
    ids = fk.fk_pages_alloc(pool.h, 3)
    rng = np.random.default_rng(0)
    kq = rng.integers(-127, 128, size=(3, 16, H, D), dtype=np.int8)
    vcp = rng.integers(0, 256, size=(3, 16, H, 3 * D // 8), dtype=np.uint8)
    vn = rng.random((3, 16, H), dtype=np.float32)
    fk.fk_pool_load_compressed(pool.h, 1, ids, torch.from_numpy(kq).cuda(),
                               torch.from_numpy(vcp).cuda(), torch.from_numpy(vn).cuda(), 0.25)
    torch.cuda.synchronize()
    NP = pool.cfg.num_pages
    gkq = pool.region(fk.FK_REGION_KQ).cpu().numpy().view(np.int8).reshape(L, NP, H, 16, D)
    gvc = pool.region(fk.FK_REGION_VC).cpu().numpy().reshape(L, NP, H, 16, 3 * D // 8)
    gvn = pool.region(fk.FK_REGION_VN).cpu().numpy().view(np.float32).reshape(L, NP, H, 16)
    for i, page in enumerate(ids):
        assert np.array_equal(gkq[1, page].transpose(1, 0, 2), kq[i])
        assert np.array_equal(gvc[1, page].transpose(1, 0, 2), vcp[i])
        assert np.array_equal(gvn[1, page].T, vn[i])
    assert pool.region(fk.FK_REGION_KS).cpu().numpy().view(np.float32)[1] == 0.25


def test_prefix_index_drives_page_references():
    """The two-tier index owns one reference per cached page; agents fork
    their own.  Evicting a prefix returns its ids for release, and a page an
    agent still holds survives the release (ForkKV guide, "Reference
    Counting and Eviction")."""
    pool = _pool(num_pages=8)
    h = pool.h
    idx = fk.RadixIndex(16)
    doc = list(range(16 * 3 + 5))
    m, _, _ = idx.match(doc)
    assert m == 0
    pages = fk.fk_pages_alloc(h, 3)                   # computed by the caller (case C)
    node = idx.insert(doc, pages)
    row = fk.fk_fork(h, pages)                        # one agent reads the prefix
    idx.adapter_attach(node, adapter=1, owner=0)
    assert [fk.fk_page_refcount(h, int(p)) for p in pages] == [2, 2, 2]
    assert idx.evict(3).size == 0                     # the adapter depends on it
    idx.adapter_detach(node, 1)
    freed = idx.evict(3)
    assert sorted(freed.tolist()) == sorted(pages.tolist())
    fk.fk_pages_release(h, freed)
    assert [fk.fk_page_refcount(h, int(p)) for p in pages] == [1, 1, 1]   # the agent's
    fk.fk_pages_release(h, row)
    assert [fk.fk_page_refcount(h, int(p)) for p in pages] == [0, 0, 0]
    again = fk.fk_pages_alloc(h, 8)                   # every page is free again
    assert again.size == 8
    pool.close()


def test_shared_a_rows_live_until_the_last_reader_is_released():
    pool = _pool(agents=4)
    h = pool.h
    Bk, Bv = _bf16((L, 16, H * D), 5), _bf16((L, 16, H * D), 6)
    fk.fk_agent_register(h, 0, 16, 1.0, Bk, Bv)
    fk.fk_agent_register_shared(h, 1, 0, 0.5, Bk, Bv)
    off0, lb0, rp0 = fk.fk_agent_rcache(h, 0)
    off1, lb1, rp1 = fk.fk_agent_rcache(h, 1)
    assert (off0, lb0, rp0) == (off1, lb1, rp1)
    with pytest.raises(fk.FKError):
        fk.fk_agent_register_shared(h, 2, 3, 1.0, Bk, Bv)     # source not registered
    fk.fk_agent_release(h, 0)
    assert fk.fk_agent_rcache(h, 1)[0] == off1                # agent 1 still reads the rows
    fk.fk_agent_register(h, 2, 16, 1.0, Bk, Bv)
    assert fk.fk_agent_rcache(h, 2)[0] != off1                # not handed out again
    fk.fk_agent_release(h, 1)
    fk.fk_agent_register(h, 3, 16, 1.0, Bk, Bv)
    assert fk.fk_agent_rcache(h, 3)[0] == off1                # reclaimed after the last reader
    pool.close()
