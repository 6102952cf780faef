"""fk_residual_attention_noalloc: the same attention for callers that may not
allocate device memory (its scratch is a fixed array inside the library).
Checked through the C ABI against fk_residual_attention on two calls in a
row; collected last so that a stop at the first failure has already run
everything else, and written to pass in a fresh process as well."""
import numpy as np
import pytest
import torch

import shared_base_kv_gb300 as fk
import workloads
from shared_base_kv_gb300 import harness

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _call(fn, dw, q):
    w = dw.w
    out = torch.full_like(q, float("nan"))
    fn(dw.pool.h, 0, q, np.arange(w.A, dtype=np.int32), dw.block_table, w.seq_lens, w.causal,
       dw.compressed is not None, out)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("name,kw", [
    ("llama8b_32k", dict(prefix=1000, A=8)),
    ("agents32_layers32", dict(prefix=200, suffix=(0, 40), A=9, n_layers=1)),
    ("qwen72b_chunk", dict(prefix=300, A=3)),          # the chunk kernel's work list
    ("compressed", dict(prefix=500, A=6)),             # the compressed pool
])
def test_noalloc_matches_pool_workspace_call(name, kw):
    w = workloads.make_workload(name, "strong", **kw)
    dw = harness.DeviceWorkload(w, compressed="gpu" if name == "compressed" else None)
    q = dw.queries(0)
    ref = _call(fk.fk_residual_attention, dw, q).float()
    for _ in range(2):                      # two calls in a row share the array
        got = _call(fk.fk_residual_attention_noalloc, dw, q).float()
        assert torch.isfinite(got).all()
        err = (got - ref).abs()
        assert err.max().item() <= 2e-2 and err.mean().item() <= 2e-3
        assert torch.equal(got, ref)        # same kernels, same work list
    dw.check()


def test_noalloc_rejects_calls_beyond_the_array():
    w = workloads.make_workload("qwen72b_chunk", prefix=4096, A=16)
    dw = harness.DeviceWorkload(w)
    q = dw.queries(0)
    with pytest.raises(fk.FKError) as e:
        _call(fk.fk_residual_attention_noalloc, dw, q)
    assert e.value.code == fk.FK_ERR_OOM
    assert "static array" in str(e.value)


def test_noalloc_replans_after_an_agent_is_registered_again():
    # the no-allocation entry point caches its work list, which carries the
    # agents' ranks and residual scales; registering an agent again (here
    # with three times the scale) must not reuse it
    w = workloads.make_workload("llama8b_32k", "strong", prefix=1000, A=8)
    dw = harness.DeviceWorkload(w)
    q = dw.queries(0)
    first = _call(fk.fk_residual_attention_noalloc, dw, q).float()
    h = dw.pool.h
    ld = w.layer(0)
    Bk = torch.stack([w.layer(l).bk[0] for l in range(w.n_layers)]).cuda().contiguous()
    Bv = torch.stack([w.layer(l).bv[0] for l in range(w.n_layers)]).cuda().contiguous()
    fk.fk_agent_release(h, 0)
    fk.fk_agent_register(h, 0, int(w.ranks[0]), 3.0 * w.s, Bk, Bv)
    fk.fk_residual_append(h, 0, 0, 0, ld.lk[0].cuda().contiguous(), ld.lv[0].cuda().contiguous())
    ref = _call(fk.fk_residual_attention, dw, q).float()
    got = _call(fk.fk_residual_attention_noalloc, dw, q).float()
    assert torch.equal(got, ref)
    assert not torch.equal(got[0], first[0])          # agent 0's rows see the new scale
    assert torch.equal(got[1:], first[1:])            # the others do not change
    dw.check()


def test_noalloc_does_not_reuse_a_destroyed_pools_work_list():
    # two pools in a row with the same call inputs (agents, block table,
    # sequence lengths) but other ranks: the second pool may get the first
    # one's address, and its work list (tiles formed by rank) differs
    kw = dict(prefix=200, suffix=(0, 40), A=9, n_layers=1)
    w1 = workloads.make_workload("agents32_layers32", "strong", **kw)
    dw1 = harness.DeviceWorkload(w1)
    _call(fk.fk_residual_attention_noalloc, dw1, dw1.queries(0))
    dw1.pool.close()
    del dw1
    w2 = workloads.make_workload("agents32_layers32", "strong", ranks=(64,), **kw)
    assert np.array_equal(w1.seq_lens, w2.seq_lens)
    dw2 = harness.DeviceWorkload(w2)
    q = dw2.queries(0)
    ref = _call(fk.fk_residual_attention, dw2, q)
    got = _call(fk.fk_residual_attention_noalloc, dw2, q)
    assert torch.equal(got, ref)
    dw2.check()


def test_noalloc_eight_slot_tiles(monkeypatch):
    # a pool planned in eight-slot tiles: the same static array carries that
    # kernel's work list
    monkeypatch.setenv("FORKKV_DECODE_SLOTS", "8")
    w = workloads.make_workload("llama8b_32k", "strong", prefix=1000, A=8)
    dw = harness.DeviceWorkload(w)
    q = dw.queries(0)
    ref = _call(fk.fk_residual_attention, dw, q)
    got = _call(fk.fk_residual_attention_noalloc, dw, q)
    assert torch.equal(got, ref)
    assert fk.fk_last_launch_count(dw.pool.h) == 2        # eight-slot kernel + combine
    dw.check()
