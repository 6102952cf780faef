"""Calls captured in a CUDA graph: once a call's work list is cached (the
first call with the same inputs), a repeat call enqueues only its kernel
launches, so it can be captured on a side stream and replayed.  Replays
must equal eager calls bit for bit, for both entry points and both decode
tilings."""
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


@pytest.mark.parametrize("slots", ["4", "8"])
@pytest.mark.parametrize("entry", ["fk_residual_attention", "fk_residual_attention_noalloc"])
def test_graph_replay_equals_eager_call(monkeypatch, slots, entry):
    monkeypatch.setenv("FORKKV_DECODE_SLOTS", slots)
    w = workloads.make_workload("llama8b_32k", "strong", prefix=900, A=8)
    dw = harness.DeviceWorkload(w)
    fn = getattr(fk, entry)
    q = dw.queries(0)
    agents = np.arange(w.A, dtype=np.int32)
    side = torch.cuda.Stream()
    eager = torch.empty_like(q)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn(dw.pool.h, 0, q, agents, dw.block_table, w.seq_lens, False, False, eager, side)
    torch.cuda.synchronize()
    out = torch.full_like(q, float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        fn(dw.pool.h, 0, q, agents, dw.block_table, w.seq_lens, False, False, out, side)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    dw.check()
