"""The multi-GPU path is replicas only: each rank runs its own copy of the
workload and the job throughput is (units of all ranks) / (slowest rank's
time).  Checked here with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    total_ms = [40.0, 50.0][rank]
    e2e_ms = [60.0, 45.0][rank]
    res = bench.reduce_over_ranks(total_ms, e2e_ms, units=800, e2e_units=400, world=world,
                                  device=torch.device("cpu"))
    out[rank] = res
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_take_slowest_rank():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        r0, r1 = out[0], out[1]
    assert r0 == r1
    value, total_ms, e2e_value, e2e_ms = r0
    assert total_ms == 50.0 and e2e_ms == 60.0
    assert value == pytest.approx(800 * 2 / 0.050)
    assert e2e_value == pytest.approx(400 * 2 / 0.060)


def test_single_rank_needs_no_process_group():
    import bench
    v, t, ev, et = bench.reduce_over_ranks(10.0, 20.0, 8, 4, 1, torch.device("cpu"))
    assert (v, t, ev, et) == (800.0, 10.0, 200.0, 20.0)



def _worker_leaves(rank, world, port, out):
    from datetime import timedelta
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=timedelta(seconds=5))
    import bench
    if rank == 1:
        # this rank leaves between steps: it never joins the step's reduction
        out[1] = "left"
        os._exit(0)
    try:
        bench.reduce_over_ranks(40.0, 60.0, units=800, e2e_units=400, world=world,
                                device=torch.device("cpu"))
        out[0] = "completed"
    except Exception as e:                          # the collective ends with an error
        out[0] = f"error: {type(e).__name__}"
    os._exit(0)


def test_a_rank_that_leaves_ends_the_reduction_with_an_error():
    # the surviving rank learns of it through its next collective, which
    # fails (closed connection or the short process-group timeout) instead
    # of waiting forever
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        ctx = mp.spawn(_worker_leaves, args=(2, port, out), nprocs=2, join=False)
        for _ in range(120):
            if ctx.join(timeout=1):
                break
        else:
            for p in ctx.processes:
                p.kill()
            pytest.fail("the surviving rank did not return")
        assert out[1] == "left"
        assert out[0].startswith("error")
