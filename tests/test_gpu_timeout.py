"""Failure detection on the GPU without a fault: a wait that nothing
completes gives up after its bound, the call's CTAs unwind through their
abort path, fk_check reports FK_ERR_TIMEOUT, and the next call on the same
pool and context is correct again."""
import numpy as np
import pytest
import torch

import shared_base_kv_gb300 as fk
import workloads
from shared_base_kv_gb300 import harness
from _gpu_util import MAX_ABS, MEAN_ABS, errors, oracle_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def test_bounded_wait_gives_up_and_the_pool_recovers():
    w = workloads.make_workload("tiny", "peaked")
    dw = harness.DeviceWorkload(w)
    good = dw.attention(0).float().cpu().numpy()
    dw.check()
    fk.fk_pool_set_test_stall(dw.pool.h, True)
    dw.attention(0)
    with pytest.raises(fk.FKError) as e:
        dw.check()                      # synchronises: the stalled call has finished
    assert e.value.code == fk.FK_ERR_TIMEOUT
    assert "waits" in str(e.value)
    fk.fk_pool_set_test_stall(dw.pool.h, False)
    dw.check()                          # the error words were cleared
    again = dw.attention(0).float().cpu().numpy()
    dw.check()
    assert np.array_equal(again, good)
    mx, mean, _ = errors(again, oracle_out(w, 0))
    assert mx <= MAX_ABS and mean <= MEAN_ABS
