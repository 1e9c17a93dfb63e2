"""GPU parity for the bulk engine's shared-memory ring under refill pressure.

A stage is read by the consumer warps through ordinary shared-memory loads
and then refilled by the producer's bulk copies, which run in the async
proxy. The consumers release a stage only after a proxy fence. Without that
fence, a release can overtake loads whose values are still in flight, and
the next bulk copy then overwrites data that a warp has not read yet. The
race is rare, so each layout and store mode runs many calls back to back.
Deep rings, few consumer warps and a CTA cap keep the producer ahead and
waiting to refill. Every output element of every call is compared with the
oracle, bit for bit, on the device.
"""
import numpy as np
import pytest
import torch

import collective_communication_planner_gb300 as tccl
import datagen
import oracle
from gpu_util import to_device

pytestmark = pytest.mark.gpu
P, COUNT, CALLS = 8, 4 << 20, 12


@pytest.fixture(scope="module")
def setup():
    xs = datagen.rank_buffers("normal_bf16", 51, P, COUNT)
    exp = to_device(oracle.allreduce(xs, "bf16", "sum", nthreads=0)[0])
    sends = [to_device(x) for x in xs]
    recvs = [torch.empty_like(s) for s in sends]
    g = tccl.Group(P)
    yield g, sends, recvs, exp
    g.close()


@pytest.mark.parametrize("layout,store", [(tccl.tcclLayoutShared, tccl.tcclStoreVec),
                                          (tccl.tcclLayoutShared, tccl.tcclStoreBulk),
                                          (tccl.tcclLayoutPerRank, tccl.tcclStoreVec)])
@pytest.mark.parametrize("stages", [2, 8])
@pytest.mark.parametrize("cap", [0, 8])
def test_ring_refill_is_exact(setup, layout, store, stages, cap):
    g, sends, recvs, exp = setup
    g.set_config(engine=tccl.tcclEngineBulk, stage_layout=layout, store_mode=store, stages=stages,
                 consumer_warps=4)
    st = torch.cuda.current_stream()
    bad = []
    for call in range(CALLS):
        for r in recvs:
            r.fill_(0)
        rc = tccl.tcclAllReduce(g.handle, sends, recvs, COUNT, tccl.DTYPES["bf16"], tccl.OPS["sum"],
                                st.cuda_stream, cap)
        assert rc == tccl.tcclSuccess, tccl.tcclGetErrorString(rc)
        for r in range(P):
            if not torch.equal(recvs[r].view(torch.int16), exp.view(torch.int16)):
                bad.append((call, r, int((recvs[r].view(torch.int16) != exp.view(torch.int16)).sum())))
    torch.cuda.synchronize()
    assert g.query_error() == tccl.tcclSuccess
    info = g.last_launch()
    assert info["engine"] == tccl.tcclEngineBulk and info["stage_layout"] == layout, info
    assert not bad, f"calls with mismatches (call, rank, elements): {bad[:8]}"
