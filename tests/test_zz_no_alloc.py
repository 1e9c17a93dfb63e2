"""tcclAllReduceNoAlloc: the allreduce for callers that cannot allocate GPU
memory (for example code running under another framework's memory manager,
or an out-of-memory handler), whose scratch is a static device array instead
of memory a group allocates.

Called through the C ABI twice in a row with different shapes, each result
must equal tcclAllReduce's output on the same inputs, bit for bit (the
tolerance every parity test here uses). This file is named to run last.
"""
import pytest
import torch

import collective_communication_planner_gb300 as tccl
import datagen
from gpu_util import DT_CODE, same_bits, to_device, to_host

pytestmark = pytest.mark.gpu

KIND = {"f32": "uniform_f32", "bf16": "normal_bf16", "i32": "int32"}


def test_no_alloc_allreduce_matches_group_allreduce_on_consecutive_calls():
    stream = torch.cuda.current_stream().cuda_stream
    cases = [(4, 1_000_003, "bf16", "sum"), (8, 77_777, "f32", "max")]
    for call, (p, n, dtype, op) in enumerate(cases):
        xs = datagen.rank_buffers(KIND[dtype], 100 + call, p, n)
        sends = [to_device(x) for x in xs]
        via_group = [torch.empty_like(s) for s in sends]
        via_static = [torch.full_like(s, 7) for s in sends]
        with tccl.Group(p) as g:
            g.set_config(engine=tccl.tcclEngineBulk)
            g.all_reduce(sends, via_group, op=op)
        r = tccl.tcclAllReduceNoAlloc(p, sends, via_static, n, DT_CODE[dtype], tccl.OPS[op],
                                      stream, 0)
        assert r == tccl.tcclSuccess, tccl.tcclGetErrorString(r)
        torch.cuda.synchronize()
        for a, b in zip(via_group, via_static):
            assert same_bits(to_host(a), to_host(b)), f"call {call}: outputs differ"


def test_no_alloc_allreduce_rejects_what_tcclallreduce_rejects():
    a = torch.zeros(64, device="cuda")
    b = torch.zeros(64, device="cuda")
    assert tccl.tcclAllReduceNoAlloc(2, [a, b], [a[:32], a[16:48]], 32, 0, 0, 0, 0) == \
        tccl.tcclInvalidArgument
    assert tccl.tcclAllReduceNoAlloc(0, [a], [a], 64, 0, 0, 0, 0) == tccl.tcclInvalidArgument
