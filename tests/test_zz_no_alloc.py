"""tcclAllReduceNoAlloc: the allreduce for callers that cannot allocate GPU
memory (for example code running under another framework's memory manager,
or an out-of-memory handler), whose scratch is a static device array instead
of memory a group allocates.

Every call goes through the C ABI and is checked bit for bit against the CPU
oracle (the tolerance every parity test here uses), with canary guard zones
around every destination. Calls come two or more in a row, so each one runs
on scratch the previous call left behind. Cases: uncapped (dynamic chunk
order, whose counters the array holds), caps 8 and 16 (cyclic order), in
place, a send buffer 4 bytes off 16-byte alignment (element-wise edges bound
to CTAs, which uses the array's per-CTA table), int32, and each result also
against tcclAllReduce's. Then the error paths: a capturing stream is refused,
and a device-side timeout, made on purpose with the library's test hook (a
bounded wait on a barrier nothing signals, no fault), is reported by the next
call. This file is named to run last.
"""
import os

import numpy as np
import pytest
import torch

import collective_communication_planner_gb300 as tccl
import datagen
import oracle
from gpu_util import DT_CODE, Guarded, first_mismatch, to_device, to_host

pytestmark = pytest.mark.gpu

KIND = {"f32": "uniform_f32", "bf16": "normal_bf16", "i32": "int32"}


def no_alloc(sends, recvs, n, dtype, op, cap=0, stream=None):
    st = torch.cuda.current_stream().cuda_stream if stream is None else stream
    return tccl.tcclAllReduceNoAlloc(len(sends), sends, recvs, n, DT_CODE[dtype], tccl.OPS[op],
                                     st, cap)


def run_case(p, n, dtype, op, cap, in_place, send_off, seed):
    xs = datagen.rank_buffers(KIND[dtype], seed, p, n)
    exp = oracle.allreduce(xs, dtype, op, nthreads=0)
    sends = [Guarded(n, dtype, send_off) for _ in range(p)]
    for s, x in zip(sends, xs):
        s.tensor.copy_(to_device(x))
    recvs = sends if in_place else [Guarded(n, dtype) for _ in range(p)]
    r = no_alloc([s.tensor for s in sends], [t.tensor for t in recvs], n, dtype, op, cap)
    assert r == tccl.tcclSuccess, tccl.tcclGetErrorString(r)
    torch.cuda.synchronize()
    assert all(t.guards_intact() for t in recvs)
    for rank, t in enumerate(recvs):
        mm = first_mismatch(t.host(), exp[rank])
        assert mm is None, f"rank {rank}: first mismatch at {mm[0]} ({mm[1]} elements)"
    return xs


CASES = [
    # (P, count, dtype, op, cap, in place, send offset in bytes)
    (4, 1_000_003, "bf16", "sum", 0, False, 0),
    (8, 77_777, "f32", "max", 0, False, 0),
    (8, 300_001, "bf16", "sum", 8, False, 0),
    (3, 250_007, "f32", "sum", 16, False, 0),
    (8, 200_003, "f32", "min", 0, True, 0),
    (5, 123_457, "f32", "sum", 0, False, 4),
    (8, 150_001, "i32", "sum", 16, False, 0),
    (2, 2_000_000, "i32", "max", 0, True, 0),
]


def test_no_alloc_allreduce_matches_the_oracle_on_consecutive_calls():
    """All cases back to back (each on the scratch the previous one left),
    twice over, so every case also follows a call of another shape."""
    for rnd in range(2):
        for i, (p, n, dtype, op, cap, in_place, off) in enumerate(CASES):
            run_case(p, n, dtype, op, cap, in_place, off, seed=200 + 10 * i + rnd)


@pytest.mark.parametrize("cap", [0, 8, 16])
def test_no_alloc_allreduce_equals_the_group_allreduce(cap):
    p, n, dtype = 8, 400_003, "bf16"
    xs = datagen.rank_buffers(KIND[dtype], 300 + cap, p, n)
    sends = [to_device(x) for x in xs]
    via_group = [torch.empty_like(s) for s in sends]
    via_static = [torch.full_like(s, 7) for s in sends]
    with tccl.Group(p) as g:
        g.set_config(engine=tccl.tcclEngineBulk)
        g.all_reduce(sends, via_group, cta_cap=cap)
    for _ in range(2):
        assert no_alloc(sends, via_static, n, dtype, "sum", cap) == tccl.tcclSuccess
    torch.cuda.synchronize()
    exp = oracle.allreduce(xs, dtype, "sum", nthreads=0)
    for rank, (a, b) in enumerate(zip(via_group, via_static)):
        assert np.array_equal(to_host(b), exp[rank]), f"rank {rank}: differs from the oracle"
        assert np.array_equal(to_host(a), to_host(b)), f"rank {rank}: differs from tcclAllReduce"


def test_no_alloc_allreduce_rejects_what_tcclallreduce_rejects():
    a = torch.zeros(64, device="cuda")
    b = torch.zeros(64, device="cuda")
    assert tccl.tcclAllReduceNoAlloc(2, [a, b], [a[:32], a[16:48]], 32, 0, 0, 0, 0) == \
        tccl.tcclInvalidArgument
    assert tccl.tcclAllReduceNoAlloc(0, [a], [a], 64, 0, 0, 0, 0) == tccl.tcclInvalidArgument


def test_no_alloc_allreduce_refuses_a_capturing_stream():
    p, n = 2, 4096
    sends = [torch.ones(n, device="cuda") for _ in range(p)]
    recvs = [torch.zeros(n, device="cuda") for _ in range(p)]
    assert no_alloc(sends, recvs, n, "f32", "sum") == tccl.tcclSuccess  # set-up outside capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        r = no_alloc(sends, recvs, n, "f32", "sum", stream=s.cuda_stream)
    assert r == tccl.tcclInvalidUsage
    del graph
    # the stream and the library work as before
    for t in recvs:
        t.zero_()
    assert no_alloc(sends, recvs, n, "f32", "sum") == tccl.tcclSuccess
    torch.cuda.synchronize()
    assert all(bool((t == p).all()) for t in recvs)


def test_no_alloc_allreduce_reports_a_device_timeout_on_the_next_call():
    p, n, dtype = 4, 600_001, "f32"
    xs = datagen.rank_buffers(KIND[dtype], 400, p, n)
    exp = oracle.allreduce(xs, dtype, "sum", nthreads=0)
    sends = [to_device(x) for x in xs]
    recvs = [torch.zeros_like(s) for s in sends]
    os.environ["TCCL_NO_ALLOC_INJECT_TIMEOUT_MS"] = "30"
    try:
        # the first CTA waits 30 ms on a barrier nothing signals, gives up,
        # records the timeout and skips its work; the call itself launched
        assert no_alloc(sends, recvs, n, dtype, "sum") == tccl.tcclSuccess
        torch.cuda.synchronize()
    finally:
        del os.environ["TCCL_NO_ALLOC_INJECT_TIMEOUT_MS"]
    # the next call finds the record, reports it, launches nothing
    for t in recvs:
        t.fill_(-1.0)
    torch.cuda.synchronize()
    assert no_alloc(sends, recvs, n, dtype, "sum") == tccl.tcclDeviceTimeout
    torch.cuda.synchronize()
    assert all(bool((t == -1.0).all()) for t in recvs), "a refused call must launch nothing"
    # the record is cleared: calls run again, and the context is intact
    for _ in range(2):
        assert no_alloc(sends, recvs, n, dtype, "sum") == tccl.tcclSuccess
    torch.cuda.synchronize()
    assert no_alloc(sends, recvs, n, dtype, "sum") == tccl.tcclSuccess
    torch.cuda.synchronize()
    for rank, t in enumerate(recvs):
        assert np.array_equal(to_host(t), exp[rank]), f"rank {rank} after the timeout"
