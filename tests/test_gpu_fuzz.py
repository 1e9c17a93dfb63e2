"""Randomised GPU parity: seeded random calls over every engine a user or
Auto can pick (Auto, bulk, warp, vec, copy-out), every collective, dtype and
op, P from 1 to 12, counts from 1 to ~300k elements, misaligned buffers,
in-place forms and CTA caps, each checked bit for bit against the CPU oracle
with guard zones around every destination."""
import numpy as np
import pytest
import torch

import collective_communication_planner_gb300 as tccl
import datagen
import oracle
from gpu_util import DT_CODE, Guarded, first_mismatch, to_device

pytestmark = pytest.mark.gpu
KIND = {"f32": "uniform_f32", "bf16": "normal_bf16", "i32": "int32"}
ES = {"f32": 4, "bf16": 2, "i32": 4}
ENGINES = [tccl.tcclEngineAuto, tccl.tcclEngineBulk, tccl.tcclEngineWarp, tccl.tcclEngineVec,
           tccl.tcclEngineCopyOut]


@pytest.fixture(scope="module")
def groups():
    made = {}

    def get(p):
        if p not in made:
            made[p] = tccl.Group(p)
        return made[p]

    yield get
    for g in made.values():
        g.close()


def draw(rng):
    coll = rng.choice(["AR", "RS", "AG"])
    p = int(rng.integers(1, 13))
    dtype = rng.choice(["f32", "bf16", "i32"])
    op = "sum" if coll == "AG" else rng.choice(["sum", "min", "max"])
    count = int(rng.choice([rng.integers(1, 100), rng.integers(100, 20_000), rng.integers(20_000, 300_000)]))
    es = ES[dtype]
    mis = [int(rng.integers(0, 16 // es)) * es, int(rng.integers(0, 16 // es)) * es]
    if rng.random() < 0.5:
        mis[1] = mis[0]  # co-aligned half the time (the vector paths)
    in_place = bool(rng.random() < 0.3)
    cap = int(rng.choice([0, 0, 1, 3, 8, 16, 40]))
    engine = int(rng.choice(ENGINES))
    seg = int(rng.choice([0, 4096, 65536]))
    return coll, p, dtype, op, count, mis, in_place, cap, engine, seg


@pytest.mark.parametrize("case", range(120))
def test_random_call(groups, case):
    rng = np.random.default_rng(1000 + case)
    coll, p, dtype, op, count, mis, in_place, cap, engine, seg = draw(rng)
    g = groups(p)
    c = tccl.tcclConfig_t()
    c.engine = engine
    c.ce_segment_bytes = seg
    assert tccl.tcclGroupSetConfig(g.handle, c) == tccl.tcclSuccess
    what = f"{coll} P={p} {dtype} {op} count={count} mis={mis} in_place={in_place} cap={cap} engine={engine} seg={seg}"
    st = torch.cuda.current_stream().cuda_stream
    if coll == "AR":
        xs = datagen.rank_buffers(KIND[dtype], case, p, count)
        sends = [Guarded(count, dtype, mis[0]) for _ in range(p)]
        for s_, x in zip(sends, xs):
            s_.tensor.copy_(to_device(x))
        recvs = sends if in_place else [Guarded(count, dtype, mis[1]) for _ in range(p)]
        r = tccl.tcclAllReduce(g.handle, [t.tensor for t in sends], [t.tensor for t in recvs], count,
                               DT_CODE[dtype], tccl.OPS[op], st, cap)
        exp = oracle.allreduce(xs, dtype, op, nthreads=0)
        outs = recvs
        views = None
    elif coll == "RS":
        xs = datagen.rank_buffers(KIND[dtype], case, p, p * count)
        sends = [Guarded(p * count, dtype, mis[0]) for _ in range(p)]
        for s_, x in zip(sends, xs):
            s_.tensor.copy_(to_device(x))
        if in_place:
            outs = None
            views = [s_.tensor[k * count:(k + 1) * count] for k, s_ in enumerate(sends)]
        else:
            outs = [Guarded(count, dtype, mis[1]) for _ in range(p)]
            views = [t.tensor for t in outs]
        r = tccl.tcclReduceScatter(g.handle, [s_.tensor for s_ in sends], views, count, DT_CODE[dtype],
                                   tccl.OPS[op], st, cap)
        exp = oracle.reduce_scatter(xs, dtype, op, nthreads=0)
    else:
        xs = datagen.rank_buffers(KIND[dtype], case, p, count)
        outs = [Guarded(p * count, dtype, mis[1]) for _ in range(p)]
        if in_place:
            for k, t in enumerate(outs):
                t.tensor[k * count:(k + 1) * count].copy_(to_device(xs[k]))
            sends_t = [t.tensor[k * count:(k + 1) * count] for k, t in enumerate(outs)]
            sends = None
        else:
            sends = [Guarded(count, dtype, mis[0]) for _ in range(p)]
            for s_, x in zip(sends, xs):
                s_.tensor.copy_(to_device(x))
            sends_t = [s_.tensor for s_ in sends]
        r = tccl.tcclAllGather(g.handle, sends_t, [t.tensor for t in outs], count, DT_CODE[dtype], st, cap)
        exp = [np.concatenate(xs)] * p
        views = None
    assert r == tccl.tcclSuccess, f"{what}: {tccl.tcclGetErrorString(r)}"
    torch.cuda.synchronize()
    assert g.query_error() == tccl.tcclSuccess, what
    if outs is not None:
        assert all(t.guards_intact() for t in outs), f"{what}: a guard zone was written"
        got = [t.host() for t in outs]
    else:
        from gpu_util import to_host
        got = [to_host(v) for v in views]
    for k in range(p):
        mm = first_mismatch(got[k], exp[k])
        assert mm is None, f"{what}: rank {k} first mismatch at {mm[0]} ({mm[1]} elements)"
