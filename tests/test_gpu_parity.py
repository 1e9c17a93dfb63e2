"""GPU parity: every engine, collective, dtype and op against the CPU oracle,
bit for bit, through the C ABI.

Sizes span several chunks per CTA and end in ragged tails; edge cases cover
P = 1, counts smaller than P, misaligned and mutually misaligned buffers,
in-place forms, CTA caps, guard zones around every destination, the
bounded-wait timeout path and CUDA graph replay.
"""
import numpy as np
import pytest
import torch

import collective_communication_planner_gb300 as tccl
import datagen
import oracle
from gpu_util import (DT_CODE, NP_OF, TORCH_OF, Guarded, first_mismatch, same_bits, to_device, to_host,
                      within_summation_bound)

pytestmark = pytest.mark.gpu

ENGINES = {"bulk": tccl.tcclEngineBulk, "warp": tccl.tcclEngineWarp, "vec": tccl.tcclEngineVec}
KIND = {"f32": "uniform_f32", "bf16": "normal_bf16", "i32": "int32"}


def inputs(dtype, p, n, seed=11):
    return datagen.rank_buffers(KIND[dtype], seed, p, n)


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


def reset_config(g, **kw):
    """Library defaults (a zeroed config) plus the given fields."""
    c = tccl.tcclConfig_t()
    for k, v in kw.items():
        setattr(c, k, v)
    assert tccl.tcclGroupSetConfig(g.handle, c) == tccl.tcclSuccess


def configure(g, engine, store=tccl.tcclStoreAuto, stage_bytes=0, stages=0):
    reset_config(g, engine=ENGINES[engine] if isinstance(engine, str) else engine,
                 store_mode=store, stage_bytes=stage_bytes, stages=stages)


def run_allreduce(g, xs, dtype, op, cap=0, send_off=0, recv_off=0, in_place=False):
    p, n = len(xs), xs[0].size
    sends = [Guarded(n, dtype, send_off) for _ in range(p)]
    for s, x in zip(sends, xs):
        s.tensor.copy_(to_device(x))
    recvs = sends if in_place else [Guarded(n, dtype, recv_off) for _ in range(p)]
    r = tccl.tcclAllReduce(g.handle, [s.tensor for s in sends], [t.tensor for t in recvs], n,
                           DT_CODE[dtype], tccl.OPS[op], torch.cuda.current_stream().cuda_stream,
                           cap)
    assert r == tccl.tcclSuccess, tccl.tcclGetErrorString(r)
    torch.cuda.synchronize()
    assert g.query_error() == tccl.tcclSuccess
    for t in recvs:
        assert t.guards_intact()
    return [t.host() for t in recvs]


def assert_ranks_equal(got, exp, what):
    for r in range(len(exp)):
        mm = first_mismatch(got[r], exp[r])
        assert mm is None, f"{what}: rank {r} first mismatch at {mm[0]} ({mm[1]} elements)"


# ------------------------------------------------------------------ allreduce
@pytest.mark.parametrize("engine", ["bulk", "warp", "vec"])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "min", "max"])
def test_allreduce_engines_dtypes_ops(groups, engine, dtype, op):
    for p, n in ((2, 70_001), (3, 1000), (8, 300_007), (5, 17), (4, 33_337)):
        g = groups(p)
        configure(g, engine)
        xs = inputs(dtype, p, n)
        exp = oracle.allreduce(xs, dtype, op, nthreads=0)
        got = run_allreduce(g, xs, dtype, op)
        assert_ranks_equal(got, exp, f"AR {engine} {dtype} {op} P={p} n={n}")


@pytest.mark.parametrize("engine", ["bulk", "warp", "vec"])
@pytest.mark.parametrize("n", [1, 2, 3, 7, 8, 9, 15, 16, 17, 63, 64, 65, 4095, 4096, 4097])
def test_allreduce_small_and_ragged_counts(groups, engine, n):
    for p in (1, 2, 8, 16):
        g = groups(p)
        configure(g, engine)
        xs = inputs("bf16", p, n, seed=n)
        exp = oracle.allreduce(xs, "bf16", "sum")
        assert_ranks_equal(run_allreduce(g, xs, "bf16", "sum"), exp, f"{engine} P={p} n={n}")


@pytest.mark.parametrize("engine", ["bulk", "vec", "warp"])
@pytest.mark.parametrize("offs", [(4, 4), (8, 8), (12, 12), (4, 8), (0, 4), (2, 2)])
def test_allreduce_misaligned_buffers(groups, engine, offs):
    p, n = 4, 50_001
    dtype = "bf16" if offs[0] % 4 or offs[1] % 4 else "f32"
    g = groups(p)
    configure(g, engine)
    xs = inputs(dtype, p, n)
    exp = oracle.allreduce(xs, dtype, "sum")
    got = run_allreduce(g, xs, dtype, "sum", send_off=offs[0], recv_off=offs[1])
    assert_ranks_equal(got, exp, f"misaligned {offs}")


@pytest.mark.parametrize("p", [4, 8])
@pytest.mark.parametrize("kib", [1, 16, 64])
def test_auto_small_engine_by_placement(groups, p, kib):
    """Under Auto a small out-of-place allreduce over 8 ranks runs on the vec
    engine and an in-place one on the warp engine; over 4 ranks both take the
    warp engine. Every result matches the oracle."""
    g = groups(p)
    reset_config(g)
    n = kib * 512  # bf16 elements
    xs = inputs("bf16", p, n, seed=kib + p)
    exp = oracle.allreduce(xs, "bf16", "sum")
    assert_ranks_equal(run_allreduce(g, xs, "bf16", "sum"), exp, f"out of place P={p} {kib} KiB")
    assert g.last_launch()["engine"] == (tccl.tcclEngineVec if p == 8 else tccl.tcclEngineWarp)
    assert_ranks_equal(run_allreduce(g, xs, "bf16", "sum", in_place=True), exp, f"in place P={p} {kib} KiB")
    assert g.last_launch()["engine"] == tccl.tcclEngineWarp


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("lanes_per_sm", [1, 27, 191, 192, 193, 300])
def test_vec_engine_grid_shapes(groups, dtype, lanes_per_sm):
    """The vec engine's grid: one CTA per SM of the lanes / SMs rounded up to a
    warp up to 192 lanes per SM, CTAs of 256 above. Counts on both sides of
    that bound, with a ragged tail of scalar elements, in place and out of
    place, the vec engine forced."""
    p = 8
    g = groups(p)
    configure(g, "vec")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    epv = 4 if dtype == "f32" else 8  # elements per 16-byte vector
    n = lanes_per_sm * sms * epv + 3
    xs = inputs(dtype, p, n, seed=lanes_per_sm)
    exp = oracle.allreduce(xs, dtype, "sum", nthreads=0)
    assert_ranks_equal(run_allreduce(g, xs, dtype, "sum"), exp, f"vec {dtype} {lanes_per_sm}/SM")
    info = g.last_launch()
    assert info["engine"] == tccl.tcclEngineVec
    if lanes_per_sm <= 192:
        assert info["ctas"] <= sms and info["threads"] % 32 == 0 and info["threads"] <= 256, info
    else:
        assert info["threads"] == 256, info
    assert_ranks_equal(run_allreduce(g, xs, dtype, "sum", in_place=True), exp, f"vec in place {dtype}")


@pytest.mark.parametrize("engine", ["bulk", "warp", "vec"])
@pytest.mark.parametrize("dtype", ["f32", "i32"])
def test_allreduce_in_place(groups, engine, dtype):
    p, n = 8, 123_457
    g = groups(p)
    configure(g, engine)
    xs = inputs(dtype, p, n)
    exp = oracle.allreduce(xs, dtype, "sum")
    got = run_allreduce(g, xs, dtype, "sum", in_place=True)
    assert_ranks_equal(got, exp, "in place")


@pytest.mark.parametrize("store", [tccl.tcclStoreBulk, tccl.tcclStoreVec])
@pytest.mark.parametrize("stage_bytes,stages", [(0, 0), (4096, 2), (65536, 3), (16384, 12)])
def test_bulk_store_modes_and_pipeline_shapes(groups, store, stage_bytes, stages):
    p, n = 4, 1_000_003
    g = groups(p)
    reset_config(g, engine=tccl.tcclEngineBulk, store_mode=store, stage_bytes=stage_bytes,
                 stages=stages, stage_layout=tccl.tcclLayoutShared)
    xs = inputs("bf16", p, n)
    exp = oracle.allreduce(xs, "bf16", "sum", nthreads=0)
    got = run_allreduce(g, xs, "bf16", "sum")
    info = g.last_launch()
    assert info["engine"] == tccl.tcclEngineBulk and info["store_mode"] == store
    assert info["stage_layout"] == tccl.tcclLayoutShared
    assert_ranks_equal(got, exp, f"store {store} stage {stage_bytes}x{stages}")


ORDERS = {"blocked": tccl.tcclOrderBlocked, "cyclic": tccl.tcclOrderCyclic,
          "dynamic": tccl.tcclOrderDynamic}


@pytest.mark.parametrize("order", ["blocked", "cyclic", "dynamic"])
@pytest.mark.parametrize("store", [tccl.tcclStoreBulk, tccl.tcclStoreVec])
def test_bulk_chunk_orders_all_collectives(groups, order, store):
    p, n = 4, 2_000_003
    g = groups(p)
    reset_config(g, engine=tccl.tcclEngineBulk, store_mode=store, chunk_order=ORDERS[order],
                 stage_bytes=0, stages=0)
    xs = inputs("bf16", p, n)
    for rep in range(2):  # the dynamic order's counter must be reset between launches
        got = run_allreduce(g, xs, "bf16", "sum", cap=17 if rep else 0)
        assert g.last_launch()["chunk_order"] == ORDERS[order]
        assert_ranks_equal(got, oracle.allreduce(xs, "bf16", "sum", nthreads=0), f"AR {order}")
    rc = n // p
    sends = [to_device(x[:p * rc]) for x in xs]
    parts = [torch.empty(rc, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    outs = [torch.empty(p * rc, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    g.reduce_scatter(sends, parts)
    g.all_gather(parts, outs)
    torch.cuda.synchronize()
    assert g.query_error() == tccl.tcclSuccess
    exp_rs = oracle.reduce_scatter([x[:p * rc] for x in xs], "bf16", "sum", nthreads=0)
    assert_ranks_equal([to_host(t) for t in parts], exp_rs, f"RS {order}")
    assert_ranks_equal([to_host(t) for t in outs], oracle.allgather(exp_rs), f"AG {order}")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "min", "max"])
@pytest.mark.parametrize("cw", [8, 16])
def test_per_rank_stage_layout(groups, dtype, op, cw):
    for p, n, cap in ((2, 1_000_003, 0), (8, 700_001, 0), (5, 123_457, 7), (8, 1 << 20, 16)):
        g = groups(p)
        reset_config(g, engine=tccl.tcclEngineBulk, stage_layout=tccl.tcclLayoutPerRank,
                     consumer_warps=cw, store_mode=0, stage_bytes=0, stages=0, chunk_order=0)
        xs = inputs(dtype, p, n)
        got = run_allreduce(g, xs, dtype, op, cap=cap)
        info = g.last_launch()
        assert info["stage_layout"] == tccl.tcclLayoutPerRank
        assert_ranks_equal(got, oracle.allreduce(xs, dtype, op, nthreads=0),
                           f"per-rank AR {dtype} {op} P={p} cap={cap}")
    # reduce-scatter through the same layout
    p, rc = 4, 250_007
    g = groups(p)
    xs = inputs(dtype, p, p * rc)
    sends = [to_device(x) for x in xs]
    parts = [torch.empty(rc, dtype=TORCH_OF[dtype], device="cuda") for _ in range(p)]
    g.reduce_scatter(sends, parts, op=op)
    torch.cuda.synchronize()
    assert g.query_error() == tccl.tcclSuccess
    assert_ranks_equal([to_host(t) for t in parts],
                       oracle.reduce_scatter(xs, dtype, op, nthreads=0), "per-rank RS")


def test_per_rank_layout_many_ranks(groups):
    p, n = 64, 200_003
    g = groups(p)
    xs = inputs("bf16", p, n)
    exp = oracle.allreduce(xs, "bf16", "sum", nthreads=0)
    for layout in (tccl.tcclLayoutShared, tccl.tcclLayoutPerRank):
        reset_config(g, engine=tccl.tcclEngineBulk, stage_layout=layout, consumer_warps=16,
                     store_mode=0, stage_bytes=0, stages=0, chunk_order=0)
        assert_ranks_equal(run_allreduce(g, xs, "bf16", "sum"), exp, f"P=64 layout {layout}")


TMA_REDUCE_PAIRS = [("f32", "sum"), ("i32", "sum"), ("i32", "min"), ("i32", "max"),
                    ("bf16", "min"), ("bf16", "max")]


@pytest.mark.parametrize("dtype,op", TMA_REDUCE_PAIRS)
def test_tma_reduce_engine(groups, dtype, op):
    for p, n, cap, offs in ((1, 10_000, 0, 0), (2, 1_000_003, 0, 0), (3, 77_777, 5, 4),
                            (8, 500_001, 0, 0), (8, 300_000, 16, 8)):
        g = groups(p)
        reset_config(g, engine=tccl.tcclEngineTmaReduce)
        xs = inputs(dtype, p, n)
        got = run_allreduce(g, xs, dtype, op, cap=cap, send_off=offs, recv_off=offs)
        assert p == 1 or g.last_launch()["engine"] == tccl.tcclEngineTmaReduce
        assert_ranks_equal(got, oracle.allreduce(xs, dtype, op, nthreads=0),
                           f"TMA-reduce AR {dtype} {op} P={p} cap={cap} off={offs}")
    p, n = 4, 200_003
    g = groups(p)
    reset_config(g, engine=tccl.tcclEngineTmaReduce)
    xs = inputs(dtype, p, n)
    got = run_allreduce(g, xs, dtype, op, in_place=True)
    assert_ranks_equal(got, oracle.allreduce(xs, dtype, op, nthreads=0), "TMA-reduce in place")
    rc = 123_457
    xs = inputs(dtype, p, p * rc)
    sends = [to_device(x) for x in xs]
    parts = [torch.empty(rc, dtype=TORCH_OF[dtype], device="cuda") for _ in range(p)]
    g.reduce_scatter(sends, parts, op=op)
    torch.cuda.synchronize()
    assert g.query_error() == tccl.tcclSuccess
    assert_ranks_equal([to_host(t) for t in parts],
                       oracle.reduce_scatter(xs, dtype, op, nthreads=0), "TMA-reduce RS")


@pytest.mark.parametrize("dtype,op", TMA_REDUCE_PAIRS)
def test_tma_reduce_arrival_order(groups, dtype, op):
    """tcclReduceArrival on the TMA-reduce engine: ranks 1..P-1 reduced back
    to back in whatever order the memory system applies them. Order-free pairs
    (int32 sum/min/max, bf16 min/max) stay bit-exact; an fp32 sum stays within
    the summation bound of the ascending fold. Allreduce and reduce-scatter,
    P = 2..8, a cap, misaligned buffers."""
    for p, n, cap, offs in ((2, 1_000_003, 0, 0), (3, 77_777, 5, 4), (8, 500_001, 0, 0),
                            (8, 300_000, 16, 8)):
        g = groups(p)
        reset_config(g, engine=tccl.tcclEngineTmaReduce, reduce_order=tccl.tcclReduceArrival)
        xs = inputs(dtype, p, n)
        got = run_allreduce(g, xs, dtype, op, cap=cap, send_off=offs, recv_off=offs)
        assert g.last_launch()["engine"] == tccl.tcclEngineTmaReduce
        exp = oracle.allreduce(xs, dtype, op, nthreads=0)
        what = f"TMA-reduce arrival AR {dtype} {op} P={p} cap={cap} off={offs}"
        if (dtype, op) == ("f32", "sum"):
            for r in range(p):
                ok, _ = within_summation_bound(got[r], exp[r], xs)
                assert ok, f"{what}: rank {r} outside the summation bound"
        else:
            assert_ranks_equal(got, exp, what)
    p, rc = 4, 123_457
    g = groups(p)
    reset_config(g, engine=tccl.tcclEngineTmaReduce, reduce_order=tccl.tcclReduceArrival)
    xs = inputs(dtype, p, p * rc)
    sends = [to_device(x) for x in xs]
    parts = [torch.empty(rc, dtype=TORCH_OF[dtype], device="cuda") for _ in range(p)]
    g.reduce_scatter(sends, parts, op=op)
    torch.cuda.synchronize()
    assert g.query_error() == tccl.tcclSuccess
    exp = oracle.reduce_scatter(xs, dtype, op, nthreads=0)
    got = [to_host(t) for t in parts]
    if (dtype, op) == ("f32", "sum"):
        for r in range(p):
            ok, _ = within_summation_bound(got[r], exp[r], [x[r * rc:(r + 1) * rc] for x in xs])
            assert ok, f"TMA-reduce arrival RS: rank {r} outside the summation bound"
    else:
        assert_ranks_equal(got, exp, "TMA-reduce arrival RS")
    reset_config(g)


@pytest.mark.parametrize("dtype,op", TMA_REDUCE_PAIRS)
@pytest.mark.parametrize("p", [2, 3, 8])
def test_tma_reduce_in_place_reduce_scatter(groups, dtype, op, p):
    """In place, shard s's owner chunk is rank s's own input chunk, which rank
    0's first store would overwrite: the engine loads it first and keeps it."""
    g = groups(p)
    for slots, cap in ((0, 0), (1, 5), (8, 0)):
        reset_config(g, engine=tccl.tcclEngineTmaReduce, reduce_slots=slots)
        rc = 50_021
        xs = inputs(dtype, p, p * rc)
        bufs = [to_device(x) for x in xs]
        parts = [b[r * rc:(r + 1) * rc] for r, b in enumerate(bufs)]
        g.reduce_scatter(bufs, parts, op=op, cta_cap=cap)
        torch.cuda.synchronize()
        assert g.query_error() == tccl.tcclSuccess
        assert g.last_launch()["engine"] == tccl.tcclEngineTmaReduce
        assert_ranks_equal([to_host(t) for t in parts], oracle.reduce_scatter(xs, dtype, op, nthreads=0),
                           f"TMA-reduce in-place RS {dtype} {op} P={p} slots={slots} cap={cap}")
    reset_config(g)


@pytest.mark.parametrize("slots,chunk", [(1, 8192), (2, 4096), (4, 0), (8, 2048), (3, 32768)])
@pytest.mark.parametrize("order", [tccl.tcclReduceAscending, tccl.tcclReduceArrival])
def test_tma_reduce_slot_shapes(groups, slots, chunk, order):
    """Every (slots, chunk) shape of the TMA-reduce engine, allreduce and
    reduce-scatter, P = 8, with ragged chunk counts per lane, bit-exact in the
    ascending order (int32 sums in the arrival order too)."""
    p, n = 8, 700_003
    g = groups(p)
    reset_config(g, engine=tccl.tcclEngineTmaReduce, reduce_slots=slots, max_chunk_bytes=chunk,
                 reduce_order=order)
    dtype = "f32" if order == tccl.tcclReduceAscending else "i32"
    xs = inputs(dtype, p, n)
    got = run_allreduce(g, xs, dtype, "sum", cap=11)
    info = g.last_launch()
    assert info["engine"] == tccl.tcclEngineTmaReduce and (slots == 0 or info["stages"] == slots)
    assert_ranks_equal(got, oracle.allreduce(xs, dtype, "sum", nthreads=0),
                       f"TMA-reduce AR slots={slots} chunk={chunk} order={order}")
    rc = 90_001
    xs = inputs(dtype, p, p * rc)
    sends = [to_device(x) for x in xs]
    parts = [torch.empty(rc, dtype=TORCH_OF[dtype], device="cuda") for _ in range(p)]
    g.reduce_scatter(sends, parts)
    torch.cuda.synchronize()
    assert g.query_error() == tccl.tcclSuccess
    assert_ranks_equal([to_host(t) for t in parts], oracle.reduce_scatter(xs, dtype, "sum", nthreads=0),
                       f"TMA-reduce RS slots={slots} chunk={chunk} order={order}")
    reset_config(g)


def test_arrival_order_leaves_other_engines_ascending(groups):
    """The order setting only changes the TMA-reduce engine: the bulk engine's
    fp32 sums stay bit-exact with it set."""
    p, n = 4, 1_000_003
    g = groups(p)
    reset_config(g, engine=tccl.tcclEngineBulk, reduce_order=tccl.tcclReduceArrival)
    xs = inputs("f32", p, n)
    assert_ranks_equal(run_allreduce(g, xs, "f32", "sum"), oracle.allreduce(xs, "f32", "sum", nthreads=0),
                       "bulk engine with the arrival order set")
    reset_config(g)


@pytest.mark.parametrize("dtype,op", [("bf16", "sum"), ("f32", "min"), ("f32", "max")])
def test_tma_reduce_engine_rejects_inexact_pairs(groups, dtype, op):
    g = groups(2)
    reset_config(g, engine=tccl.tcclEngineTmaReduce)
    a = torch.zeros(4096, dtype=TORCH_OF[dtype], device="cuda")
    b = torch.zeros_like(a)
    c = torch.zeros_like(a)
    d = torch.zeros_like(a)
    r = tccl.tcclAllReduce(g.handle, [a, b], [c, d], 4096, DT_CODE[dtype], tccl.OPS[op],
                           torch.cuda.current_stream().cuda_stream, 0)
    assert r == tccl.tcclInvalidUsage


def test_tma_reduce_engine_timeout_path(groups):
    p, n = 4, 1 << 20
    g = groups(p)
    reset_config(g, engine=tccl.tcclEngineTmaReduce)
    xs = inputs("f32", p, n)
    sends = [to_device(x) for x in xs]
    recvs = [torch.empty_like(s) for s in sends]
    assert tccl.tcclGroupInjectWaitTimeout(g.handle, True, 50.0) == tccl.tcclSuccess
    g.all_reduce(sends, recvs)
    assert g.query_error() == tccl.tcclDeviceTimeout
    assert tccl.tcclGroupInjectWaitTimeout(g.handle, False, 0.0) == tccl.tcclSuccess
    g.all_reduce(sends, recvs)
    torch.cuda.synchronize()
    assert g.query_error() == tccl.tcclSuccess
    assert_ranks_equal([to_host(r) for r in recvs], oracle.allreduce(xs, "f32", "sum", nthreads=0),
                       "TMA-reduce after timeout")


@pytest.mark.parametrize("cap", [1, 3, 8, 16, 32])
def test_cta_cap_results_and_sm_footprint(groups, cap):
    p, n = 8, 2_000_001
    g = groups(p)
    configure(g, "bulk")
    xs = inputs("bf16", p, n)
    exp = oracle.allreduce(xs, "bf16", "sum", nthreads=0)
    g.read_sm_record()
    g.record_sms(True)
    got = run_allreduce(g, xs, "bf16", "sum", cap=cap)
    sms = g.read_sm_record()
    g.record_sms(False)
    assert g.last_launch()["ctas"] == cap
    assert 1 <= sms <= cap
    assert_ranks_equal(got, exp, f"cap {cap}")


def test_sm_record_launch_by_launch(groups):
    """The SM record keeps one bitmap per launch: 70 capped launches (caps 1
    to 7 in turn) give 70 recorded launches, the first 64 reported one by
    one, each within its own cap; later launches share the last bitmap; the
    union covers them all. Reading clears the record."""
    p, n = 4, 200_000
    g = groups(p)
    configure(g, "bulk")
    xs = inputs("f32", p, n)
    sends = [to_device(x) for x in xs]
    recvs = [torch.empty_like(s) for s in sends]
    g.read_sm_record()
    g.record_sms(True)
    caps = [1 + i % 7 for i in range(70)]
    for cap in caps:
        g.all_reduce(sends, recvs, cta_cap=cap)
    per_launch, union = g.read_sm_record_launches()
    g.record_sms(False)
    assert len(per_launch) == 64
    assert all(1 <= m <= cap for m, cap in zip(per_launch[:63], caps[:63])), per_launch
    assert 1 <= per_launch[63] <= sum(caps[63:]) and max(per_launch) <= union <= sum(caps)
    assert g.read_sm_record_launches() == ([], 0)
    torch.cuda.synchronize()
    assert_ranks_equal([to_host(t) for t in recvs], oracle.allreduce(xs, "f32", "sum", nthreads=0),
                       "after 70 recorded launches")


def test_one_rank_copy_and_count_zero(groups):
    g = groups(1)
    configure(g, tccl.tcclEngineAuto)
    x = inputs("f32", 1, 1000)
    assert_ranks_equal(run_allreduce(g, x, "f32", "sum"), x, "P=1 copy")
    t = torch.zeros(4, device="cuda")
    assert tccl.tcclAllReduce(g.handle, [t], [t], 0, 0, 0, 0, 0) == tccl.tcclSuccess


def test_same_send_buffer_for_every_rank(groups):
    p, n = 8, 100_000
    g = groups(p)
    configure(g, "bulk")
    small = (np.arange(n) % 61 - 30).astype(np.float32)
    src = to_device(small)
    recvs = [torch.empty_like(src) for _ in range(p)]
    g.all_reduce([src] * p, recvs)
    torch.cuda.synchronize()
    for r in recvs:
        assert np.array_equal(to_host(r), (p * small).astype(np.float32))


# ------------------------------------------------------------------ reduce-scatter / all-gather
@pytest.mark.parametrize("engine", ["bulk", "warp", "vec"])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
def test_reduce_scatter_then_allgather(groups, engine, dtype):
    for p, rc in ((4, 100_003), (2, 9), (8, 4096), (3, 77_777)):
        g = groups(p)
        configure(g, engine)
        xs = inputs(dtype, p, p * rc)
        exp_rs = oracle.reduce_scatter(xs, dtype, "sum", nthreads=0)
        exp_ar = oracle.allreduce(xs, dtype, "sum", nthreads=0)
        sends = [to_device(x) for x in xs]
        parts = [Guarded(rc, dtype) for _ in range(p)]
        g.reduce_scatter(sends, [t.tensor for t in parts], op="sum")
        gathered = [Guarded(p * rc, dtype) for _ in range(p)]
        g.all_gather([t.tensor for t in parts], [t.tensor for t in gathered])
        torch.cuda.synchronize()
        assert g.query_error() == tccl.tcclSuccess
        assert all(t.guards_intact() for t in parts + gathered)
        assert_ranks_equal([t.host() for t in parts], exp_rs, f"RS {engine} {dtype} P={p}")
        assert_ranks_equal([t.host() for t in gathered], exp_ar, f"RS+AG {engine} {dtype} P={p}")


@pytest.mark.parametrize("engine", ["bulk", "warp", "vec"])
@pytest.mark.parametrize("op", ["min", "max"])
def test_reduce_scatter_min_max(groups, engine, op):
    p, rc = 8, 33_333
    g = groups(p)
    configure(g, engine)
    xs = inputs("f32", p, p * rc)
    exp = oracle.reduce_scatter(xs, "f32", op)
    sends = [to_device(x) for x in xs]
    parts = [torch.empty(rc, dtype=torch.float32, device="cuda") for _ in range(p)]
    g.reduce_scatter(sends, parts, op=op)
    torch.cuda.synchronize()
    assert_ranks_equal([to_host(t) for t in parts], exp, f"RS {op}")


@pytest.mark.parametrize("engine", ["bulk", "warp", "vec"])
@pytest.mark.parametrize("store", [tccl.tcclStoreBulk, tccl.tcclStoreVec])
def test_allgather_store_modes(groups, engine, store):
    p, sc = 8, 250_001
    g = groups(p)
    configure(g, engine, store=store)
    xs = inputs("bf16", p, sc)
    exp = oracle.allgather(xs)
    recvs = [Guarded(p * sc, "bf16") for _ in range(p)]
    g.all_gather([to_device(x) for x in xs], [t.tensor for t in recvs])
    torch.cuda.synchronize()
    assert all(t.guards_intact() for t in recvs)
    assert_ranks_equal([t.host() for t in recvs], exp, f"AG {engine} store {store}")


@pytest.mark.parametrize("engine", ["bulk", "warp", "vec"])
def test_reduce_scatter_and_allgather_in_place(groups, engine):
    p, n = 4, 10_007
    g = groups(p)
    configure(g, engine)
    xs = inputs("f32", p, p * n)
    exp_rs = oracle.reduce_scatter(xs, "f32", "sum")
    bufs = [to_device(x) for x in xs]
    # reduce-scatter in place: rank r's result lands in block r of its send buffer
    tccl_r = tccl.tcclReduceScatter(g.handle, bufs, [b[r * n:] for r, b in enumerate(bufs)], n,
                                    0, 0, torch.cuda.current_stream().cuda_stream, 0)
    assert tccl_r == tccl.tcclSuccess
    torch.cuda.synchronize()
    for r in range(p):
        assert same_bits(to_host(bufs[r][r * n:(r + 1) * n]), exp_rs[r])
    # all-gather in place: rank r's input is block r of its recv buffer
    exp_ag = oracle.allgather(exp_rs)
    r2 = tccl.tcclAllGather(g.handle, [b[r * n:] for r, b in enumerate(bufs)], bufs, n, 0,
                            torch.cuda.current_stream().cuda_stream, 0)
    assert r2 == tccl.tcclSuccess
    torch.cuda.synchronize()
    assert_ranks_equal([to_host(b) for b in bufs], exp_ag, "AG in place")


# ------------------------------------------------------------------ runtime behaviour
@pytest.mark.parametrize("order", ["blocked", "dynamic"])
@pytest.mark.parametrize("store", [tccl.tcclStoreBulk, tccl.tcclStoreVec, "per_rank"])
@pytest.mark.parametrize("coll", ["allreduce", "allgather"])
def test_bounded_wait_timeout_is_reported_and_context_survives(groups, order, store, coll):
    p, n = 4, 1 << 20
    g = groups(p)
    layout = tccl.tcclLayoutPerRank if store == "per_rank" else tccl.tcclLayoutShared
    reset_config(g, engine=tccl.tcclEngineBulk, store_mode=0 if store == "per_rank" else store,
                 chunk_order=ORDERS[order], stage_bytes=0, stages=0, stage_layout=layout)
    xs = inputs("f32", p, n)
    sends = [to_device(x) for x in xs]
    if coll == "allreduce":
        recvs = [torch.empty_like(s) for s in sends]
        run = lambda: g.all_reduce(sends, recvs)
        exp = oracle.allreduce(xs, "f32", "sum", nthreads=0)
    else:
        recvs = [torch.empty(p * n, dtype=torch.float32, device="cuda") for _ in range(p)]
        run = lambda: g.all_gather(sends, recvs)
        exp = oracle.allgather(xs)
    assert tccl.tcclGroupInjectWaitTimeout(g.handle, True, 50.0) == tccl.tcclSuccess
    run()
    assert g.query_error() == tccl.tcclDeviceTimeout
    assert g.query_error() == tccl.tcclSuccess  # cleared by the read
    assert tccl.tcclGroupInjectWaitTimeout(g.handle, False, 0.0) == tccl.tcclSuccess
    for _ in range(2):  # later launches (and the dynamic order's counter) are sound
        run()
        torch.cuda.synchronize()
        assert g.query_error() == tccl.tcclSuccess
        assert_ranks_equal([to_host(r) for r in recvs], exp, "after timeout")


def test_graph_capture_replay(groups):
    p, n = 8, 8192 * 8
    g = groups(p)
    configure(g, tccl.tcclEngineAuto)
    xs = inputs("bf16", p, n)
    sends = [to_device(x) for x in xs]
    recvs = [torch.zeros_like(s) for s in sends]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g.all_reduce(sends, recvs)  # plans the shape outside the capture
    torch.cuda.synchronize()
    for r in recvs:
        r.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        g.all_reduce(sends, recvs, stream=s.cuda_stream)
    for r in recvs:
        r.zero_()
    graph.replay()
    torch.cuda.synchronize()
    exp = oracle.allreduce(xs, "bf16", "sum")
    assert_ranks_equal([to_host(r) for r in recvs], exp, "graph replay")


def test_runs_on_a_side_stream(groups):
    p, n = 4, 500_000
    g = groups(p)
    configure(g, "bulk")
    xs = inputs("bf16", p, n)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        sends = [to_device(x) for x in xs]
        recvs = [torch.empty_like(t) for t in sends]
        g.all_reduce(sends, recvs)
    s.synchronize()
    exp = oracle.allreduce(xs, "bf16", "sum")
    assert_ranks_equal([to_host(r) for r in recvs], exp, "side stream")


def test_invalid_arguments_on_device(groups):
    g = groups(2)
    a = torch.zeros(64, device="cuda")
    b = torch.zeros(64, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    # overlapping recv buffers
    assert tccl.tcclAllReduce(g.handle, [a, b], [a[:32], a[16:48]], 32, 0, 0, st, 0) == \
        tccl.tcclInvalidArgument
    # bad op / dtype
    assert tccl.tcclAllReduce(g.handle, [a, b], [a, b], 64, 0, 5, st, 0) == tccl.tcclInvalidArgument
    assert tccl.tcclAllReduce(g.handle, [a, b], [a, b], 64, 9, 0, st, 0) == tccl.tcclInvalidArgument
    # misaligned for the element size
    assert tccl.tcclAllReduce(g.handle, [a.data_ptr() + 2, b], [a, b], 8, 0, 0, st, 0) == \
        tccl.tcclInvalidArgument


@pytest.mark.parametrize("p,n", [(4, 1 << 22), (8, 3 << 20), (2, (1 << 23) + 40)])
@pytest.mark.parametrize("in_place", [False, True])
def test_back_to_back_chain_reads_the_previous_result(groups, p, n, in_place):
    """Six uncapped allreduces on one stream, each reading what the one before
    it wrote (ping-pong between two buffer sets, or in place). Every launch
    starts early and prefetches its first chunks into L2 before it waits for
    the previous one, so this checks that no call reads its input stale.
    int32 sums wrap exactly: after k calls every rank holds P^(k-1) times the
    first call's sum."""
    g = groups(p)
    reset_config(g)  # Auto: the bulk engine at these sizes, dynamic order, early launch
    xs = inputs("i32", p, n, seed=21)
    a = [to_device(x) for x in xs]
    b = a if in_place else [torch.empty_like(t) for t in a]
    sets = [a, b]
    for k in range(6):
        src, dst = sets[k % 2], sets[(k + 1) % 2]
        assert tccl.tcclAllReduce(g.handle, src, dst, n, DT_CODE["i32"], tccl.tcclSum,
                                  torch.cuda.current_stream().cuda_stream, 0) == tccl.tcclSuccess
    assert g.last_launch()["engine"] == tccl.tcclEngineBulk
    torch.cuda.synchronize()
    assert g.query_error() == tccl.tcclSuccess
    total = np.zeros(n, dtype=np.int64)
    for x in xs:
        total += x.astype(np.int64)
    exp = ((total * p ** 5) % (1 << 32)).astype(np.uint64).astype(np.uint32).view(np.int32)
    for r in range(p):
        got = to_host(sets[6 % 2][r])
        mm = first_mismatch(got, exp)
        assert mm is None, f"P={p} in_place={in_place}: rank {r} first mismatch {mm}"


def test_reduce_order_setting_round_trip(groups):
    g = groups(2)
    reset_config(g, reduce_order=tccl.tcclReduceArrival)
    r, c = tccl.tcclGroupGetConfig(g.handle)
    assert r == tccl.tcclSuccess and c.reduce_order == tccl.tcclReduceArrival
    c.reduce_order = 2
    assert tccl.tcclGroupSetConfig(g.handle, c) == tccl.tcclInvalidArgument
    reset_config(g)
    r, c = tccl.tcclGroupGetConfig(g.handle)
    assert c.reduce_order == tccl.tcclReduceAscending


@pytest.mark.parametrize("tokens,cap", [(1, 0), (64, 0), (512, 16)])
def test_prepared_allreduce_call(tokens, cap):
    """Group.prepare_all_reduce marshals the arguments once; each call then
    issues the same allreduce, on the given stream, and a call on fresh
    inputs in the same buffers gives the oracle's result for them."""
    p, hidden = 8, 8192
    n = tokens * hidden
    with tccl.Group(p) as g:
        s = torch.cuda.Stream()
        sends = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
        recvs = [torch.empty_like(t) for t in sends]
        call = g.prepare_all_reduce(sends, recvs, cta_cap=cap, stream=s)
        for seed in (5, 6):
            xs = datagen.rank_buffers("normal_bf16", seed, p, n)
            for t, x in zip(sends, xs):
                t.copy_(to_device(x))
            torch.cuda.synchronize()
            for _ in range(3):
                call()
            s.synchronize()
            assert g.query_error() == tccl.tcclSuccess
            exp = oracle.allreduce(xs, "bf16", "sum", nthreads=0)
            for r in range(p):
                assert same_bits(to_host(recvs[r]), exp[r]), (tokens, cap, seed, r)


def test_prepared_reduce_scatter_and_all_gather_calls():
    """The prepared reduce-scatter and all-gather match the oracle, and
    chained (RS then AG) they equal the allreduce."""
    p, rc = 4, 123_456
    with tccl.Group(p) as g:
        xs = datagen.rank_buffers("normal_bf16", 7, p, p * rc)
        sends = [to_device(x) for x in xs]
        parts = [torch.empty(rc, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
        outs = [torch.empty(p * rc, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
        rs = g.prepare_reduce_scatter(sends, parts, cta_cap=8)
        ag = g.prepare_all_gather(parts, outs)
        for _ in range(2):
            rs()
            ag()
        torch.cuda.synchronize()
        assert g.query_error() == tccl.tcclSuccess
        exp_rs = oracle.reduce_scatter(xs, "bf16", "sum", nthreads=0)
        exp_ar = oracle.allreduce(xs, "bf16", "sum", nthreads=0)
        for r in range(p):
            assert same_bits(to_host(parts[r]), exp_rs[r])
            assert same_bits(to_host(outs[r]), exp_ar[r])
