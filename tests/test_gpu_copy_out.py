"""GPU parity for the copy-out engine (shard-in on SMs, shard-out on the
copy engines) against the CPU oracle, bit for bit, through the C ABI.

The allreduce is cut into segments; each segment's kernel stores the folded
result to rank 0 only and device-to-device copies carry it to ranks 1..P-1.
Small segment sizes make many segments (and a ragged last one) out of
test-sized buffers. The all-gather is copies only. Cases cover every dtype
and op, P = 2, 3 and 8, in-place and misaligned buffers, CTA caps and the SM
footprint, Auto's choice, stream order on either side of the call, CUDA graph
replay and the bounded-wait timeout path.
"""
import numpy as np
import pytest
import torch

import collective_communication_planner_gb300 as tccl
import datagen
import oracle
from gpu_util import DT_CODE, Guarded, first_mismatch, to_device, to_host

pytestmark = pytest.mark.gpu
KIND = {"f32": "uniform_f32", "bf16": "normal_bf16", "i32": "int32"}
CE = tccl.tcclEngineCopyOut


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
    c = tccl.tcclConfig_t()
    for k, v in kw.items():
        setattr(c, k, v)
    assert tccl.tcclGroupSetConfig(g.handle, c) == tccl.tcclSuccess


def check(got, exp, what):
    for r in range(len(exp)):
        mm = first_mismatch(got[r], exp[r])
        assert mm is None, f"{what}: rank {r} first mismatch at {mm[0]} ({mm[1]} elements)"


def allreduce(g, xs, dtype, op, cap=0, send_off=0, recv_off=0, in_place=False):
    p, n = len(xs), xs[0].size
    sends = [Guarded(n, dtype, send_off) for _ in range(p)]
    for s, x in zip(sends, xs):
        s.tensor.copy_(to_device(x))
    recvs = sends if in_place else [Guarded(n, dtype, recv_off) for _ in range(p)]
    r = tccl.tcclAllReduce(g.handle, [s.tensor for s in sends], [t.tensor for t in recvs], n,
                           DT_CODE[dtype], tccl.OPS[op], torch.cuda.current_stream().cuda_stream, cap)
    assert r == tccl.tcclSuccess, tccl.tcclGetErrorString(r)
    torch.cuda.synchronize()
    assert g.query_error() == tccl.tcclSuccess
    assert all(t.guards_intact() for t in recvs)
    return [t.host() for t in recvs]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "min", "max"])
@pytest.mark.parametrize("p", [2, 3, 8])
def test_allreduce_segments_dtypes_ops(groups, dtype, op, p):
    g = groups(p)
    reset_config(g, engine=CE, ce_segment_bytes=64 * 1024)
    n = 300_007
    xs = datagen.rank_buffers(KIND[dtype], 21, p, n)
    got = allreduce(g, xs, dtype, op, cap=7)
    info = g.last_launch()
    es = 2 if dtype == "bf16" else 4
    seg = 64 * 1024 // es
    assert info["engine"] == CE and info["ctas"] <= 7
    assert info["ce_segments"] == -(-n // seg) and info["ce_copies"] == info["ce_segments"] * (p - 1)
    check(got, oracle.allreduce(xs, dtype, op, nthreads=0), f"copy-out {dtype} {op} P={p}")


@pytest.mark.parametrize("offs", [(0, 0), (4, 4), (4, 8), (2, 6), (12, 0)])
@pytest.mark.parametrize("in_place", [False, True])
def test_allreduce_misaligned_and_in_place(groups, offs, in_place):
    p = 4
    g = groups(p)
    reset_config(g, engine=CE, ce_segment_bytes=32 * 1024)
    dtype = "bf16" if offs[0] % 4 else "f32"
    xs = datagen.rank_buffers(KIND[dtype], 22, p, 123_457)
    got = allreduce(g, xs, dtype, "sum", cap=16, send_off=offs[0], recv_off=offs[1], in_place=in_place)
    check(got, oracle.allreduce(xs, dtype, "sum", nthreads=0), f"offs {offs} in_place {in_place}")


@pytest.mark.parametrize("n", [1, 2, 7, 64, 4097, 65_536, 65_537])
def test_allreduce_small_counts_and_exact_segments(groups, n):
    p = 3
    g = groups(p)
    reset_config(g, engine=CE, ce_segment_bytes=4096)
    xs = datagen.rank_buffers("int32", 23, p, n)
    got = allreduce(g, xs, "i32", "sum", cap=4)
    assert g.last_launch()["ce_segments"] == min(64, -(-n // 1024)) or n > 64 * 1024
    check(got, oracle.allreduce(xs, "i32", "sum", nthreads=0), f"n={n}")


def test_segment_count_is_bounded(groups):
    p = 2
    g = groups(p)
    reset_config(g, engine=CE, ce_segment_bytes=4096)
    xs = datagen.rank_buffers("uniform_f32", 24, p, 3_000_001)
    got = allreduce(g, xs, "f32", "sum")
    assert 1 <= g.last_launch()["ce_segments"] <= 64
    check(got, oracle.allreduce(xs, "f32", "sum", nthreads=0), "64-segment bound")


@pytest.mark.parametrize("cap", [1, 5, 16])
def test_sm_footprint_stays_within_the_cap(groups, cap):
    p = 8
    g = groups(p)
    reset_config(g, engine=CE, ce_segment_bytes=1 << 20)
    xs = datagen.rank_buffers("normal_bf16", 25, p, 2_000_001)
    g.read_sm_record()
    g.record_sms(True)
    got = allreduce(g, xs, "bf16", "sum", cap=cap)
    per_launch, sms = g.read_sm_record_launches()
    g.record_sms(False)
    # every segment's kernel has `cap` CTAs and the segments run one after the
    # other on the stream, so at most `cap` SMs are busy at any time: each
    # launch's own record holds at most `cap` SMs, and the union over the
    # call's launches at most cap x segments
    info = g.last_launch()
    assert info["ctas"] == cap and 1 <= sms <= cap * info["ce_segments"]
    assert len(per_launch) == info["ce_segments"]
    assert all(1 <= n <= cap for n in per_launch), per_launch
    assert max(per_launch) <= sms
    check(got, oracle.allreduce(xs, "bf16", "sum", nthreads=0), f"cap {cap}")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("p", [2, 4, 8])
def test_allgather_copies_only(groups, dtype, p):
    g = groups(p)
    reset_config(g, engine=CE)
    rc = 50_001
    xs = datagen.rank_buffers(KIND[dtype], 26, p, rc)
    exp = [np.concatenate(xs)] * p
    sends = [to_device(x) for x in xs]
    outs = [Guarded(p * rc, dtype) for _ in range(p)]
    g.read_sm_record()
    g.record_sms(True)
    g.all_gather(sends, [t.tensor for t in outs])
    torch.cuda.synchronize()
    sms = g.read_sm_record()
    g.record_sms(False)
    info = g.last_launch()
    assert info["engine"] == CE and info["ctas"] == 0 and info["ce_copies"] == p * p and sms == 0
    assert all(t.guards_intact() for t in outs)
    check([t.host() for t in outs], exp, f"AG {dtype} P={p}")
    # in place: rank r's shard already sits in its own slot
    bufs = [to_device(np.zeros(p * rc, dtype=xs[0].dtype)) for _ in range(p)]
    es = bufs[0].element_size()
    for r in range(p):
        bufs[r][r * rc:(r + 1) * rc].copy_(sends[r])
    r = tccl.tcclAllGather(g.handle, [b[i * rc:(i + 1) * rc] for i, b in enumerate(bufs)], bufs, rc,
                           DT_CODE[dtype], torch.cuda.current_stream().cuda_stream, 0)
    assert r == tccl.tcclSuccess and es in (2, 4)
    torch.cuda.synchronize()
    assert g.last_launch()["ce_copies"] == p * (p - 1)
    check([to_host(b) for b in bufs], exp, f"AG in place {dtype} P={p}")


def reduce_scatter(g, xs, rc, dtype, op, cap=0, send_off=0, recv_off=0, in_place=False):
    p = len(xs)
    sends = [Guarded(p * rc, dtype, send_off) for _ in range(p)]
    for s_, x in zip(sends, xs):
        s_.tensor.copy_(to_device(x))
    if in_place:
        recv_t = [s_.tensor[r * rc:(r + 1) * rc] for r, s_ in enumerate(sends)]
        recvs = None
    else:
        recvs = [Guarded(rc, dtype, recv_off) for _ in range(p)]
        recv_t = [t.tensor for t in recvs]
    r = tccl.tcclReduceScatter(g.handle, [s_.tensor for s_ in sends], recv_t, rc, DT_CODE[dtype],
                               tccl.OPS[op], torch.cuda.current_stream().cuda_stream, cap)
    assert r == tccl.tcclSuccess, tccl.tcclGetErrorString(r)
    torch.cuda.synchronize()
    assert g.query_error() == tccl.tcclSuccess
    if recvs is not None:
        assert all(t.guards_intact() for t in recvs)
    assert all(s_.guards_intact() for s_ in sends)
    return [to_host(t) for t in recv_t]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "min", "max"])
@pytest.mark.parametrize("p", [2, 3, 4, 8])
def test_reduce_scatter_register_fold(groups, dtype, op, p):
    """Reduce-scatter on the copy-out engine: one launch of the register-load
    fold with one job per owner shard, no copies."""
    g = groups(p)
    reset_config(g, engine=CE)
    rc = 40_000  # shard bytes a multiple of 16 for every dtype
    xs = datagen.rank_buffers(KIND[dtype], 33, p, p * rc)
    got = reduce_scatter(g, xs, rc, dtype, op, cap=5)
    info = g.last_launch()
    assert info["engine"] == CE and info["threads"] == 1024 and info["ctas"] <= 5, info
    assert info["ce_copies"] == 0
    check(got, oracle.reduce_scatter(xs, dtype, op, nthreads=0), f"RS {dtype} {op} P={p}")


@pytest.mark.parametrize("case", ["in_place", "offset_co_aligned", "misaligned", "ragged_shard"])
def test_reduce_scatter_layouts(groups, case):
    """In place and co-aligned offsets (element-wise edges) take the register
    fold; misaligned buffers and shards that are not a multiple of 16 bytes
    take the bulk engine. All exact."""
    p = 4
    g = groups(p)
    reset_config(g, engine=CE)
    rc = 12_347 if case == "ragged_shard" else 12_352
    xs = datagen.rank_buffers("normal_bf16", 34, p, p * rc)
    kw = {"in_place": dict(in_place=True), "offset_co_aligned": dict(send_off=6, recv_off=6),
          "misaligned": dict(send_off=2, recv_off=0), "ragged_shard": {}}[case]
    got = reduce_scatter(g, xs, rc, "bf16", "sum", cap=8, **kw)
    fold = case in ("in_place", "offset_co_aligned")
    assert g.last_launch()["engine"] == (CE if fold else tccl.tcclEngineBulk), (case, g.last_launch())
    check(got, oracle.reduce_scatter(xs, "bf16", "sum", nthreads=0), f"RS {case}")


@pytest.mark.parametrize("p", [4, 8])
def test_reduce_scatter_auto_choice(groups, p):
    """Auto: the register fold under any cap, and uncapped for up to four
    ranks; the bulk engine uncapped for more ranks and below 4 MiB."""
    g = groups(p)
    reset_config(g)
    rc = (1 << 23) // p  # 8 Mi bf16 per rank send buffer: 16 MiB
    sends = [torch.ones(p * rc, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    recvs = [torch.empty(rc, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    g.reduce_scatter(sends, recvs, cta_cap=16)
    assert g.last_launch()["engine"] == CE
    g.reduce_scatter(sends, recvs)
    assert g.last_launch()["engine"] == (CE if p <= 4 else tccl.tcclEngineBulk)
    small = rc // 8  # 2 MiB per rank send buffer
    g.reduce_scatter([s[:p * small] for s in sends], [r[:small] for r in recvs], cta_cap=16)
    assert g.last_launch()["engine"] == tccl.tcclEngineBulk
    torch.cuda.synchronize()
    assert all(bool((r == p).all()) for r in recvs)


@pytest.mark.parametrize("p", [16, 33, 64])
def test_many_ranks(groups, p):
    """Rank counts with no compiled-in specialisation: the fold takes the
    ranks in batches of 8 (allreduce and reduce-scatter), exact either way."""
    g = groups(p)
    reset_config(g, engine=CE, ce_segment_bytes=16 * 1024)
    xs = datagen.rank_buffers("normal_bf16", 35, p, 20_003)
    got = allreduce(g, xs, "bf16", "sum", cap=6)
    info = g.last_launch()
    assert info["engine"] == CE and info["threads"] == 1024 and info["ce_copies"] == info["ce_segments"] * (p - 1)
    check(got, oracle.allreduce(xs, "bf16", "sum", nthreads=0), f"AR P={p}")
    rc = 1024
    ys = datagen.rank_buffers("int32", 36, p, p * rc)
    got = reduce_scatter(g, ys, rc, "i32", "max", cap=3)
    assert g.last_launch()["engine"] == CE
    check(got, oracle.reduce_scatter(ys, "i32", "max", nthreads=0), f"RS P={p}")


def test_one_rank_falls_back_to_the_bulk_engine(groups):
    g = groups(1)
    reset_config(g, engine=CE)
    xs = datagen.rank_buffers("uniform_f32", 28, 1, 10_000)
    check(allreduce(g, xs, "f32", "sum"), xs, "P=1")
    assert g.last_launch()["engine"] == tccl.tcclEngineBulk


def test_auto_picks_copy_out_for_large_capped_calls(groups):
    p = 4
    g = groups(p)
    reset_config(g)
    n = 4 * 1024 * 1024  # 8 MiB of bf16 per rank
    sends = [torch.ones(n, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    recvs = [torch.empty_like(s) for s in sends]
    picks = {}
    edge = torch.cuda.get_device_properties(0).multi_processor_count * 5 // 12  # P = 4
    for cap in (0, 8, 16, edge, edge + 1, 2 * edge):
        g.all_reduce(sends, recvs, cta_cap=cap)
        picks[cap] = g.last_launch()["engine"]
    assert picks == {0: 1, 8: CE, 16: CE, edge: CE, edge + 1: 1, 2 * edge: 1}, picks
    small = [s[:1 << 20] for s in sends]  # 2 MiB per rank: below the threshold
    g.all_reduce(small, [r[:1 << 20] for r in recvs], cta_cap=8)
    assert g.last_launch()["engine"] == tccl.tcclEngineBulk
    reset_config(g, ce_auto_max_cap=-1)
    g.all_reduce(sends, recvs, cta_cap=8)
    assert g.last_launch()["engine"] == tccl.tcclEngineBulk
    reset_config(g, ce_auto_max_cap=2 * edge)
    g.all_reduce(sends, recvs, cta_cap=2 * edge)
    assert g.last_launch()["engine"] == CE
    torch.cuda.synchronize()
    assert all(bool((r == 4).all()) for r in recvs)
    reset_config(g)


def test_stream_order_on_both_sides(groups):
    """Inputs written by a kernel queued just before the call, and results
    read by a kernel queued just after it, on a side stream, with no host
    synchronisation in between: the copy streams join in both directions."""
    p, n = 8, 3_000_001
    g = groups(p)
    reset_config(g, engine=CE, ce_segment_bytes=1 << 20)
    xs = datagen.rank_buffers("uniform_f32", 29, p, n)
    host = [to_device(x) for x in xs]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        sends = [torch.zeros_like(h) for h in host]
        recvs = [torch.zeros_like(h) for h in host]
        for _ in range(3):
            for d, h in zip(sends, host):
                d.copy_(h * 1.0)  # a kernel on s
            g.all_reduce(sends, recvs, cta_cap=8, stream=s.cuda_stream)
            outs = [r.clone() for r in recvs]  # kernels on s
            for r in recvs:
                r.fill_(0.0)
    s.synchronize()
    check([to_host(o) for o in outs], oracle.allreduce(xs, "f32", "sum", nthreads=0), "stream order")


def test_graph_capture_replay(groups):
    p, n = 4, 1_000_003
    g = groups(p)
    reset_config(g, engine=CE, ce_segment_bytes=256 * 1024)
    xs = datagen.rank_buffers("normal_bf16", 30, p, n)
    sends = [to_device(x) for x in xs]
    recvs = [torch.zeros_like(t) for t in sends]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g.all_reduce(sends, recvs, cta_cap=16, stream=s.cuda_stream)  # plans outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        g.all_reduce(sends, recvs, cta_cap=16, stream=s.cuda_stream)
    for r in recvs:
        r.zero_()
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    check([to_host(r) for r in recvs], oracle.allreduce(xs, "bf16", "sum"), "graph replay")


@pytest.mark.parametrize("what", ["allreduce_uncapped", "reduce_scatter_capped",
                                  "reduce_scatter_uncapped", "allgather"])
def test_graph_capture_of_every_copy_out_path(groups, what):
    """Each copy-out path captured into a CUDA graph and replayed: the
    uncapped allreduce (early-launched segment kernels between events), the
    register-fold reduce-scatter with and without a cap, and the copy-only
    all-gather."""
    p = 4
    g = groups(p)
    reset_config(g, engine=CE, ce_segment_bytes=128 * 1024)
    s = torch.cuda.Stream()
    if what == "allreduce_uncapped":
        n = 400_000
        xs = datagen.rank_buffers("normal_bf16", 37, p, n)
        ins = [to_device(x) for x in xs]
        outs = [torch.zeros_like(t) for t in ins]
        call = lambda: g.all_reduce(ins, outs, stream=s.cuda_stream)
        exp = oracle.allreduce(xs, "bf16", "sum", nthreads=0)
    elif what.startswith("reduce_scatter"):
        rc = 100_000
        xs = datagen.rank_buffers("uniform_f32", 38, p, p * rc)
        ins = [to_device(x) for x in xs]
        outs = [torch.zeros(rc, dtype=torch.float32, device="cuda") for _ in range(p)]
        cap = 8 if what == "reduce_scatter_capped" else 0
        call = lambda: g.reduce_scatter(ins, outs, cta_cap=cap, stream=s.cuda_stream)
        exp = oracle.reduce_scatter(xs, "f32", "sum", nthreads=0)
    else:
        sc = 150_000
        xs = datagen.rank_buffers("int32", 39, p, sc)
        ins = [to_device(x) for x in xs]
        outs = [torch.zeros(p * sc, dtype=torch.int32, device="cuda") for _ in range(p)]
        call = lambda: g.all_gather(ins, outs, stream=s.cuda_stream)
        exp = [np.concatenate(xs)] * p
    with torch.cuda.stream(s):
        call()  # first call outside the capture: plans, copy streams, events
    torch.cuda.synchronize()
    assert g.last_launch()["engine"] == CE, g.last_launch()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        call()
    for o in outs:
        o.zero_()
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert g.query_error() == tccl.tcclSuccess
    check([to_host(o) for o in outs], exp, f"graph {what}")


def test_timeout_is_reported_and_the_next_call_is_right(groups):
    """Send and receive buffers that are not co-aligned take the TMA shard-in
    (the register-load fold has no waits to run out); its injected wait runs
    out, the status says so, and the next call is right."""
    p, n = 4, 500_000
    g = groups(p)
    reset_config(g, engine=CE, ce_segment_bytes=256 * 1024, wait_timeout_ms=1000.0)
    xs = datagen.rank_buffers("uniform_f32", 31, p, n)
    sends = [Guarded(n, "f32", 4) for _ in range(p)]
    for s_, x in zip(sends, xs):
        s_.tensor.copy_(to_device(x))
    recvs = [Guarded(n, "f32", 0) for _ in range(p)]
    st = torch.cuda.current_stream().cuda_stream

    def call():
        return tccl.tcclAllReduce(g.handle, [t.tensor for t in sends], [t.tensor for t in recvs], n,
                                  DT_CODE["f32"], tccl.tcclSum, st, 4)

    assert tccl.tcclGroupInjectWaitTimeout(g.handle, 1, 20.0) == tccl.tcclSuccess
    assert call() == tccl.tcclSuccess
    torch.cuda.synchronize()
    assert g.query_error() == tccl.tcclDeviceTimeout
    assert g.last_launch()["threads"] == 544
    assert tccl.tcclGroupInjectWaitTimeout(g.handle, 0, 0.0) == tccl.tcclSuccess
    assert call() == tccl.tcclSuccess
    torch.cuda.synchronize()
    assert g.query_error() == tccl.tcclSuccess
    assert all(t.guards_intact() for t in recvs)
    check([t.host() for t in recvs], oracle.allreduce(xs, "f32", "sum", nthreads=0), "after timeout")


@pytest.mark.parametrize("offs,fast", [((0, 0), True), ((4, 4), True), ((6, 6), True),
                                       ((4, 0), False), ((0, 2), False)])
@pytest.mark.parametrize("p", [2, 4, 8])
def test_shard_in_kernel_choice(groups, offs, fast, p):
    """Co-aligned buffers (same address mod 16, any offset) take the register
    fold (1024 threads per CTA, unaligned edges element-wise); the rest take
    the TMA pipeline (544 threads). Both are exact."""
    g = groups(p)
    reset_config(g, engine=CE, ce_segment_bytes=64 * 1024)
    xs = datagen.rank_buffers("normal_bf16", 32, p, 200_003)
    got = allreduce(g, xs, "bf16", "sum", cap=6, send_off=offs[0], recv_off=offs[1])
    info = g.last_launch()
    assert info["threads"] == (1024 if fast else 544) and info["ctas"] <= 6, info
    check(got, oracle.allreduce(xs, "bf16", "sum", nthreads=0), f"offs {offs} P={p}")


@pytest.mark.parametrize("layout,warps", [(0, 0), (2, 0), (2, 8)])
@pytest.mark.parametrize("dtype,op,p", [("bf16", "sum", 8), ("f32", "max", 3), ("i32", "sum", 4)])
def test_tma_fold_when_asked(groups, layout, warps, dtype, op, p):
    """ce_fold = 2 puts the segments of co-aligned buffers on the TMA pipeline
    (shared or per-rank stage layout) instead of the register fold; the
    result is the same bits."""
    g = groups(p)
    reset_config(g, engine=CE, ce_segment_bytes=256 * 1024, ce_fold=2, stage_layout=layout,
                 consumer_warps=warps)
    xs = datagen.rank_buffers(KIND[dtype], 33, p, 500_009)
    got = allreduce(g, xs, dtype, op, cap=5)
    info = g.last_launch()
    assert info["engine"] == CE and info["threads"] != 1024 and info["ctas"] <= 5, info
    assert info["stage_layout"] == (2 if layout == 2 else 1), info
    check(got, oracle.allreduce(xs, dtype, op, nthreads=0), f"TMA fold layout {layout} P={p}")


SPECIAL_BF16 = np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x007F, 0x807F, 0x0080, 0x8080,
                         0x0040, 0x8040, 0x3F80, 0xBF80, 0x3F81, 0x4000, 0xC000, 0x0100],
                        dtype=np.uint16)


@pytest.mark.parametrize("p", [2, 3, 4, 8])
def test_register_fold_bf16_special_values(groups, p):
    """bf16 sums on the register fold with subnormals, signed zeros and
    values that cancel exactly planted among normal data: every output element
    equals the oracle's (fp32 accumulation without flushing, one rounding)."""
    g = groups(p)
    reset_config(g, engine=CE, ce_segment_bytes=256 * 1024)
    n = 300_007
    xs = datagen.rank_buffers("normal_bf16", 34, p, n)
    rng = np.random.default_rng(34)
    for r in range(p):
        pick = rng.random(n) < 0.5
        xs[r] = xs[r].copy()
        xs[r][pick] = SPECIAL_BF16[rng.integers(0, SPECIAL_BF16.size, int(pick.sum()))]
    got = allreduce(g, xs, "bf16", "sum", cap=9)
    assert g.last_launch()["threads"] == 1024  # the register fold
    check(got, oracle.allreduce(xs, "bf16", "sum", nthreads=0), f"special bf16 P={p}")


@pytest.mark.parametrize("mid,tail", [(0, 0), (1, 4), (2, 2), (3, 1), (4, 4)])
@pytest.mark.parametrize("cap", [5, 16, 40])
def test_copy_stream_splits(groups, mid, tail, cap):
    """Any split of the copy streams between the overlapped segments and the
    last one (0 = the default: by the cap, and ce_streams) gives the same bits."""
    p = 8
    g = groups(p)
    reset_config(g, engine=CE, ce_segment_bytes=128 * 1024, ce_ar_streams=mid, ce_tail_streams=tail)
    xs = datagen.rank_buffers("normal_bf16", 35, p, 400_009)
    got = allreduce(g, xs, "bf16", "sum", cap=cap)
    info = g.last_launch()
    assert info["engine"] == CE and info["ce_segments"] >= 4 and info["ce_copies"] == 7 * info["ce_segments"]
    check(got, oracle.allreduce(xs, "bf16", "sum", nthreads=0), f"streams {mid}/{tail} cap {cap}")


TMA_REDUCE_PAIRS = [("f32", "sum"), ("i32", "sum"), ("i32", "min"), ("i32", "max"),
                    ("bf16", "min"), ("bf16", "max")]


@pytest.mark.parametrize("dtype,op", TMA_REDUCE_PAIRS)
@pytest.mark.parametrize("p,cap,offs,in_place", [(2, 0, 0, False), (3, 7, 4, False), (8, 16, 0, False),
                                                 (8, 0, 0, True), (8, 5, 8, False)])
def test_tma_reduce_fold(groups, dtype, op, p, cap, offs, in_place):
    """ce_fold = 3: each segment is bulk-reduced into the anchor by the
    TMA-reduce engine (rank 0 stored, ranks 1..P-1 reduced in order) and the
    copy engines carry it to the other ranks; the same bits as the oracle,
    capped or not, misaligned or in place."""
    g = groups(p)
    reset_config(g, engine=CE, ce_segment_bytes=256 * 1024, ce_fold=3)
    xs = datagen.rank_buffers(KIND[dtype], 36, p, 300_007)
    got = allreduce(g, xs, dtype, op, cap=cap, send_off=offs, recv_off=offs, in_place=in_place)
    info = g.last_launch()
    assert info["engine"] == CE and info["threads"] != 1024 and info["ce_segments"] > 1, info
    check(got, oracle.allreduce(xs, dtype, op, nthreads=0), f"TMA-reduce fold {dtype} {op} P={p}")


def test_tma_reduce_fold_falls_back_for_other_pairs(groups):
    """A pair the copy hardware cannot reduce exactly (bf16 sum) takes the
    register fold under ce_fold = 3, with the same bits."""
    g = groups(8)
    reset_config(g, engine=CE, ce_segment_bytes=256 * 1024, ce_fold=3)
    xs = datagen.rank_buffers("normal_bf16", 37, 8, 300_007)
    got = allreduce(g, xs, "bf16", "sum", cap=16)
    assert g.last_launch()["threads"] == 1024
    check(got, oracle.allreduce(xs, "bf16", "sum", nthreads=0), "bf16 sum under ce_fold 3")


@pytest.mark.parametrize("p", [2, 3, 4, 5, 6, 7, 8, 12, 16])
@pytest.mark.parametrize("dtype,op", [("bf16", "sum"), ("f32", "sum"), ("i32", "max"), ("bf16", "min")])
@pytest.mark.parametrize("case", ["aligned", "odd_vectors", "head_32", "head_16"])
def test_wide_fold_layouts(groups, p, dtype, op, case):
    """The register fold's 256-bit loads (P = 2 to 8, 16, or a multiple of 4
    read at run time, here 12; every buffer 32-byte
    aligned past the head): an even and an odd count of 16-byte vectors (the
    odd last one folded on its own), and a head that leaves the body 32-byte
    aligned; a head that leaves it only 16-byte aligned takes the 128-bit
    loads. Both bit-exact against the oracle."""
    g = groups(p)
    es = 2 if dtype == "bf16" else 4
    reset_config(g, engine=CE, ce_segment_bytes=256 * 1024)
    n = {"aligned": 200_000 * 16 // es, "odd_vectors": (100_001 * 16 + 6) // es}.get(case, 150_001)
    # head_32: start 18 bytes past a 32-byte boundary (bf16) or 20 (4-byte
    # types), so the 14- / 12-byte head ends on one; head_16: 2 or 4 bytes
    # past it, so the head ends 16 bytes short of one
    off = {"head_32": 18 if es == 2 else 20, "head_16": 2 if es == 2 else 4}.get(case, 0)
    xs = datagen.rank_buffers(KIND[dtype], 41, p, n)
    got = allreduce(g, xs, dtype, op, cap=16, send_off=off, recv_off=off)
    info = g.last_launch()
    assert info["engine"] == CE and info["ctas"] <= 16, info
    want_wide = info["ce_segments"] if case != "head_16" else 0
    assert info["ce_wide_folds"] == want_wide, (case, info)
    check(got, oracle.allreduce(xs, dtype, op, nthreads=0), f"wide fold {case} {dtype} {op} P={p}")


@pytest.mark.parametrize("p", [2, 3, 4, 5, 8, 9, 12, 16])
@pytest.mark.parametrize("rc", [40_000, 40_008])
def test_wide_fold_reduce_scatter(groups, p, rc):
    """Reduce-scatter on the register fold: shards of a multiple of 32 bytes
    keep every job 32-byte aligned and take the 256-bit loads; shards of an
    odd multiple of 16 bytes leave every other job 16 bytes off and take the
    128-bit loads, as P = 9 does always. All exact."""
    g = groups(p)
    reset_config(g, engine=CE)
    xs = datagen.rank_buffers("normal_bf16", 42, p, p * rc)
    got = reduce_scatter(g, xs, rc, "bf16", "sum", cap=8)
    info = g.last_launch()
    assert info["engine"] == CE and info["ce_copies"] == 0, info
    assert info["ce_wide_folds"] == (1 if rc * 2 % 32 == 0 and p != 9 else 0), info
    check(got, oracle.reduce_scatter(xs, "bf16", "sum", nthreads=0), f"RS wide rc={rc} P={p}")
