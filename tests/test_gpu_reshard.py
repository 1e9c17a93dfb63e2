"""GPU parity for tcclReshard against the reshard oracle, bit for bit:
the article's example A, many (mesh, placement) pairs, three dtypes, 2-D and
3-D tensors, misaligned buffers (element-wise path), CTA caps, and a
weight-sized reshard."""
import numpy as np
import pytest
import torch

import collective_communication_planner_gb300 as tccl
import datagen
from gpu_util import Guarded, first_mismatch, to_device, to_host
from oracle import reshard as rs

pytestmark = pytest.mark.gpu
R = tccl.TCCL_REPLICATE
KIND = {"f32": "uniform_f32", "bf16": "normal_bf16", "i32": "int32"}


def global_tensor(dtype, shape, seed=5):
    n = int(np.prod(shape))
    return datagen.rank_buffers(KIND[dtype], seed, 1, n)[0].reshape(shape)


def src_blocks(glob, dims, place):
    out = []
    for m in range(rs.nranks(dims)):
        box = rs.local_box(glob.shape, dims, place, m)
        out.append(np.ascontiguousarray(glob[tuple(slice(lo, hi) for lo, hi in box)]).ravel())
    return out


ENGINES = {"auto": tccl.tcclEngineAuto, "bulk": tccl.tcclEngineBulk, "warp": tccl.tcclEngineWarp}


def edges_aligned(shape, layout, es):
    """Every block of the layout starts and ends on a 16-byte boundary of its
    rows (so every piece, offset and pitch of a reshard between two such
    layouts is whole 16-byte vectors)."""
    return all(lo * es % 16 == 0 and hi * es % 16 == 0
               for m in range(rs.nranks(layout[0]))
               for lo, hi in [rs.local_box(shape, layout[0], layout[1], m)[-1]])


def set_engine(g, engine):
    c = tccl.tcclConfig_t()
    c.engine = ENGINES[engine]
    assert tccl.tcclGroupSetConfig(g.handle, c) == tccl.tcclSuccess


def run(g, glob, src, dst, dtype, cap=0, mis=0, engine="auto"):
    set_engine(g, engine)
    shape = glob.shape
    sb = src_blocks(glob, *src)
    exp = rs.reshard(sb, src[0], src[1], dst[0], dst[1], shape)
    sends = []
    for b in sb:
        t = Guarded(b.size, dtype, mis)
        t.tensor.copy_(to_device(b))
        sends.append(t)
    recvs = [Guarded(e.size, dtype, mis) for e in exp]
    g.reshard([t.tensor for t in sends], tccl.make_layout(src[0], src[1], 0),
              [t.tensor for t in recvs], tccl.make_layout(dst[0], dst[1], rs.nranks(src[0])),
              shape, cta_cap=cap)
    torch.cuda.synchronize()
    assert g.query_error() == tccl.tcclSuccess
    # asked for, the bulk ring runs every 16-byte co-aligned plan; a plan
    # with an element-wise piece, or a request for warps, runs on warps
    es = np.dtype(exp[0].dtype).itemsize
    aligned = mis % 16 == 0 and edges_aligned(shape, src, es) and edges_aligned(shape, dst, es)
    misaligned = mis % 16 != 0 or any(e.size * es % 16 for e in exp)
    info = g.last_launch()
    if engine == "warp" or misaligned:
        assert info["engine"] == tccl.tcclEngineWarp, info
    if engine == "bulk" and aligned:
        assert info["engine"] == tccl.tcclEngineBulk and info["threads"] == 64, info
    for m, (t, e) in enumerate(zip(recvs, exp)):
        assert t.guards_intact()
        mm = first_mismatch(t.host(), e)
        assert mm is None, f"{src} -> {dst} {dtype} ({engine}): rank {m} first mismatch {mm}"
    return info


@pytest.fixture(scope="module")
def group():
    g = tccl.Group(64)
    yield g
    g.close()


def test_article_example_a(group, golden_dir):
    glob = global_tensor("bf16", (4, 8))
    run(group, glob, ((1, 4), (R, 0)), ((2, 2), (R, 0)), "bf16")


@pytest.mark.parametrize("shape", [(4, 8), (4096, 1024)])
def test_article_example_b(group, shape):
    """Example B, both pipeline stages: trainer mesh [2] Shard(0) -> generator
    mesh [1] Replicate(), the generator gathering each stage's whole weight."""
    for stage in range(2):
        glob = global_tensor("bf16", shape, seed=40 + stage)
        run(group, glob, ((2,), (0,)), ((1,), (R,)), "bf16")


LAYOUTS = [((4,), (0,)), ((4,), (R,)), ((2, 2), (R, 0)), ((2, 2), (0, R)), ((2, 2), (1, R)),
           ((1, 4), (R, 1)), ((2, 4), (R, 0)), ((8,), (1,)), ((2, 1, 2), (R, R, 1))]


@pytest.mark.parametrize("engine", ["bulk", "warp"])
@pytest.mark.parametrize("src", LAYOUTS)
@pytest.mark.parametrize("dst", LAYOUTS[::2])
def test_layout_pairs(group, src, dst, engine):
    glob = global_tensor("f32", (64, 96))
    info = run(group, glob, src, dst, "f32", engine=engine)
    if engine == "bulk":
        assert info["engine"] == tccl.tcclEngineBulk, info


@pytest.mark.parametrize("src,dst,bulk", [
    (((2,), (0,)), ((8,), (R,)), True),            # 8 replicas, whole rows
    (((8,), (0,)), ((4, 2), (R, 1)), True),        # 4 replicas, 8 KiB row pieces
    (((1, 4), (R, 0)), ((2, 2), (R, 0)), False),   # 2 replicas
    (((8,), (1,)), ((8,), (0,)), False),           # 1 replica, 2 KiB row pieces
    (((8,), (1,)), ((4,), (R,)), False),           # 4 replicas, but 2 KiB row pieces
    (((8,), (0,)), ((16,), (R,)), True)])          # 16 replicas, whole blocks
def test_auto_engine_choice(group, src, dst, bulk):
    """Auto takes the bulk ring for co-aligned plans that write every block
    to three or more replicas on average in row pieces of 4 KiB or more, and
    warp copies otherwise."""
    glob = global_tensor("bf16", (512, 8192), seed=13)
    info = run(group, glob, src, dst, "bf16", engine="auto")
    assert (info["engine"] == tccl.tcclEngineBulk) == bulk, info


@pytest.mark.parametrize("engine", ["bulk", "warp"])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("mis", [0, 4])
@pytest.mark.parametrize("cap", [0, 3])
def test_dtypes_alignment_caps(group, dtype, mis, cap, engine):
    glob = global_tensor(dtype, (256, 1000))
    run(group, glob, ((8,), (1,)), ((2, 2), (R, 0)), dtype, cap=cap, mis=mis, engine=engine)
    run(group, glob, ((4,), (0,)), ((2, 4), (R, 1)), dtype, cap=cap, mis=mis, engine=engine)
    if cap:
        assert group.last_launch()["ctas"] <= cap


@pytest.mark.parametrize("shape", [(3, 40000), (40000, 24), (7, 8192 + 16), (1, 16384 * 3 + 16)])
def test_bulk_unit_shapes(group, shape):
    """The bulk ring's work units: rows longer than a stage cut into 16 KiB
    segments with a ragged last one, rows shorter than a stage packed many
    to a stage with a ragged last stage, and a single row."""
    glob = global_tensor("bf16", shape, seed=11)
    ran = 0
    for src, dst in ((((1,), (R,)), ((2, 2), (R, 1))), (((2,), (0,)), ((4,), (R,))),
                     (((1,), (R,)), ((3,), (R,)))):
        if any(d != R and shape[d] % n for dims, place in (src, dst) for n, d in zip(dims, place)):
            continue
        info = run(group, glob, src, dst, "bf16", engine="bulk")
        if edges_aligned(shape, src, 2) and edges_aligned(shape, dst, 2):
            assert info["engine"] == tccl.tcclEngineBulk, info
            ran += 1
    assert ran >= 1


def test_bulk_timeout_path(group):
    """A bulk-ring wait that runs out (the test hook holds CTA 0's first stage
    on a barrier nothing completes) is reported as a device timeout, and the
    next reshard on the same group is exact."""
    glob = global_tensor("bf16", (1024, 2048), seed=12)
    set_engine(group, "bulk")  # a 2-replica plan: on the ring only when asked for
    src, dst = ((4,), (0,)), ((2, 2), (R, 1))
    sb = src_blocks(glob, *src)
    exp = rs.reshard(sb, src[0], src[1], dst[0], dst[1], glob.shape)
    sends = [to_device(b) for b in sb]
    recvs = [torch.empty(e.size, dtype=torch.bfloat16, device="cuda") for e in exp]
    args = (sends, tccl.make_layout(src[0], src[1], 0), recvs, tccl.make_layout(dst[0], dst[1], 4), glob.shape)
    assert tccl.tcclGroupInjectWaitTimeout(group.handle, True, 50.0) == tccl.tcclSuccess
    try:
        group.reshard(*args)
        assert group.query_error() == tccl.tcclDeviceTimeout
    finally:
        assert tccl.tcclGroupInjectWaitTimeout(group.handle, False, 0.0) == tccl.tcclSuccess
    group.reshard(*args)
    torch.cuda.synchronize()
    assert group.query_error() == tccl.tcclSuccess
    assert group.last_launch()["engine"] == tccl.tcclEngineBulk
    for t, e in zip(recvs, exp):
        assert first_mismatch(to_host(t), e) is None


def test_three_dimensional(group):
    glob = global_tensor("bf16", (8, 16, 64))
    run(group, glob, ((2, 2), (R, 2)), ((4,), (1,)), "bf16")
    run(group, glob, ((4,), (0,)), ((2, 4), (R, 2)), "bf16")


def test_weight_sized_reshard(group):
    # an 8192 x 8192 bf16 weight: TP8 (row shards) -> TP2 x DP4 (column shards, replicated)
    glob = global_tensor("bf16", (8192, 8192), seed=9)
    run(group, glob, ((8,), (0,)), ((4, 2), (R, 1)), "bf16")


def random_layout(rng, ndim):
    naxes = int(rng.integers(1, 4))
    dims = (64,)
    while int(np.prod(dims)) > 32:  # both meshes fit the 64-rank group
        dims = tuple(int(rng.integers(1, 5)) for _ in range(naxes))
    place = [R] * naxes
    if rng.random() < 0.8:
        place[int(rng.integers(0, naxes))] = int(rng.integers(0, ndim))
    return dims, tuple(place)


@pytest.mark.parametrize("engine", ["bulk", "warp"])
@pytest.mark.parametrize("case", range(40))
def test_random_reshard(group, case, engine):
    """Seeded random layout pairs: meshes of one to three axes (each of size
    one to four), Replicate or one Shard per layout, tensors of one to three
    dimensions whose sharded extents the mesh axes divide, three dtypes,
    misaligned buffers and caps."""
    rng = np.random.default_rng(9000 + case)
    ndim = int(rng.integers(1, 4))
    src = random_layout(rng, ndim)
    dst = random_layout(rng, ndim)
    shape = [int(rng.integers(1, 40 if ndim > 1 else 400)) for _ in range(ndim)]
    for dims, place in (src, dst):
        for a, d in enumerate(place):
            if d != R:
                shape[d] = dims[a] * max(1, shape[d] // dims[a])
    # both meshes' axes must divide the same extent: take a common multiple
    for d in range(ndim):
        m = 1
        for dims, place in (src, dst):
            for a, dd in enumerate(place):
                if dd == d:
                    m = int(np.lcm(m, dims[a]))
        shape[d] = m * max(1, shape[d] // m)
    dtype = str(rng.choice(["f32", "bf16", "i32"]))
    es = 2 if dtype == "bf16" else 4
    mis = int(rng.integers(0, 16 // es)) * es if rng.random() < 0.3 else 0
    cap = int(rng.choice([0, 0, 1, 5, 40]))
    glob = global_tensor(dtype, tuple(shape), seed=case)
    run(group, glob, src, dst, dtype, cap=cap, mis=mis, engine=engine)


@pytest.mark.parametrize("engine", ["bulk", "warp"])
def test_graph_capture_replay(group, engine):
    """Reshards captured into a CUDA graph (three back-to-back calls of one
    plan, so the bulk ring's claim counter must reset between launches) and
    replayed twice: every replay rebuilds the destination blocks exactly."""
    set_engine(group, engine)
    glob = global_tensor("bf16", (2048, 4096), seed=14)
    src, dst = ((2,), (0,)), ((4, 2), (R, 1))
    sb = src_blocks(glob, *src)
    exp = rs.reshard(sb, src[0], src[1], dst[0], dst[1], glob.shape)
    sends = [to_device(b) for b in sb]
    recvs = [torch.zeros(e.size, dtype=torch.bfloat16, device="cuda") for e in exp]
    sl, dl = tccl.make_layout(src[0], src[1], 0), tccl.make_layout(dst[0], dst[1], 2)
    s = torch.cuda.Stream()
    group.reshard(sends, sl, recvs, dl, glob.shape, stream=s.cuda_stream)  # plans outside the capture
    torch.cuda.synchronize()
    assert group.last_launch()["engine"] == ENGINES[engine]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for _ in range(3):
            group.reshard(sends, sl, recvs, dl, glob.shape, stream=s.cuda_stream)
    for _ in range(2):
        for r in recvs:
            r.zero_()
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert group.query_error() == tccl.tcclSuccess
        for m, (t, e) in enumerate(zip(recvs, exp)):
            mm = first_mismatch(to_host(t), e)
            assert mm is None, f"{engine} replay: rank {m} first mismatch {mm}"
