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


def run(g, glob, src, dst, dtype, cap=0, mis=0):
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
    for m, (t, e) in enumerate(zip(recvs, exp)):
        assert t.guards_intact()
        mm = first_mismatch(t.host(), e)
        assert mm is None, f"{src} -> {dst} {dtype}: rank {m} first mismatch {mm}"


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


@pytest.mark.parametrize("src", LAYOUTS)
@pytest.mark.parametrize("dst", LAYOUTS[::2])
def test_layout_pairs(group, src, dst):
    glob = global_tensor("f32", (64, 96))
    run(group, glob, src, dst, "f32")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("mis", [0, 4])
@pytest.mark.parametrize("cap", [0, 3])
def test_dtypes_alignment_caps(group, dtype, mis, cap):
    glob = global_tensor(dtype, (256, 1000))
    run(group, glob, ((8,), (1,)), ((2, 2), (R, 0)), dtype, cap=cap, mis=mis)
    run(group, glob, ((4,), (0,)), ((2, 4), (R, 1)), dtype, cap=cap, mis=mis)


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


@pytest.mark.parametrize("case", range(40))
def test_random_reshard(group, case):
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
    run(group, glob, src, dst, dtype, cap=cap, mis=mis)
