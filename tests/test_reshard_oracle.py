"""Pins for the M2N reshard oracle (oracle/reshard.py).

  * the article's worked example A (TP4 -> TP2 x DP2, tests/golden): the
    destination ownership it prints, and the values that land there;
  * an element-by-element check in pure Python against the layout definition,
    over many meshes, placements and shapes;
  * round trips, full replication, and a planted mistake (column-major mesh
    coordinates) that the golden example catches.
"""
import itertools

import numpy as np
import pytest

from oracle import reshard as rs

R = rs.REPLICATE


def golden(golden_dir):
    rows = []
    for ln in (golden_dir / "m2n_example_tp4_to_tp2dp2.txt").read_text().splitlines():
        if ln and not ln.startswith("#"):
            rows.append([int(v) for v in ln.split()])
    return rows


def value(g):
    return 1000 * g[0] + g[1] if len(g) == 2 else sum((i + 7) * 31 ** k for k, i in enumerate(g))


def make_src(shape, dims, place, dtype=np.float32):
    bufs = []
    for m in range(rs.nranks(dims)):
        box = rs.local_box(shape, dims, place, m)
        bufs.append(np.array([value(g) for g in itertools.product(*[range(lo, hi) for lo, hi in box])],
                             dtype=dtype))
    return bufs


def test_article_example_a_ownership(golden_dir):
    shape = (4, 8)
    dst_dims, dst_place, start = (2, 2), (R, 0), 4
    for grank, r0, r1, c0, c1 in golden(golden_dir):
        box = rs.local_box(shape, dst_dims, dst_place, grank - start)
        assert box == [(r0, r1), (c0, c1)]
    # the trainer side: rank k holds row k
    for k in range(4):
        assert rs.local_box(shape, (1, 4), (R, 0), k) == [(k, k + 1), (0, 8)]


def test_article_example_a_values(golden_dir):
    shape = (4, 8)
    src = make_src(shape, (1, 4), (R, 0))
    out = rs.reshard(src, (1, 4), (R, 0), (2, 2), (R, 0), shape)
    for grank, r0, r1, c0, c1 in golden(golden_dir):
        exp = np.array([[value((r, c)) for c in range(c0, c1)] for r in range(r0, r1)],
                       dtype=np.float32).ravel()
        assert np.array_equal(out[grank - 4], exp)


@pytest.mark.parametrize("shape", [(4, 8), (6, 3), (2, 5, 4)])
def test_article_example_b_stage_gather(shape):
    """The article's example B (TP2,PP2 -> TP1,PP1), one reshard per pipeline
    stage: in a stage's communicator the trainer mesh [2] from c-rank 0 holds
    Shard(0), the generator mesh [1] at c-rank 2 holds Replicate(). So the
    generator ends with the whole stage weight, which in row-major order is
    trainer c-rank 0's block followed by c-rank 1's."""
    for stage in range(2):
        src = [b + 100000 * stage for b in make_src(shape, (2,), (0,))]
        out = rs.reshard(src, (2,), (0,), (1,), (R,), shape)
        assert len(out) == 1
        assert np.array_equal(out[0], np.concatenate(src))
        half = shape[0] // 2
        assert rs.local_box(shape, (2,), (0,), 1)[0] == (half, shape[0])


def test_planted_column_major_coordinates_fail_the_golden(golden_dir, monkeypatch):
    def col_major(dims, m):
        out = []
        for n in dims:
            out.append(m % n)
            m //= n
        return tuple(out)

    monkeypatch.setattr(rs, "mesh_coords", col_major)
    bad = 0
    for grank, r0, r1, c0, c1 in golden(golden_dir):
        if rs.local_box((4, 8), (2, 2), (R, 0), grank - 4) != [(r0, r1), (c0, c1)]:
            bad += 1
    assert bad > 0


LAYOUTS = [
    ((4,), (0,)), ((4,), (R,)), ((2, 2), (R, 0)), ((2, 2), (0, R)), ((2, 2), (1, R)),
    ((1, 4), (R, 1)), ((2, 4), (R, 0)), ((8,), (1,)), ((2,), (0,)), ((1,), (R,)),
    ((2, 1, 2), (R, R, 1)),
]


@pytest.mark.parametrize("src", LAYOUTS)
@pytest.mark.parametrize("dst", LAYOUTS[::2])
def test_element_by_element(src, dst):
    shape = (8, 16)
    src_bufs = make_src(shape, *src)
    out = rs.reshard(src_bufs, src[0], src[1], dst[0], dst[1], shape)
    assert rs.element_owner_check(out, dst[0], dst[1], shape, value)
    for m, o in enumerate(out):
        box = rs.local_box(shape, dst[0], dst[1], m)
        assert o.size == np.prod([hi - lo for lo, hi in box])


def test_three_dimensional_tensor():
    shape = (4, 8, 8)
    src = ((2, 2), (R, 2))
    dst = ((4,), (1,))
    out = rs.reshard(make_src(shape, *src), *src, *dst, shape)
    assert rs.element_owner_check(out, *dst, shape, value)


def test_round_trip_and_full_replication():
    shape = (8, 16)
    a = ((2, 4), (R, 0))
    b = ((4, 2), (1, R))
    src = make_src(shape, *a)
    there = rs.reshard(src, *a, *b, shape)
    back = rs.reshard(there, *b, *a, shape)
    for x, y in zip(src, back):
        assert np.array_equal(x, y)
    full = rs.reshard(src, *a, (3,), (R,), shape)
    glob = np.array([[value((r, c)) for c in range(16)] for r in range(8)], np.float32).ravel()
    for f in full:
        assert np.array_equal(f, glob)


def test_rejects_layouts_the_article_excludes():
    with pytest.raises(ValueError):
        rs.local_box((4, 4), (2, 2), (0, 1), 0)       # two sharded axes
    with pytest.raises(ValueError):
        rs.local_box((4, 4), (3,), (0,), 0)           # 4 rows over 3 ranks
    with pytest.raises(ValueError):
        rs.local_box((4, 4), (2,), (2,), 0)           # no dimension 2
