"""Reshard planner on the host (tcclReshardInspect), no GPU.

  * every element of every destination block arrives exactly once per
    destination replica, from a source block that holds it;
  * each transfer is read once (from one source replica) and written to all
    replicas of its destination block; source replicas' loads differ by at
    most one (the article's leader balancing);
  * the article's example A (TP4 -> TP2 x DP2) plans four transfers, one per
    trainer rank, each written to a generator replica pair;
  * the article's constraints are enforced.
"""
import itertools

import numpy as np
import pytest

import collective_communication_planner_gb300 as tccl
from oracle import reshard as rs

R = tccl.TCCL_REPLICATE
BASE = 1 << 40


def fake_bufs(n, stride=1 << 32, mis=0):
    return [BASE + i * stride + mis for i in range(n)]


def inspect(src, dst, shape, dtype=tccl.tcclFloat32, mis=0):
    s = tccl.make_layout(*src)
    d = tccl.make_layout(*dst)
    ns, nd = rs.nranks(src[0]), rs.nranks(dst[0])
    sb = fake_bufs(ns, mis=mis)
    db = [BASE + (1 << 38) + i * (1 << 32) + mis for i in range(nd)]
    return tccl.tcclReshardInspect(s, d, shape, dtype, sb, db)


def test_article_example_a_plan(golden_dir):
    shape = [4, 8]
    r, tr, br, bw, nw = inspect(((1, 4), (R, 0), 0), ((2, 2), (R, 0), 4), shape)
    assert r == 0 and len(tr) == 4
    by_src = {t["src"]: t for t in tr}
    for k in range(4):
        t = by_src[k]
        assert t["lo"] == [k, 0] and t["hi"] == [k + 1, 8]
        # rows 0-1 go to mesh ranks 0 and 2 (G4, G6); rows 2-3 to 1 and 3 (G5, G7)
        assert t["dst_mask"] == (0b0101 if k < 2 else 0b1010)
    assert br == 4 * 8 * 4 and bw == 2 * br


def test_article_example_b_plan():
    """Example B per pipeline stage: trainer mesh [2] Shard(0) from c-rank 0 to
    generator mesh [1] Replicate() at c-rank 2. Two transfers, one per trainer
    rank, each its half of the rows, both into the single generator block."""
    shape = [6, 10]
    r, tr, br, bw, nw = inspect(((2,), (0,), 0), ((1,), (R,), 2), shape)
    assert r == 0 and len(tr) == 2
    by_src = {t["src"]: t for t in tr}
    assert by_src[0]["lo"] == [0, 0] and by_src[0]["hi"] == [3, 10]
    assert by_src[1]["lo"] == [3, 0] and by_src[1]["hi"] == [6, 10]
    assert all(t["dst_mask"] == 1 for t in tr)
    assert br == 6 * 10 * 4 and bw == br


LAYOUTS = [((4,), (0,)), ((4,), (R,)), ((2, 2), (R, 0)), ((2, 2), (0, R)), ((2, 2), (1, R)),
           ((1, 4), (R, 1)), ((2, 4), (R, 0)), ((8,), (1,)), ((2, 1, 2), (R, R, 1))]


@pytest.mark.parametrize("src,dst", [(a, b) for a in LAYOUTS for b in LAYOUTS])
def test_exact_delivery_and_balanced_sources(src, dst):
    shape = [8, 16]
    r, tr, br, bw, nw = inspect((src[0], src[1], 0), (dst[0], dst[1], 8), shape)
    assert r == 0
    nd = rs.nranks(dst[0])
    got = {m: np.zeros(shape, np.int32) for m in range(nd)}
    loads = [0] * rs.nranks(src[0])
    for t in tr:
        sbox = rs.local_box(shape, src[0], src[1], t["src"])
        # the source really holds the piece
        assert all(sl <= lo and hi <= sh for (sl, sh), lo, hi in zip(sbox, t["lo"], t["hi"]))
        loads[t["src"]] += 1
        for m in range(nd):
            if (t["dst_mask"] >> m) & 1:
                got[m][t["lo"][0]:t["hi"][0], t["lo"][1]:t["hi"][1]] += 1
    for m in range(nd):
        box = rs.local_box(shape, dst[0], dst[1], m)
        want = np.zeros(shape, np.int32)
        want[box[0][0]:box[0][1], box[1][0]:box[1][1]] = 1
        assert np.array_equal(got[m], want), (src, dst, m)
    # replicas of one source block share its transfers evenly
    blocks = {}
    for m in range(rs.nranks(src[0])):
        blocks.setdefault(tuple(map(tuple, rs.local_box(shape, src[0], src[1], m))), []).append(m)
    for ranks in blocks.values():
        ls = [loads[m] for m in ranks]
        assert max(ls) - min(ls) <= 1
    # bytes: every destination block written once per replica
    written = sum(int(np.prod([hi - lo for lo, hi in rs.local_box(shape, dst[0], dst[1], m)]))
                  for m in range(nd)) * 4
    assert bw == written


def test_three_dimensional_plan_covers_blocks():
    shape = [4, 8, 8]
    r, tr, br, bw, nw = inspect(((2, 2), (R, 2), 0), ((4,), (1,), 4), shape)
    assert r == 0
    assert bw == 4 * 8 * 8 * 4 and nw >= len(tr)


def test_rejects_what_the_article_excludes():
    shape = [8, 8]
    assert inspect(((2, 2), (0, 1), 0), ((4,), (0,), 4), shape)[0] == tccl.tcclInvalidArgument
    assert inspect(((3,), (0,), 0), ((4,), (0,), 4), shape)[0] == tccl.tcclInvalidArgument
    assert inspect(((4,), (2,), 0), ((4,), (0,), 4), shape)[0] == tccl.tcclInvalidArgument
    # meshes sharing ranks
    assert inspect(((4,), (0,), 0), ((4,), (0,), 2), shape)[0] == tccl.tcclInvalidArgument


def test_misaligned_buffers_plan_element_wise_windows():
    shape = [8, 16]
    r, tr, br, bw, nw = inspect(((4,), (0,), 0), ((2,), (0,), 4), shape, mis=4)
    assert r == 0 and bw == 8 * 16 * 4
