"""The tolerance for the arrival-order mode, checked on the CPU: an fp32 sum
folded in any rank order stays within 2 (P-1) 2^-24 sum_r |x_r| of the
oracle's ascending fold (the textbook bound for recursive summation, applied
to both sides), and the check rejects a planted error that is larger."""
import numpy as np
import pytest

import datagen
import oracle
from gpu_util import within_summation_bound


def any_order_fold(xs, rng):
    """Per element, the ranks summed in an independent random order (fp32)."""
    x = np.stack(xs)
    perm = np.argsort(rng.random(x.shape), axis=0)
    xp = np.take_along_axis(x, perm, axis=0)
    acc = xp[0].copy()
    for r in range(1, len(xs)):
        acc = (acc + xp[r]).astype(np.float32)
    return acc


@pytest.mark.parametrize("p", [2, 3, 5, 8, 16])
def test_any_order_is_within_the_bound(p):
    rng = np.random.default_rng(p)
    xs = datagen.rank_buffers("uniform_f32", 40 + p, p, 20_000)
    exp = oracle.allreduce(xs, "f32", "sum")[0]
    got = any_order_fold(xs, rng)
    ok, _ = within_summation_bound(got, exp, xs)
    assert ok
    if p >= 5:  # with five or more ranks the order really changes some results
        assert np.count_nonzero(got != exp) > 0


def test_identical_results_need_no_bound():
    xs = datagen.rank_buffers("uniform_f32", 7, 4, 1000)
    exp = oracle.allreduce(xs, "f32", "sum")[0]
    assert within_summation_bound(exp.copy(), exp, xs) == (True, 0)


@pytest.mark.parametrize("p", [2, 8])
def test_planted_errors_are_caught(p):
    xs = datagen.rank_buffers("uniform_f32", 9, p, 1000)
    exp = oracle.allreduce(xs, "f32", "sum")[0]
    abs_sum = np.sum(np.abs(np.stack(xs).astype(np.float64)), axis=0)
    for i, scale in ((3, 4.0), (500, 100.0)):
        bad = exp.copy()
        bad[i] = np.float32(exp[i] + scale * 2 * (p - 1) * 2.0 ** -24 * abs_sum[i] + 1e-6)
        ok, _ = within_summation_bound(bad, exp, xs)
        assert not ok
    # a dropped rank is far outside
    dropped = oracle.allreduce(xs[:-1], "f32", "sum")[0]
    assert not within_summation_bound(dropped, exp, xs)[0]
