"""GPU parity for tcclAllReduceRMSNorm against the RMSNorm oracle.

Tolerance (derived from the arithmetic, the pages give none): the rank sum is
bit-exact (the same ascending fp32 fold as the allreduce); the row's sum of
squares is a fp32 tree reduction (relative error below log2(hidden) * 2^-24 ~
1e-6), rsqrtf adds at most 2 ulp, two fp32 products 2^-23. All of it is far
below half a bf16 ulp (2^-9), so a bf16 output differs from the fp64-evaluated
oracle by at most one ulp and only rarely; a fp32 output agrees to 2^-18
relative."""
import numpy as np
import pytest
import torch

import collective_communication_planner_gb300 as tccl
import datagen
from gpu_util import to_device, to_host
from oracle import rmsnorm as rn

pytestmark = pytest.mark.gpu
KIND = {"f32": "uniform_f32", "bf16": "normal_bf16"}
TORCH = {"f32": torch.float32, "bf16": torch.bfloat16}


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


def check(got, exp_rounded, exp64, dtype, what):
    if dtype == "bf16":
        d = np.abs(got.astype(np.int64) - exp_rounded.astype(np.int64))
        sign_flip = (got >> 15) != (exp_rounded >> 15)
        assert not np.any(sign_flip & (d > 1)), what
        assert d.max() <= 1, f"{what}: max bf16 ulp distance {d.max()}"
        assert np.count_nonzero(d) <= max(2, got.size // 1000), f"{what}: {np.count_nonzero(d)} differ"
    else:
        err = np.abs(got.astype(np.float64) - exp64)
        assert np.all(err <= 2.0 ** -18 * np.abs(exp64) + 1e-30), f"{what}: max rel {np.max(err / (np.abs(exp64) + 1e-30))}"


def run(g, dtype, p, rows, hidden, eps=1e-6, cap=0, in_place=False, seed=4):
    xs = datagen.rank_buffers(KIND[dtype], seed, p, rows * hidden)
    gamma = datagen.rank_buffers(KIND[dtype], seed + 100, 1, hidden)[0]
    exp, exp64 = rn.allreduce_rmsnorm(xs, gamma, rows, hidden, eps, dtype)
    sends = [to_device(x).view(rows, hidden) for x in xs]
    recvs = sends if in_place else [torch.empty_like(s) for s in sends]
    g.all_reduce_rmsnorm(sends, recvs, to_device(gamma), eps=eps, cta_cap=cap)
    torch.cuda.synchronize()
    assert g.query_error() == tccl.tcclSuccess
    for r in range(p):
        check(to_host(recvs[r]).ravel(), exp, exp64, dtype, f"{dtype} P={p} rows={rows} hidden={hidden} rank {r}")


@pytest.mark.parametrize("tokens", [1, 8, 64, 512, 4096])
def test_tp_activations_bf16(groups, tokens):
    run(groups(8), "bf16", 8, tokens, 8192)


@pytest.mark.parametrize("dtype,hidden", [("bf16", 256), ("bf16", 1000), ("bf16", 16384),
                                          ("f32", 4), ("f32", 4096), ("f32", 8192)])
@pytest.mark.parametrize("p", [1, 3, 8])
def test_shapes_and_types(groups, dtype, hidden, p):
    run(groups(p), dtype, p, 37, hidden)


def test_in_place_caps_and_eps(groups):
    run(groups(4), "bf16", 4, 300, 4096, cap=3, in_place=True)
    run(groups(4), "f32", 4, 64, 2048, eps=0.5)


@pytest.mark.parametrize("dtype,hidden", [("bf16", 8192), ("bf16", 1000), ("bf16", 16384),
                                          ("f32", 4), ("f32", 8192)])
@pytest.mark.parametrize("rows", [1, 3, 19, 76])
def test_cluster_split_matches_single_cta_rows(monkeypatch, dtype, hidden, rows):
    """Few rows take the cluster path (a row split over C CTAs whose partial
    sums of squares meet in distributed shared memory); the same call with the
    cluster path switched off takes one CTA per row. Both meet the oracle's
    tolerance, and the rank sums they normalise are the same."""
    p = 4
    g = tccl.Group(p)
    try:
        run(g, dtype, p, rows, hidden, seed=rows)
        info = g.last_launch()
        c = info["ctas"] // min(rows, info["ctas"])
        assert info["threads"] == 256 and c in (2, 4, 8) and info["ctas"] == rows * c, info
        run(g, dtype, p, rows, hidden, seed=rows, cap=5)
        assert g.last_launch()["ctas"] == 4, g.last_launch()
    finally:
        g.close()
    monkeypatch.setenv("TCCL_RMSNORM_CLUSTER", "0")
    g = tccl.Group(p)
    try:
        run(g, dtype, p, rows, hidden, seed=rows)
        assert g.last_launch()["ctas"] == rows
    finally:
        g.close()


def test_rejects_unsupported_calls(groups):
    g = groups(2)
    st = torch.cuda.current_stream().cuda_stream

    def bufs(rows, hidden, dtype=torch.bfloat16):
        return [torch.zeros(rows, hidden, dtype=dtype, device="cuda") for _ in range(2)]

    gam = torch.ones(32768, dtype=torch.bfloat16, device="cuda")
    s, r = bufs(4, 32768), bufs(4, 32768)
    assert tccl.tcclAllReduceRMSNorm(g.handle, s, r, 4, 32768, gam, 1e-6, 1, st) == \
        tccl.tcclInvalidArgument  # hidden above the limit
    s, r = bufs(4, 1003), bufs(4, 1003)
    assert tccl.tcclAllReduceRMSNorm(g.handle, s, r, 4, 1003, gam, 1e-6, 1, st) == \
        tccl.tcclInvalidArgument  # not a whole number of 16-byte vectors
    s, r = bufs(4, 64, torch.int32), bufs(4, 64, torch.int32)
    assert tccl.tcclAllReduceRMSNorm(g.handle, s, r, 4, 64, gam, 1e-6, 2, st) == \
        tccl.tcclInvalidArgument  # int32
    s, r = bufs(4, 64), bufs(4, 64)
    assert tccl.tcclAllReduceRMSNorm(g.handle, s, r, 4, 64, gam.data_ptr() + 2, 1e-6, 1, st) == \
        tccl.tcclInvalidArgument  # misaligned gamma
    assert tccl.tcclAllReduceRMSNorm(g.handle, s, r, 4, 64, gam, -1.0, 1, st) == \
        tccl.tcclInvalidArgument  # negative eps
    assert tccl.tcclAllReduceRMSNorm(g.handle, s, r, 4, 64, gam, 1e-6, 1, st) == tccl.tcclSuccess
    torch.cuda.synchronize()


@pytest.mark.parametrize("case", range(48))
def test_random_call(groups, case):
    """Seeded random fused calls: dtype, P from 1 to 12, rows from 1 to 700
    (both sides of the cluster-split threshold), any hidden that is a whole
    number of 16-byte vectors up to the limit (16384 bf16, 8192 fp32), caps,
    eps and the in-place form; the oracle's work is kept to a few million
    elements."""
    rng = np.random.default_rng(7000 + case)
    dtype = str(rng.choice(["bf16", "f32"]))
    vec, limit = (8, 16384) if dtype == "bf16" else (4, 8192)
    p = int(rng.integers(1, 13))
    hidden = vec * int(rng.integers(1, limit // vec + 1))
    max_rows = max(1, min(700, 4_000_000 // (hidden * p)))
    rows = int(rng.integers(1, max_rows + 1))
    cap = int(rng.choice([0, 0, 1, 3, 8, 40]))
    eps = float(rng.choice([1e-6, 1e-5, 0.25]))
    in_place = bool(rng.random() < 0.3)
    run(groups(p), dtype, p, rows, hidden, eps=eps, cap=cap, in_place=in_place, seed=case)


@pytest.mark.parametrize("cap,rows", [(4, 4), (4, 5), (4, 9), (1, 7), (3, 300), (0, 700), (0, 4096)])
def test_row_claiming_back_to_back(groups, cap, rows):
    """With more rows than CTAs the fused kernel's CTAs claim rows from a
    counter that the last CTA resets for the next launch: three calls on
    different data, enqueued back to back with no synchronisation between
    them, each equal to the oracle (rows = CTAs takes no counter)."""
    p, hidden = 8, 1024
    g = groups(p)
    cases = []
    for k in range(3):
        xs = datagen.rank_buffers("normal_bf16", 60 + k, p, rows * hidden)
        gamma = datagen.rank_buffers("normal_bf16", 70 + k, 1, hidden)[0]
        sends = [to_device(x).view(rows, hidden) for x in xs]
        recvs = [torch.empty_like(s) for s in sends]
        cases.append((xs, gamma, sends, recvs, to_device(gamma)))
    for xs, gamma, sends, recvs, gamma_d in cases:
        g.all_reduce_rmsnorm(sends, recvs, gamma_d, eps=1e-6, cta_cap=cap)
    torch.cuda.synchronize()
    assert g.query_error() == tccl.tcclSuccess
    if cap:
        assert g.last_launch()["ctas"] <= cap
    for k, (xs, gamma, sends, recvs, _) in enumerate(cases):
        exp, exp64 = rn.allreduce_rmsnorm(xs, gamma, rows, hidden, 1e-6, "bf16")
        for r in range(p):
            check(to_host(recvs[r]).ravel(), exp, exp64, "bf16", f"call {k} cap {cap} rows {rows} rank {r}")


def test_prepared_fused_call(groups):
    """prepare_all_reduce_rmsnorm issues the same fused call as
    all_reduce_rmsnorm; repeated on new data in the same buffers it follows
    the data."""
    p, rows, hidden = 8, 4, 8192
    g = groups(p)
    gamma = datagen.rank_buffers("normal_bf16", 81, 1, hidden)[0]
    gamma_d = to_device(gamma)
    sends = [torch.empty(rows, hidden, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    recvs = [torch.empty_like(s) for s in sends]
    call = g.prepare_all_reduce_rmsnorm(sends, recvs, gamma_d, eps=1e-6)
    for seed in (82, 83):
        xs = datagen.rank_buffers("normal_bf16", seed, p, rows * hidden)
        for t, x in zip(sends, xs):
            t.copy_(to_device(x).view(rows, hidden))
        call()
        torch.cuda.synchronize()
        assert g.query_error() == tccl.tcclSuccess
        exp, exp64 = rn.allreduce_rmsnorm(xs, gamma, rows, hidden, 1e-6, "bf16")
        for r in range(p):
            check(to_host(recvs[r]).ravel(), exp, exp64, "bf16", f"prepared seed {seed} rank {r}")
