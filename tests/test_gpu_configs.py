"""The five workload configurations at full size, in the default launch
configuration (Auto engine), checked bit for bit against the oracle on every
output element (the C oracle's threaded variant, whose bits equal the plain
one's, keeps this to seconds).

  C1  P=2 fp32 sum allreduce, out of place, 1,048,576 elements per rank,
      uniform[-1,1) seed 0
  C2  P=4 bf16: reduce-scatter (8 Mi per rank out) then all-gather, and the
      fused allreduce, 32 Mi elements (64 MiB) per rank, N(0,1) seed 1;
      reduce-scatter + all-gather equals the allreduce bit for bit
  C3  P=8 fp32 allreduce in place, sum/min/max, 4 KiB .. 256 MiB per rank in
      powers of two, uniform[-1,1) seed 2; int32 sum, uniform [-1000,1000]
  C4  P=8 bf16 sum allreduce, 128 MiB per rank, N(0,0.02) seed 3, CTA caps
      8, 16, 32 and uncapped
  C5  P=8 bf16 sum allreduce of [tokens, 8192] activations, tokens in
      {1, 8, 64, 512, 4096}, N(0,1) seed 4
"""
import numpy as np
import pytest
import torch

import collective_communication_planner_gb300 as tccl
import datagen
import oracle
from gpu_util import first_mismatch, same_bits, to_device, to_host

pytestmark = pytest.mark.gpu


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


def oracle_ar(xs, dtype, op="sum"):
    out = np.empty_like(xs[0])
    oracle.allreduce(xs, dtype, op, recvs=[out] * len(xs), nthreads=0)
    return out


def check_all(recvs, exp, what):
    for r, t in enumerate(recvs):
        got = to_host(t)
        mm = first_mismatch(got, exp)
        assert mm is None, f"{what}: rank {r} first mismatch at {mm[0]} ({mm[1]} elements)"


def test_c1_p2_fp32_sum_out_of_place(groups):
    p, n = 2, 1_048_576
    xs = datagen.rank_buffers("uniform_f32", 0, p, n)
    exp = oracle_ar(xs, "f32")
    g = groups(p)
    sends = [to_device(x) for x in xs]
    recvs = [torch.full_like(s, float("nan")) for s in sends]
    g.all_reduce(sends, recvs)
    torch.cuda.synchronize()
    assert g.query_error() == tccl.tcclSuccess
    check_all(recvs, exp, "C1")


def test_c2_p4_bf16_reduce_scatter_allgather_and_allreduce(groups):
    p, n = 4, 32 * 1024 * 1024
    rc = n // p
    xs = datagen.rank_buffers("normal_bf16", 1, p, n, mu=0.0, sigma=1.0)
    exp_ar = oracle_ar(xs, "bf16")
    exp_rs = oracle.reduce_scatter(xs, "bf16", "sum", nthreads=0)
    g = groups(p)
    sends = [to_device(x) for x in xs]
    parts = [torch.empty(rc, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    g.reduce_scatter(sends, parts)
    gathered = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    g.all_gather(parts, gathered)
    fused = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    g.all_reduce(sends, fused)
    torch.cuda.synchronize()
    assert g.query_error() == tccl.tcclSuccess
    for r in range(p):
        assert same_bits(to_host(parts[r]), exp_rs[r]), f"C2 RS rank {r}"
    check_all(gathered, exp_ar, "C2 RS+AG")
    check_all(fused, exp_ar, "C2 AR")
    for r in range(p):
        assert torch.equal(gathered[r].view(torch.int16), fused[r].view(torch.int16))


C3_SIZES = [4096 << k for k in range(17)]  # 4 KiB .. 256 MiB per rank


@pytest.mark.parametrize("dtype,op", [("f32", "sum"), ("f32", "min"), ("f32", "max"),
                                      ("i32", "sum")])
def test_c3_p8_in_place_sweep(groups, dtype, op):
    p = 8
    g = groups(p)
    for nbytes in C3_SIZES:
        n = nbytes // 4
        if dtype == "f32":
            xs = datagen.rank_buffers("uniform_f32", 2, p, n)
        else:
            xs = datagen.rank_buffers("int32", 2, p, n, lo=-1000, hi=1000)
        exp = oracle_ar(xs, dtype, op)
        bufs = [to_device(x) for x in xs]
        del xs
        g.all_reduce(bufs, None, op=op)  # in place
        torch.cuda.synchronize()
        assert g.query_error() == tccl.tcclSuccess
        check_all(bufs, exp, f"C3 {dtype} {op} {nbytes} B/rank")
        del bufs
        torch.cuda.empty_cache()


@pytest.mark.parametrize("cap", [8, 16, 32, 0])
def test_c4_p8_bf16_128mib_caps(groups, cap):
    p, n = 8, 64 * 1024 * 1024
    xs = datagen.rank_buffers("normal_bf16", 3, p, n, mu=0.0, sigma=0.02)
    exp = oracle_ar(xs, "bf16")
    g = groups(p)
    sends = [to_device(x) for x in xs]
    del xs
    recvs = [torch.empty_like(s) for s in sends]
    g.record_sms(True)
    g.read_sm_record()
    g.all_reduce(sends, recvs, cta_cap=cap)
    sms = g.read_sm_record()
    g.record_sms(False)
    assert g.query_error() == tccl.tcclSuccess
    info = g.last_launch()
    if cap:
        # per launch at most `cap` CTAs; the copy-out engine's segment kernels
        # run one after the other, so the SM record (a union) may hold more
        assert info["ctas"] <= cap and sms <= cap * max(1, info["ce_segments"])
    check_all(recvs, exp, f"C4 cap {cap}")


@pytest.mark.parametrize("tokens", [1, 8, 64, 512, 4096])
def test_c5_p8_bf16_tp_activations(groups, tokens):
    p, n = 8, tokens * 8192
    xs = datagen.rank_buffers("normal_bf16", 4, p, n, mu=0.0, sigma=1.0)
    exp = oracle_ar(xs, "bf16")
    g = groups(p)
    sends = [to_device(x).view(tokens, 8192) for x in xs]
    recvs = [torch.empty_like(s) for s in sends]
    g.all_reduce(sends, recvs)
    torch.cuda.synchronize()
    assert g.query_error() == tccl.tcclSuccess
    check_all([r.view(-1) for r in recvs], exp, f"C5 tokens {tokens}")
