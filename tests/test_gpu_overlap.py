"""Allreduce beside a concurrent GEMM (T-CCL's overlap study, "NCCL M2N vs
T-CCL" article, section 2.2: a collective running while a GEMM computes).

A loop of bf16 GEMMs (torch.matmul, so cuBLAS) runs on one stream; C4-shaped
allreduces (P=8, bf16 sum, N(0, 0.02)) run on another, queued right behind
the first GEMMs so the two overlap: under caps 16 and 32 with Auto's engine
(the copy-out engine: capped fold plus copy-engine copies) and with the
SM-only bulk engine, and uncapped. Every output element of every allreduce
is compared with the CPU oracle, bit for bit, and every GEMM result with the
same GEMM computed alone beforehand, so neither side corrupts the other.
"""
import pytest
import torch

import collective_communication_planner_gb300 as tccl
import datagen
import oracle
from gpu_util import first_mismatch, to_device, to_host

pytestmark = pytest.mark.gpu

P = 8
COUNT = 16 * 1024 * 1024   # 32 MiB per rank: four copy-out segments of 8 MiB
GEMM_N = 4096
GEMMS = 24
CALLS = 3


@pytest.fixture(scope="module")
def data():
    xs = datagen.rank_buffers("normal_bf16", 3, P, COUNT, mu=0.0, sigma=0.02)
    exp = oracle.allreduce(xs, "bf16", "sum", nthreads=0)
    gen = torch.Generator(device="cpu").manual_seed(7)
    a = torch.randn(GEMM_N, GEMM_N, generator=gen).to(torch.bfloat16).cuda()
    b = torch.randn(GEMM_N, GEMM_N, generator=gen).to(torch.bfloat16).cuda()
    alone = torch.matmul(a, b)
    torch.cuda.synchronize()
    return xs, exp, a, b, alone


@pytest.mark.parametrize("cap,sm_only", [(16, False), (32, False), (16, True), (32, True),
                                         (0, False)])
def test_allreduce_beside_a_gemm_matches_the_oracle(data, cap, sm_only):
    xs, exp, a, b, alone = data
    sends = [to_device(x) for x in xs]
    recv_sets = [[torch.empty_like(s) for s in sends] for _ in range(CALLS)]
    gemm_out = [torch.empty_like(alone) for _ in range(GEMMS)]
    s_gemm, s_ar = torch.cuda.Stream(), torch.cuda.Stream()
    with tccl.Group(P) as g:
        if sm_only:
            g.set_config(ce_auto_max_cap=-1)
        # plan (and for the copy-out engine create its copy streams) before
        # the timed overlap, so the calls below only enqueue work
        g.all_reduce(sends, recv_sets[0], cta_cap=cap)
        torch.cuda.synchronize()
        engine = g.last_launch()["engine"]
        expected_engine = (tccl.tcclEngineCopyOut if (cap and not sm_only) else tccl.tcclEngineBulk)
        assert engine == expected_engine
        for rs in recv_sets:
            for t in rs:
                t.fill_(0)
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        ev[0].record(s_gemm)
        with torch.cuda.stream(s_gemm):
            for out in gemm_out:
                torch.matmul(a, b, out=out)
        ev[1].record(s_gemm)
        s_ar.wait_event(ev[0])  # start the allreduces with the GEMMs
        ev[2].record(s_ar)
        for rs in recv_sets:
            g.all_reduce(sends, rs, cta_cap=cap, stream=s_ar.cuda_stream)
        ev[3].record(s_ar)
        torch.cuda.synchronize()
        assert g.query_error() == tccl.tcclSuccess
    # the allreduces were queued at the start of the GEMM loop; report how
    # much of them fell inside it (timing is not asserted: the block
    # scheduler decides how the two kernels interleave)
    print(f"cap {cap} sm_only {sm_only}: GEMM loop {ev[0].elapsed_time(ev[1]):.3f} ms, "
          f"allreduces {ev[2].elapsed_time(ev[3]):.3f} ms, "
          f"both done after {ev[0].elapsed_time(ev[3]):.3f} ms")
    for c, rs in enumerate(recv_sets):
        for r, t in enumerate(rs):
            mm = first_mismatch(to_host(t), exp[r])
            assert mm is None, f"call {c}, rank {r}: first mismatch at {mm[0]} ({mm[1]} elements)"
    for i, out in enumerate(gemm_out):
        assert torch.equal(out, alone), f"GEMM {i} differs from the GEMM run alone"
