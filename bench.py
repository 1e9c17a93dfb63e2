"""Benchmark: allreduce of P logical rank buffers on one GB300.

Default workload (one step = one fused allreduce through the C ABI):
  C4: P = 8 ranks, bf16 sum, 64 Mi elements (128 MiB) per rank, out of
  place, values N(0, 0.02) from seed 3, uncapped. Footprint 2 GiB > 129 MB of
  L2, so timed iterations stream from HBM without an explicit L2 flush.

Reported (one JSON line on rank 0):
  value      algbw = P * count * bytes / time (GB/s), device-resident inputs
  roofline   HBM bound: algorithmic bytes 2 * P * S per launch (read every
             rank's shard once, write every rank's result once) / mean
             launch time (the timed region between two CUDA events on the
             launching stream, divided by its launches), against the
             measured copy bandwidth
  caps, cap16  the same allreduce under CTA caps 8, 16 and 32 with the
             default engine choice (the copy-out engine), timed the same way:
             HBM fraction of 2 * P * S, the fraction of every byte the call
             moves, engine, CTAs per launch, distinct SMs per launch and over
             the call; cap 16 also with the SM-only bulk engine
  c2         the P = 4, 64 MiB-per-rank allreduce, uncapped, for comparison
  e2e        same metric through the C ABI with the inputs copied from pinned
             host memory and every result copied back, inside the timed region
  cpu_baseline  the CPU oracle (threaded, same per-element order) on the
             host cores, on the same workload

`--impl reference` times the CPU oracle as the reference arm. Under torchrun
(N > 1) every rank runs an independent replica on its own GPU (the path has
no data exchange between GPUs); value = all ranks' bytes / slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time
from datetime import datetime
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "allreduce algbw GB/s & HBM-peak fraction vs P, msg size, CTA cap (1 GB300)"
FALLBACK_HBM_GBS = 6800.0

WORKLOADS = {
    "c1": dict(name="C1: P=2 fp32 sum allreduce, out of place, 1,048,576 elems (4 MiB)/rank, "
                    "uniform[-1,1) seed 0", p=2, count=1_048_576, dtype="f32", op="sum",
               kind="uniform_f32", seed=0, kw={}, in_place=False, cap=0),
    "c2": dict(name="C2: P=4 bf16 sum allreduce, out of place, 32 Mi elems (64 MiB)/rank, "
                    "N(0,1) seed 1", p=4, count=32 * 1024 * 1024, dtype="bf16", op="sum",
               kind="normal_bf16", seed=1, kw=dict(mu=0.0, sigma=1.0), in_place=False, cap=0),
    "c3": dict(name="C3 at 64 MiB/rank: P=8 fp32 sum allreduce, in place, 16 Mi elems/rank, "
                    "uniform[-1,1) seed 2", p=8, count=16 * 1024 * 1024, dtype="f32", op="sum",
               kind="uniform_f32", seed=2, kw={}, in_place=True, cap=0),
    "c4": dict(name="C4: P=8 bf16 sum allreduce, 64 Mi elems (128 MiB)/rank, N(0,0.02) seed 3",
               p=8, count=64 * 1024 * 1024, dtype="bf16", op="sum", kind="normal_bf16", seed=3,
               kw=dict(mu=0.0, sigma=0.02), in_place=False, cap=0),
}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ------------------------------------------------------------------ helpers
def measured_peak():
    p = ROOT / "MEASURED_PEAKS.json"
    try:
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy burst)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 copy measurement)"


def kernel_source_hash() -> str:
    """Hash of the sources the bulk allreduce kernel is compiled from (its
    template, its launch file and the shared argument structs) and of the
    planner that picks its launch shape."""
    h = hashlib.sha256()
    csrc = ROOT / "collective_communication_planner_gb300" / "csrc"
    for f in sorted(csrc / n for n in ("kernels_common.cuh", "dispatch.cuh", "kernels_bulk.cu", "internal.h",
                                       "plan.h", "plan.cpp")):
        h.update(f.name.encode())
        h.update(f.read_bytes())
    return h.hexdigest()[:16]


def recorded_traffic(workload_key: str):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    p = ROOT / "profiles" / "dram_traffic.json"
    try:
        d = json.loads(p.read_text())
    except Exception:
        return None
    e = d.get(workload_key)
    if not e or e.get("kernel_source_sha") != kernel_source_hash():
        return None
    return int(e["dram_bytes_read"]) + int(e["dram_bytes_write"])


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.time(), ln.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self.t:
                self.t.join(timeout=2)

    def summary(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for ts, ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                stamp = datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except Exception:
                stamp = ts
            rows.append((stamp, parts))
        sel = [r for s, r in rows if t0 - 0.15 <= s <= t1 + 0.15]
        window = "soak + timed region"
        if not sel:
            sel = [r for _, r in rows]
            window = "whole run (no sample fell inside the timed region)"
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except Exception:
                return None

        sm = sorted(v for v in (num(r[2]) for r in sel) if v is not None)
        mx = [v for v in (num(r[3]) for r in sel) if v is not None]
        pw = [v for v in (num(r[4]) for r in sel) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in sel for i in range(4)
                          if r[6 + i].lower() in ("active", "0x1", "1")})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(sel), "window": window}


# ------------------------------------------------------------------ replicas
def replica_time(dist, local_ms: float) -> float:
    """Slowest replica's time (max over ranks); a host-side scalar exchange,
    not a data-path collective. Without a process group, the local time."""
    if dist is None:
        return local_ms
    import torch
    t = torch.tensor([local_ms], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, bytes_per_replica: int, slowest_ms: float) -> float:
    """GB/s of all replicas together: every replica moves the same bytes
    (weak scaling), and the job takes as long as its slowest replica."""
    return world * bytes_per_replica / (slowest_ms * 1e-3) / 1e9


# ------------------------------------------------------------------ workload data
def make_inputs(w):
    import datagen
    return datagen.rank_buffers(w["kind"], w["seed"], w["p"], w["count"], **w["kw"])


def host_to_torch(x):
    import numpy as np
    import torch
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(x)


# ------------------------------------------------------------------ CPU oracle timing
def time_oracle(w, xs, min_seconds: float, max_reps: int = 1000, elems: int | None = None):
    """Times the threaded oracle allreduce over the first `elems` elements of
    each rank; returns (seconds per call, threads used, reps)."""
    import numpy as np
    import oracle
    n = elems or w["count"]
    sub = [x[:n] for x in xs]
    out = np.empty(n, dtype=xs[0].dtype)
    recvs = [out] * len(sub)
    nthreads = os.cpu_count() or 1
    oracle.allreduce(sub, w["dtype"], w["op"], recvs=recvs, nthreads=nthreads)  # warm
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.allreduce(sub, w["dtype"], w["op"], recvs=recvs, nthreads=nthreads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            break
    return el / reps, min(nthreads, n // 4096 + 1), reps


# ------------------------------------------------------------------ our arm
def run_ours(args, w, rank, world, dist):
    import numpy as np
    import torch
    import collective_communication_planner_gb300 as tccl

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    p, n, es = w["p"], w["count"], (2 if w["dtype"] == "bf16" else 4)
    S = n * es
    alg_bytes = p * S                      # algbw numerator
    hbm_bytes = 2 * p * S                  # read P shards, write P results
    xs = make_inputs(w)
    host = [host_to_torch(x) for x in xs]
    sends = [h.to(dev) for h in host]
    recvs = sends if w["in_place"] else [torch.empty_like(s) for s in sends]
    stream = torch.cuda.Stream(device=dev)
    st = stream.cuda_stream
    g = tccl.Group(p)
    dt = tccl.DTYPES[w["dtype"]]
    op = tccl.OPS[w["op"]]
    cap = args.cap if args.cap is not None else w["cap"]

    def step():
        r = tccl.tcclAllReduce(g.handle, sends, recvs, n, dt, op, st, cap)
        if r != tccl.tcclSuccess:
            raise tccl.TcclError(r, "tcclAllReduce")

    # parity spot check of this exact launch configuration before timing
    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    import oracle
    k = min(n, 1 << 16)
    idx = np.random.default_rng(0).choice(n, size=k, replace=False)
    idx.sort()
    exp = oracle.allreduce([x[idx].copy() for x in xs], w["dtype"], w["op"])[0]
    got = recvs[p - 1].view(torch.int16 if w["dtype"] == "bf16" else recvs[0].dtype)
    got = got.cpu().numpy()[idx].view(exp.dtype)
    if not np.array_equal(got.view(np.uint8), exp.view(np.uint8)):
        raise SystemExit("bench: result differs from the oracle on sampled elements")
    info = g.last_launch()

    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(args.warmup):
        with torch.cuda.stream(stream):
            step()
    # soak: keep the GPU under this load for ~1 s so clocks settle and the
    # sampler sees the loaded state
    t_soak = time.time()
    stream.synchronize()
    while time.time() - t_soak < args.soak:
        for _ in range(50):
            step()
        stream.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    # the timed region: K back-to-back launches between two events on the
    # launching stream. Only this kernel runs there, so the region divided by
    # K is its average launch duration, inter-launch gaps included (an event
    # pair around every launch would add gaps of its own).
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    t_start = time.time()
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(args.steps):
            step()
        ev[1].record(stream)
    torch.cuda.synchronize()
    t_end = time.time()
    if dist is not None:
        dist.barrier()
    sampler.stop()
    total_ms = ev[0].elapsed_time(ev[1])
    launch_ms = total_ms / args.steps
    clocks = sampler.summary(t_soak, t_end)

    total_ms = replica_time(dist, total_ms)
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(world, alg_bytes, ms_per_step)
    peak, peak_src = measured_peak()
    achieved = hbm_bytes / (launch_ms * 1e-3) / 1e9
    traffic = recorded_traffic(args.workload)

    # the same allreduce under CTA caps, with the default engine choice (the
    # copy-out engine: segment kernels within the cap fold into one anchor
    # rank, the copy engines carry the result to the others) and, at cap 16,
    # with the SM-only bulk engine; each point timed like the main line: K
    # back-to-back calls between one event pair after three warm-up calls
    def reset_config(**kw):
        c = tccl.tcclConfig_t()
        for key, val in kw.items():
            setattr(c, key, val)
        r = tccl.tcclGroupSetConfig(g.handle, c)
        if r != tccl.tcclSuccess:
            raise tccl.TcclError(r, "tcclGroupSetConfig")

    def timed_calls(fn, k):
        for _ in range(3):
            fn()
        stream.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(k):
            fn()
        b.record(stream)
        b.synchronize()
        return a.elapsed_time(b) / k

    def sampled_exact():
        got_s = recvs[p - 1].view(torch.int16 if w["dtype"] == "bf16" else recvs[0].dtype)
        return bool(np.array_equal(got_s.cpu().numpy()[idx].view(np.uint8), exp.view(np.uint8)))

    def cap_point(cap_k, sm_only):
        reset_config(**({"ce_auto_max_cap": -1} if sm_only else {}))

        def call():
            r = tccl.tcclAllReduce(g.handle, sends, recvs, n, dt, op, st, cap_k)
            if r != tccl.tcclSuccess:
                raise tccl.TcclError(r, "tcclAllReduce")

        for t in recvs:
            t.fill_(0)
        call()
        stream.synchronize()
        g.read_sm_record()
        g.record_sms(True)
        call()
        per_launch, union = g.read_sm_record_launches()
        g.record_sms(False)
        pinfo = g.last_launch()
        kc = max(10, min(args.steps, 50))
        ms = timed_calls(call, kc)
        copy_out = pinfo["engine"] == tccl.tcclEngineCopyOut
        # the copy-out call moves more than the collective's 2 P S: the fold
        # reads P S and writes S (the anchor), the copies read and write
        # (P - 1) S (their reads of the anchor can come from L2)
        moved = (3 * p - 1) * S if copy_out else hbm_bytes
        row = {"cap": cap_k, "variant": "sm_only" if sm_only else "auto",
               "engine": pinfo["engine"], "engine_name": "copy-out" if copy_out else "bulk",
               "ctas_per_launch": pinfo["ctas"], "launches_per_call": len(per_launch),
               "copies_per_call": pinfo["ce_copies"], "calls_timed": kc,
               "ms_per_call": round(ms, 5),
               "algbw": round(alg_bytes / (ms * 1e-3) / 1e9, 2),
               "hbm_fraction": round(hbm_bytes / (ms * 1e-3) / 1e9 / peak, 4),
               "moved_fraction": round(moved / (ms * 1e-3) / 1e9 / peak, 4),
               "sms_per_launch_max": max(per_launch) if per_launch else 0,
               "sms_per_launch": per_launch, "sms_union": union,
               "sampled_exact": sampled_exact()}
        if not row["sampled_exact"]:
            raise SystemExit(f"bench: capped result (cap {cap_k}) differs from the oracle on sampled elements")
        return row

    cap_rows = []
    c2_row = None
    if not args.no_caps:
        for cap_k in (8, 16, 32):
            cap_rows.append(cap_point(cap_k, False))
        cap_rows.append(cap_point(16, True))
        reset_config()
        if args.workload != "c2":
            w2 = WORKLOADS["c2"]
            p2, n2 = w2["p"], w2["count"]
            xs2 = make_inputs(w2)
            s2 = [host_to_torch(x).to(dev) for x in xs2]
            r2 = [torch.empty_like(t) for t in s2]
            with tccl.Group(p2) as g2:
                def call2():
                    r = tccl.tcclAllReduce(g2.handle, s2, r2, n2, tccl.DTYPES[w2["dtype"]],
                                           tccl.OPS[w2["op"]], st, 0)
                    if r != tccl.tcclSuccess:
                        raise tccl.TcclError(r, "tcclAllReduce")
                ms2 = timed_calls(call2, max(10, min(args.steps, 200)))
                i2 = g2.last_launch()
            got2 = r2[p2 - 1].view(torch.int16).cpu().numpy()[:4096].view(np.uint16)
            exp2 = oracle.allreduce([x[:4096].copy() for x in xs2], w2["dtype"], w2["op"])[0]
            S2 = n2 * 2
            c2_row = {"workload": w2["name"], "ms_per_call": round(ms2, 5),
                      "algbw": round(p2 * S2 / (ms2 * 1e-3) / 1e9, 2),
                      "hbm_fraction": round(2 * p2 * S2 / (ms2 * 1e-3) / 1e9 / peak, 4),
                      "engine": i2["engine"], "ctas": i2["ctas"],
                      "sampled_exact": bool(np.array_equal(got2, exp2))}
            del s2, r2, xs2

    # reduce-scatter then all-gather on the same workload (two launches)
    rc = n // p
    parts = [torch.empty(rc, dtype=sends[0].dtype, device=dev) for _ in range(p)]
    outs = [torch.empty(n, dtype=sends[0].dtype, device=dev) for _ in range(p)]
    rs_steps = max(10, min(args.steps, 200))

    def rs_ag():
        r1 = tccl.tcclReduceScatter(g.handle, sends, parts, rc, dt, op, st, cap)
        r2 = tccl.tcclAllGather(g.handle, parts, outs, rc, dt, st, cap)
        if r1 or r2:
            raise tccl.TcclError(r1 or r2, "reduce-scatter / all-gather")

    for _ in range(3):
        rs_ag()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(rs_steps):
        rs_ag()
    e1.record(stream)
    e1.synchronize()
    rs_ms = e0.elapsed_time(e1) / rs_steps

    # end to end through the C ABI: every step copies its inputs in from
    # pinned host memory, reduces, and copies every result back. Two device
    # buffer sets and three streams let step i+1's inputs travel while step
    # i's results come back (the host link carries both directions at once).
    # Each step goes in `pieces` slices of the rank buffers (one allreduce
    # call per slice), so a slice's results travel back while the next
    # slice's inputs arrive: only a slice's reduction is not overlapped.
    h_in = [h.pin_memory() for h in host]
    h_out = [torch.empty_like(h).pin_memory() for h in host]
    e2e_steps = max(3, min(args.steps, 20))
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    sets = [(sends, recvs)]
    d2 = [torch.empty_like(t) for t in sends]
    sets.append((d2, d2 if w["in_place"] else [torch.empty_like(t) for t in sends]))
    pieces = max(1, min(args.e2e_pieces, n // 4096))
    cut = [n * k // pieces // 4096 * 4096 for k in range(pieces)] + [n]  # 16-byte aligned slices
    ev_in = [[torch.cuda.Event() for _ in range(pieces)] for _ in range(2)]
    ev_piece = [[torch.cuda.Event() for _ in range(pieces)] for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(nsteps):
        for i in range(nsteps):
            b = i % 2
            snd, rcv = sets[b]
            if i >= 2:
                s_in.wait_event(ev_done[b])   # the kernels of step i-2 have read this set
                s_in.wait_event(ev_out[b])    # and its results have left
            for k in range(pieces):
                lo, hi = cut[k], cut[k + 1]
                with torch.cuda.stream(s_in):
                    for d, h in zip(snd, h_in):
                        d[lo:hi].copy_(h[lo:hi], non_blocking=True)
                    ev_in[b][k].record(s_in)
                stream.wait_event(ev_in[b][k])
                r = tccl.tcclAllReduce(g.handle, [t[lo:hi] for t in snd], [t[lo:hi] for t in rcv], hi - lo,
                                       dt, op, st, cap)
                if r != tccl.tcclSuccess:
                    raise tccl.TcclError(r, "tcclAllReduce")
                ev_piece[b][k].record(stream)
                s_out.wait_event(ev_piece[b][k])
                with torch.cuda.stream(s_out):
                    for h, d in zip(h_out, rcv):
                        h[lo:hi].copy_(d[lo:hi], non_blocking=True)
            ev_done[b].record(stream)
            ev_out[b].record(s_out)

    def e2e_serial_step():
        with torch.cuda.stream(stream):
            for d, h in zip(sends, h_in):
                d.copy_(h, non_blocking=True)
            step()
            for h, d in zip(h_out, recvs):
                h.copy_(d, non_blocking=True)

    e2e_run(2)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    stream.wait_event(t0)
    s_out.wait_event(t0)
    e2e_run(e2e_steps)
    t1.record(s_out)
    t1.synchronize()
    e2e_ms = t0.elapsed_time(t1) / e2e_steps
    # the result of the last step is on the host and correct
    exp_last = oracle.allreduce([x[idx].copy() for x in xs], w["dtype"], w["op"])[0]
    got_last = h_out[p - 1].view(torch.int16 if w["dtype"] == "bf16" else h_out[0].dtype)
    if not np.array_equal(got_last.numpy()[idx].view(np.uint8), exp_last.view(np.uint8)):
        raise SystemExit("bench: end-to-end result differs from the oracle on sampled elements")
    for _ in range(2):
        e2e_serial_step()
    stream.synchronize()
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_serial_step()
    e1.record(stream)
    e1.synchronize()
    e2e_serial_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_ms = replica_time(dist, e2e_ms)
    e2e_serial_ms = replica_time(dist, e2e_serial_ms)
    del d2, sets

    out = None
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            sec, cores, reps = time_oracle(w, xs, args.cpu_seconds)
            cpu = {"value": alg_bytes / sec / 1e9, "unit": "GB/s", "cores": cores,
                   "kind": "oracle",
                   "sample": f"whole workload ({p} x {n} elements), {reps} repetitions, "
                             f"threaded oracle (same per-element order as the plain one)"}
        out = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if w["dtype"] != "i32" else "int32",
            "data": "synthetic (seeded SplitMix64 streams per rank)",
            "config": {"workload": w["name"], "P": p, "count": n, "bytes_per_rank": S,
                       "elem_dtype": w["dtype"], "op": w["op"], "in_place": w["in_place"],
                       "cta_cap": cap, "engine": info["engine"], "ctas": info["ctas"],
                       "stages": info["stages"], "chunk_bytes": info["chunk_bytes"],
                       "l2": f"inputs larger than L2 ({2 * p * S >> 20} MiB footprint), no flush",
                       "parallelism": f"replicas{world}" if world > 1 else "single"},
            "hbm_fraction": round(achieved / peak, 4),
            "busbw": round(S / (ms_per_step * 1e-3) * 2 * (p - 1) / p / 1e9, 2),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": traffic, "peak_source": peak_src,
                         "algorithmic_bytes_per_launch": hbm_bytes,
                         "mean_launch_ms": round(launch_ms, 5)},
            "cap16": next((r for r in cap_rows if r["cap"] == 16 and r["variant"] == "auto"), None),
            "caps": cap_rows,
            "c2": c2_row,
            "rs_then_ag": {"ms_per_step": round(rs_ms, 5),
                           "algbw": round(alg_bytes / (rs_ms * 1e-3) / 1e9, 2),
                           "hbm_bytes_per_step": 2 * (p + 1) * S},
            "e2e": {"value": round(whole_job_rate(world, alg_bytes, e2e_ms), 2), "unit": "GB/s",
                    "h2d_bytes_per_step": p * S, "d2h_bytes_per_step": p * S,
                    "ms_per_step": round(e2e_ms, 4),
                    "pipelining": f"each step in {pieces} slices (one allreduce call per slice); a slice's "
                                  "results copy out while the next slice's, and the next step's, inputs copy "
                                  "in (two device buffer sets, three streams)",
                    "serial_value": round(whole_job_rate(world, alg_bytes, e2e_serial_ms), 2),
                    "serial_ms_per_step": round(e2e_serial_ms, 4)},
            "cpu_baseline": cpu,
            "gpu_launches": args.steps,
            "clocks": clocks,
        }
    g.close()
    return out


# ------------------------------------------------------------------ reference arm
def run_reference(args, w):
    """The CPU oracle as the reference arm: each step is the threaded oracle
    on a bounded prefix of the same workload."""
    xs = make_inputs(w)
    p, n, es = w["p"], w["count"], (2 if w["dtype"] == "bf16" else 4)
    full_sec, _, _ = time_oracle(w, xs, 0.0, max_reps=1)
    budget = 60.0  # seconds for warm-up + timed steps
    per_step = budget / max(1, args.steps + args.warmup)
    elems = n
    while elems > 4096 and full_sec * elems / n > per_step:
        elems //= 2
    import numpy as np
    import oracle
    sub = [x[:elems] for x in xs]
    out = np.empty(elems, dtype=xs[0].dtype)
    nthreads = os.cpu_count() or 1
    for _ in range(args.warmup):
        oracle.allreduce(sub, w["dtype"], w["op"], recvs=[out] * p, nthreads=nthreads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.allreduce(sub, w["dtype"], w["op"], recvs=[out] * p, nthreads=nthreads)
    sec = (time.perf_counter() - t0) / args.steps
    value = p * elems * es / sec / 1e9
    cores = min(nthreads, elems // 4096 + 1)
    sample = f"first {elems} of {n} elements per rank ({p} ranks) per step"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(sec * 1e3, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w["name"], "P": p, "count": n, "bytes_per_rank": n * es},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------ sweep mode
def sweep(args):
    """One JSON line per configuration point of the five workloads (C1..C5):
    device time per op (CUDA events around batches of back-to-back launches:
    `us` is the median of five batches, `us_min` the fastest; graph-captured
    too for small messages), algbw, bus bandwidth, HBM fraction, SMs used, and
    the CPU oracle on 1 core and on all cores for one point per workload.
    Points whose traffic fits three times in L2 are also timed cold: before
    each of 20 single-launch timings, a 3 x L2 write and then a 2 x L2 read
    leave L2 holding clean lines of other data (cold_l2_us, the median)."""
    import numpy as np
    import torch
    import collective_communication_planner_gb300 as tccl
    import datagen
    import oracle

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    st = stream.cuda_stream
    peak, _ = measured_peak()
    ncores = os.cpu_count() or 1

    def ev_stats(fn, min_ms=60.0, batches=5):
        """Per-call ms of back-to-back calls: `batches` batches, each between
        one event pair and at least min_ms / batches long (and at least 200
        calls when a call is short); returns (median, min) over the batches."""
        for _ in range(3):
            fn()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def batch(it):
            e0.record(stream)
            for _ in range(it):
                fn()
            e1.record(stream)
            e1.synchronize()
            return e0.elapsed_time(e1)

        want = min_ms / batches
        it = 1
        while True:
            ms = batch(it)
            if ms >= want or it >= 20000:
                break
            it = min(20000, max(it * 2, int(it * want / max(ms, 1e-3)) + 1))
        if ms / it < 1e-2:
            it = max(it, 200)
        per = sorted(batch(it) / it for _ in range(batches))
        return per[len(per) // 2], per[0]

    def graph_time(fn, reps=20):
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                fn()
        def replay():
            with torch.cuda.stream(stream):  # the timed stream (replay uses the current one)
                g.replay()

        t = ev_stats(replay, 30.0)[0] / reps
        del g
        return t

    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (129 << 20))
    flush_buf = torch.empty(3 * l2_bytes // 4, dtype=torch.int32, device=dev)

    # read after the flush write, so that the flush's dirty lines are written
    # back before the timed launch rather than inside it
    clean_buf = torch.zeros(2 * l2_bytes // 4, dtype=torch.int32, device=dev)

    def cold_time(fn, reps=20):
        times = []
        for _ in range(reps):
            with torch.cuda.stream(stream):
                flush_buf.fill_(1)
                clean_buf.max()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        times.sort()
        return times[len(times) // 2]

    def cpu_time(fn, min_s=0.5):
        fn()
        n, t0 = 0, time.perf_counter()
        while True:
            fn()
            n += 1
            el = time.perf_counter() - t0
            if el >= min_s:
                return el / n

    def emit(**kw):
        print(json.dumps(kw), flush=True)

    def set_cfg(g, **kw):
        c = tccl.tcclConfig_t()
        for k, v in kw.items():
            setattr(c, k, v)
        assert tccl.tcclGroupSetConfig(g.handle, c) == 0

    def copy_out_moved(row, p, nbytes):
        """Copy-out allreduce rows: every byte the call moves (the fold reads
        P x S and writes S; the copies read and write (P-1) x S) beside the
        collective's own 2 x P x S. The copies' reads of the anchor can be
        served from L2, so this can exceed the HBM peak."""
        if row["engine"] == tccl.tcclEngineCopyOut:
            moved = (p + 1) * nbytes + 2 * (p - 1) * nbytes
            row["moved_bytes_fraction"] = round(moved / (row["us"] * 1e-6) / 1e9 / peak, 4)

    def to_dev(x):
        return host_to_torch(x).to(dev)

    def run_point(cfg, g, coll, p, n, dtype, op, sends, recvs, cap=0, graph=False, sms=False):
        es = 2 if dtype == "bf16" else 4
        dt, o = tccl.DTYPES[dtype], tccl.OPS[op]
        if coll == "AR":
            # arguments marshalled once, so small calls measure the library,
            # not Python's per-call packing of pointer arrays
            prepared = g.prepare_all_reduce(sends, recvs, op=op, cta_cap=cap, stream=st)
            fn = lambda: prepared() or 0
            S, hbm = n * es, 2 * p * n * es
        elif coll == "RS":
            fn = lambda: tccl.tcclReduceScatter(g.handle, sends, recvs, n, dt, o, st, cap)
            S, hbm = p * n * es, (p + 1) * p * n * es   # S = per-rank send bytes
        else:
            fn = lambda: tccl.tcclAllGather(g.handle, sends, recvs, n, dt, st, cap)
            S, hbm = p * n * es, (p + 1) * p * n * es   # S = per-rank recv bytes
        assert fn() == 0
        info = g.last_launch()
        used = per_launch = None
        if sms:
            g.read_sm_record()
            g.record_sms(True)
            fn()
            per, used = g.read_sm_record_launches()
            per_launch = max(per) if per else 0
            g.record_sms(False)
        ms, ms_min = ev_stats(fn)
        row = dict(config=cfg, coll=coll, P=p, dtype=dtype, op=op, count=n,
                   bytes_per_rank=(n * es if coll == "AR" else S), cap=cap,
                   us=round(ms * 1e3, 3), us_min=round(ms_min * 1e3, 3),
                   algbw=round(p * (n * es if coll == "AR" else S) / (ms * 1e-3) / 1e9, 2),
                   busbw=round(S / (ms * 1e-3) * (2 if coll == "AR" else 1) * (p - 1) / p / 1e9, 2),
                   hbm_GBps=round(hbm / (ms * 1e-3) / 1e9, 1),
                   hbm_fraction=round(hbm / (ms * 1e-3) / 1e9 / peak, 4),
                   # near or below L2: back-to-back calls hit L2 and read above the HBM peak
                   l2_resident=hbm < 1.5 * l2_bytes, engine=info["engine"], ctas=info["ctas"],
                   sms_used=used, sms_per_launch_max=per_launch)
        if graph:
            row["graph_us"] = round(graph_time(fn) * 1e3, 3)
        if hbm < 3 * l2_bytes:
            # L2 honesty: the same call with L2 flushed (a write of 3 x L2)
            # before each timed launch, median of 20 single-launch timings
            cold = cold_time(fn)
            row["cold_l2_us"] = round(cold * 1e3, 3)
            row["cold_l2_hbm_fraction"] = round(hbm / (cold * 1e-3) / 1e9 / peak, 4)
        assert g.query_error() == 0
        return row

    only = set(args.sweep_configs.split(",")) if args.sweep_configs else None

    # C1
    if not only or "c1" in only:
        p, n = 2, 1_048_576
        xs = datagen.rank_buffers("uniform_f32", 0, p, n)
        g = tccl.Group(p)
        sends = [to_dev(x) for x in xs]
        recvs = [torch.empty_like(t) for t in sends]
        row = run_point("C1", g, "AR", p, n, "f32", "sum", sends, recvs, graph=True)
        row["cpu_1core_s"] = cpu_time(lambda: oracle.allreduce(xs, "f32", "sum", nthreads=1))
        row["cpu_all_s"] = cpu_time(lambda: oracle.allreduce(xs, "f32", "sum", nthreads=0))
        row["cpu_cores"] = ncores
        emit(**row)
        g.close()
    # C2
    if not only or "c2" in only:
        p, n = 4, 32 << 20
        rc = n // p
        xs = datagen.rank_buffers("normal_bf16", 1, p, n, mu=0.0, sigma=1.0)
        g = tccl.Group(p)
        sends = [to_dev(x) for x in xs]
        recvs = [torch.empty_like(t) for t in sends]
        parts = [torch.empty(rc, dtype=torch.bfloat16, device=dev) for _ in range(p)]
        row = run_point("C2", g, "AR", p, n, "bf16", "sum", sends, recvs)
        row["cpu_1core_s"] = cpu_time(lambda: oracle.allreduce(xs, "bf16", "sum", nthreads=1), 1.0)
        row["cpu_all_s"] = cpu_time(lambda: oracle.allreduce(xs, "bf16", "sum", nthreads=0))
        row["cpu_cores"] = ncores
        emit(**row)
        # reduce-scatter: Auto (the register fold) and the SM-only bulk engine,
        # uncapped and under caps
        for cap in (0, 8, 16, 32):
            emit(**run_point("C2", g, "RS", p, rc, "bf16", "sum", sends, parts, cap=cap, sms=cap > 0))
            set_cfg(g, ce_auto_max_cap=-1)
            row = run_point("C2", g, "RS", p, rc, "bf16", "sum", sends, parts, cap=cap, sms=cap > 0)
            row["variant"] = "sm_only"
            emit(**row)
            set_cfg(g)
        emit(**run_point("C2", g, "AG", p, rc, "bf16", "sum", parts, recvs))
        set_cfg(g, engine=tccl.tcclEngineCopyOut)  # the all-gather as copies only
        emit(**run_point("C2", g, "AG", p, rc, "bf16", "sum", parts, recvs, sms=True))
        set_cfg(g)
        # all-gather under caps: Auto (copies only) and the SM-only bulk engine
        for cap in (8, 16, 32):
            emit(**run_point("C2", g, "AG", p, rc, "bf16", "sum", parts, recvs, cap=cap, sms=True))
            set_cfg(g, ce_auto_max_cap=-1)
            row = run_point("C2", g, "AG", p, rc, "bf16", "sum", parts, recvs, cap=cap, sms=True)
            row["variant"] = "sm_only"
            emit(**row)
            set_cfg(g)
        g.close()
        del sends, recvs, parts
    # C3
    if not only or "c3" in only:
        p = 8
        g = tccl.Group(p)
        sizes = [4096 << k for k in range(17)]
        if args.c3_bytes:
            sizes = [int(b) for b in args.c3_bytes.split(",")]
        for nbytes in sizes:
            n = nbytes // 4
            for dtype, op in (("f32", "sum"), ("f32", "min"), ("f32", "max"), ("i32", "sum")):
                xs = (datagen.rank_buffers("uniform_f32", 2, p, n) if dtype == "f32" else
                      datagen.rank_buffers("int32", 2, p, n, lo=-1000, hi=1000))
                bufs = [to_dev(x) for x in xs]
                row = run_point("C3", g, "AR", p, n, dtype, op, bufs, bufs, graph=nbytes <= (1 << 20))
                if nbytes == (256 << 20) and op == "sum" and dtype == "f32":
                    row["cpu_1core_s"] = cpu_time(lambda: oracle.allreduce(xs, dtype, op, nthreads=1), 1.0)
                    row["cpu_all_s"] = cpu_time(lambda: oracle.allreduce(xs, dtype, op, nthreads=0))
                    row["cpu_cores"] = ncores
                emit(**row)
                del bufs
            torch.cuda.empty_cache()
        g.close()
    # C4
    if not only or "c4" in only:
        p, n = 8, 64 << 20
        xs = datagen.rank_buffers("normal_bf16", 3, p, n, mu=0.0, sigma=0.02)
        g = tccl.Group(p)
        sends = [to_dev(x) for x in xs]
        recvs = [torch.empty_like(t) for t in sends]
        for cap in (8, 16, 32, 0):
            row = run_point("C4", g, "AR", p, n, "bf16", "sum", sends, recvs, cap=cap, sms=True)
            if cap == 0:
                row["cpu_1core_s"] = cpu_time(lambda: oracle.allreduce(xs, "bf16", "sum", nthreads=1), 1.0)
                row["cpu_all_s"] = cpu_time(lambda: oracle.allreduce(xs, "bf16", "sum", nthreads=0))
                row["cpu_cores"] = ncores
            copy_out_moved(row, p, n * 2)
            emit(**row)
            if cap:
                # the same cap on the SM-only path (Auto told never to pick copy-out)
                set_cfg(g, ce_auto_max_cap=-1)
                row = run_point("C4", g, "AR", p, n, "bf16", "sum", sends, recvs, cap=cap, sms=True)
                row["variant"] = "sm_only"
                emit(**row)
                set_cfg(g)
        g.close()
        del sends, recvs
        torch.cuda.empty_cache()
    # C5
    if not only or "c5" in only:
        p = 8
        g = tccl.Group(p)
        for tokens in (1, 8, 64, 512, 4096):
            n = tokens * 8192
            xs = datagen.rank_buffers("normal_bf16", 4, p, n, mu=0.0, sigma=1.0)
            sends = [to_dev(x) for x in xs]
            recvs = [torch.empty_like(t) for t in sends]
            row = run_point("C5", g, "AR", p, n, "bf16", "sum", sends, recvs, graph=tokens <= 64)
            row["tokens"] = tokens
            if tokens == 4096:
                row["cpu_1core_s"] = cpu_time(lambda: oracle.allreduce(xs, "bf16", "sum", nthreads=1), 1.0)
                row["cpu_all_s"] = cpu_time(lambda: oracle.allreduce(xs, "bf16", "sum", nthreads=0))
                row["cpu_cores"] = ncores
            emit(**row)
        g.close()
    # the rank count at a fixed size: bf16 sum, 32 Mi elements (64 MiB) per
    # rank, uncapped and at a 16-CTA cap (Auto's engine). Timing only: the
    # inputs are torch's N(0, 1) draws, and parity at these rank counts is
    # the GPU tests' job
    if only and "vs_p" in only:
        n = 32 << 20
        for p in (2, 3, 4, 8, 16, 32, 64):
            g = tccl.Group(p)
            sends = [torch.randn(n, device=dev).to(torch.bfloat16) for _ in range(p)]
            recvs = [torch.empty_like(t) for t in sends]
            for cap in (0, 16):
                emit(**run_point("vs_P", g, "AR", p, n, "bf16", "sum", sends, recvs, cap=cap, sms=cap > 0))
            g.close()
            del sends, recvs
            torch.cuda.empty_cache()


# ------------------------------------------------------------------ overlap mode
def overlap(args):
    """Allreduce beside a concurrent GEMM (the T-CCL GEMM-overlap study, on one
    GPU): a cuBLAS bf16 GEMM loop on one stream, the C4 allreduce (P=8, bf16,
    128 MiB per rank) on another, for several CTA caps. Reports each alone,
    both together, the GEMM slowdown and the overlapped / serial speedup. The
    allreduce result under contention is checked against the oracle."""
    import numpy as np
    import torch
    import collective_communication_planner_gb300 as tccl
    import datagen
    import oracle

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = WORKLOADS["c4"]
    p, n = w["p"], w["count"]
    xs = make_inputs(w)
    if args.overlap_engine == tccl.tcclEngineTmaReduce:
        # bf16 sums round at every step in the copy hardware: use the fp32 form
        # of the same values (half the elements, same bytes per rank)
        n //= 2
        xs = [((x[:n].astype(np.uint32) << 16).view(np.float32)).copy() for x in xs]
    sends = [host_to_torch(x).to(dev) for x in xs]
    recvs = [torch.empty_like(t) for t in sends]
    dt_code = tccl.tcclFloat32 if xs[0].dtype == np.float32 else tccl.tcclBfloat16
    m = args.gemm_n
    A = torch.randn(m, m, device=dev, dtype=torch.bfloat16)
    B = torch.randn(m, m, device=dev, dtype=torch.bfloat16)
    C = torch.empty(m, m, device=dev, dtype=torch.bfloat16)
    s_g, s_c = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    g = tccl.Group(p)
    if args.overlap_engine:
        g.set_config(engine=args.overlap_engine)
    reps = args.overlap_reps
    flops = 2.0 * m ** 3
    hbm = 2 * p * n * xs[0].dtype.itemsize

    def gemm():
        with torch.cuda.stream(s_g):
            torch.matmul(A, B, out=C)

    def ar(cap):
        r = tccl.tcclAllReduce(g.handle, sends, recvs, n, dt_code, tccl.tcclSum,
                               s_c.cuda_stream, cap)
        if r != tccl.tcclSuccess:
            raise tccl.TcclError(r, "tcclAllReduce")

    def timed(fn_g, fn_c):
        torch.cuda.synchronize()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        e[0].record(s_g)
        s_c.wait_event(e[0])
        for _ in range(reps):
            if fn_g:
                fn_g()
            if fn_c:
                fn_c()
        e[1].record(s_g)
        e[2].record(s_c)
        torch.cuda.synchronize()
        return e[0].elapsed_time(e[1]), e[0].elapsed_time(e[2])

    for _ in range(3):
        gemm()
        ar(0)
    torch.cuda.synchronize()
    gemm_alone, _ = timed(gemm, None)
    idx = np.random.default_rng(1).choice(n, size=1 << 15, replace=False)
    otype = "f32" if xs[0].dtype == np.float32 else "bf16"
    exp = oracle.allreduce([x[idx].copy() for x in xs], otype, "sum")[0]
    for cap in args.overlap_caps:
        for _ in range(3):  # warm: a new cap's first call may create copy streams and events
            ar(cap)
        _, ar_alone = timed(None, lambda: ar(cap))
        for t in recvs:
            t.zero_()
        g_ms, c_ms = timed(gemm, lambda: ar(cap))
        got = recvs[3].cpu().numpy()[idx] if otype == "f32" else \
            recvs[3].view(torch.int16).cpu().numpy()[idx].view(np.uint16)
        both = max(g_ms, c_ms)
        print(json.dumps({
            "mode": "overlap", "cap": cap, "engine": g.last_launch()["engine"], "gemm": f"bf16 {m}x{m}x{m}", "reps": reps,
            "gemm_alone_ms": round(gemm_alone / reps, 4),
            "gemm_tflops_alone": round(flops / (gemm_alone / reps * 1e-3) / 1e12, 1),
            "allreduce_alone_ms": round(ar_alone / reps, 4),
            "allreduce_alone_GBps": round(hbm / (ar_alone / reps * 1e-3) / 1e9, 1),
            "gemm_with_allreduce_ms": round(g_ms / reps, 4),
            "allreduce_with_gemm_ms": round(c_ms / reps, 4),
            "allreduce_with_gemm_GBps": round(hbm / (c_ms / reps * 1e-3) / 1e9, 1),
            "gemm_slowdown": round(g_ms / gemm_alone, 3),
            "overlap_speedup_vs_serial": round((gemm_alone + ar_alone) / both, 3),
            "allreduce_correct": bool(np.array_equal(got, exp))}), flush=True)
    assert g.query_error() == tccl.tcclSuccess
    g.close()


# ------------------------------------------------------------------ reshard mode
def reshard_bench(args):
    """M-to-N reshard throughput (the M2N workload on logical ranks): an
    8192 x 8192 bf16 weight between several training and generation layouts.
    Bytes moved = each source piece read once + every destination block
    written once per replica. Results checked against the reshard oracle."""
    import numpy as np
    import torch
    import collective_communication_planner_gb300 as tccl
    import datagen
    from oracle import reshard as rs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    R = tccl.TCCL_REPLICATE
    shape = (8192, 8192)
    glob = datagen.rank_buffers("normal_bf16", 7, 1, shape[0] * shape[1])[0].reshape(shape)
    peak, _ = measured_peak()
    g = tccl.Group(64)
    cases = [("TP8 rows -> TP2xDP4 cols", ((8,), (0,)), ((4, 2), (R, 1))),
             ("TP4 rows -> TP2xDP2 rows (article example A shape)", ((1, 4), (R, 0)), ((2, 2), (R, 0))),
             ("TP8 cols -> TP8 rows", ((8,), (1,)), ((8,), (0,))),
             ("TP2 rows -> DP8 replicas", ((2,), (0,)), ((8,), (R,)))]
    stream = torch.cuda.current_stream()
    for name, src, dst in cases:
        sb = []
        for m in range(rs.nranks(src[0])):
            box = rs.local_box(shape, src[0], src[1], m)
            sb.append(np.ascontiguousarray(glob[tuple(slice(lo, hi) for lo, hi in box)]).ravel())
        exp = rs.reshard(sb, src[0], src[1], dst[0], dst[1], shape)
        sends = [host_to_torch(b).to(dev) for b in sb]
        recvs = [torch.empty(e.size, dtype=torch.bfloat16, device=dev) for e in exp]
        sl = tccl.make_layout(src[0], src[1], 0)
        dl = tccl.make_layout(dst[0], dst[1], rs.nranks(src[0]))
        r, tr, br, bw, nw = tccl.tcclReshardInspect(sl, dl, list(shape), tccl.tcclBfloat16,
                                                    sends, recvs)
        # the default (the bulk ring for these co-aligned buffers), then the
        # register-copy kernel the group uses when asked for the warp engine
        for engine in (tccl.tcclEngineAuto, tccl.tcclEngineWarp):
            c = tccl.tcclConfig_t()
            c.engine = engine
            assert tccl.tcclGroupSetConfig(g.handle, c) == tccl.tcclSuccess
            for t in recvs:
                t.zero_()
            fn = lambda: g.reshard(sends, sl, recvs, dl, shape)
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                fn()
            e1.record(stream)
            e1.synchronize()
            ms = e0.elapsed_time(e1) / args.steps
            info = g.last_launch()
            ok = all(np.array_equal(t.view(torch.int16).cpu().numpy().view(np.uint16), e)
                     for t, e in zip(recvs, exp))
            print(json.dumps({"mode": "reshard", "case": name, "tensor": "bf16 8192x8192",
                              "engine": "bulk ring" if info["engine"] == tccl.tcclEngineBulk else "warp copies",
                              "ctas": info["ctas"], "transfers": len(tr), "windows": nw, "bytes_read": br,
                              "bytes_written": bw, "us": round(ms * 1e3, 2),
                              "GBps": round((br + bw) / (ms * 1e-3) / 1e9, 1),
                              "hbm_fraction": round((br + bw) / (ms * 1e-3) / 1e9 / peak, 4),
                              "correct": ok}), flush=True)
        del sends, recvs
    assert g.query_error() == tccl.tcclSuccess
    g.close()


# ------------------------------------------------------------------ rmsnorm mode
def rmsnorm_bench(args):
    """The allreduce fused with RMSNorm against the plain allreduce, on the
    C5 shapes (P=8, bf16 [tokens, 8192]): device time per op (and per op in a
    CUDA graph for small token counts), GB/s of 2*P*S + gamma bytes. Results
    checked against the RMSNorm oracle (within one bf16 ulp)."""
    import numpy as np
    import torch
    import collective_communication_planner_gb300 as tccl
    import datagen
    from oracle import rmsnorm as rn

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    p, hidden = 8, 8192
    g = tccl.Group(p)
    os.environ["TCCL_RMSNORM_CLUSTER"] = "0"  # a second group with one CTA per row, for comparison
    g_row = tccl.Group(p)
    del os.environ["TCCL_RMSNORM_CLUSTER"]
    stream = torch.cuda.current_stream()
    peak, _ = measured_peak()
    gamma_h = datagen.rank_buffers("normal_bf16", 104, 1, hidden)[0]
    gamma = host_to_torch(gamma_h).to(dev)

    def ev(fn, reps):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / reps

    def graph_us(fn):
        s2 = torch.cuda.Stream()
        with torch.cuda.stream(s2):
            fn()
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s2):
            for _ in range(20):
                fn()
        return ev(gr.replay, 20) / 20 * 1e3

    for tokens in (int(t) for t in args.rmsnorm_tokens.split(",")):
        n = tokens * hidden
        xs = datagen.rank_buffers("normal_bf16", 4, p, n)
        exp, exp64 = rn.allreduce_rmsnorm(xs, gamma_h, tokens, hidden, 1e-6, "bf16")
        sends = [host_to_torch(x).to(dev).view(tokens, hidden) for x in xs]
        recvs = [torch.empty_like(t) for t in sends]
        fused = lambda: g.all_reduce_rmsnorm(sends, recvs, gamma)
        fused_row = lambda: g_row.all_reduce_rmsnorm(sends, recvs, gamma)
        plain = lambda: g.all_reduce(sends, recvs)
        reps = 200 if tokens <= 64 else 30
        f_ms, p_ms = ev(fused, reps), ev(plain, reps)
        fused()
        info = g.last_launch()
        torch.cuda.synchronize()
        got = recvs[5].view(torch.int16).cpu().numpy().ravel().view(np.uint16)
        d = np.abs(got.astype(np.int64) - exp.astype(np.int64))
        row = {"mode": "rmsnorm", "P": p, "tokens": tokens, "hidden": hidden,
               "fused_us": round(f_ms * 1e3, 2), "allreduce_us": round(p_ms * 1e3, 2),
               "fused_hbm_fraction": round((2 * p * n * 2 + hidden * 2) / (f_ms * 1e-3) / 1e9 / peak, 4),
               "max_ulp": int(d.max()), "ulp_mismatches": int(np.count_nonzero(d)),
               "fused_ctas": info["ctas"]}
        if tokens <= 64:
            row["fused_graph_us"] = round(graph_us(fused), 2)
            row["fused_one_cta_per_row_graph_us"] = round(graph_us(fused_row), 2)
            row["allreduce_graph_us"] = round(graph_us(plain), 2)
        print(json.dumps(row), flush=True)
    assert g.query_error() == tccl.tcclSuccess and g_row.query_error() == tccl.tcclSuccess
    g.close()
    g_row.close()


# ------------------------------------------------------------------ host-cost mode
def build_host_cost() -> Path:
    """Compiles tests/host_cost.cu (a C++ program that calls the C ABI) against the
    in-tree libtccl.so; returns the executable's path."""
    pkg = ROOT / "collective_communication_planner_gb300"
    out = pkg / "_build" / "host_cost"
    out.parent.mkdir(exist_ok=True)
    subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                           f"-I{ROOT / 'include'}", str(ROOT / "tests" / "host_cost.cu"), "-o", str(out),
                           f"-L{pkg}", "-ltccl", "-Xlinker", "-rpath", "-Xlinker", str(pkg)])
    return out


def host_cost(args):
    """Per-call host cost of tcclAllReduce from C++ (no ctypes): enqueue time,
    device time and graph-replay time for decode-sized messages, beside the
    empty-kernel launch floor. One JSON line per case."""
    exe = build_host_cost()
    r = subprocess.run([str(exe), str(args.host_cost_batches)], capture_output=True, text=True)
    sys.stdout.write(r.stdout)
    if r.returncode != 0:
        raise SystemExit(f"host-cost program failed ({r.returncode}): {r.stderr.strip()}")


# ------------------------------------------------------------------ TMA-reduce mode
def tma_reduce_bench(args):
    """The TMA-reduce engine (the copy hardware applies the reduction) beside
    the bulk engine's register fold: fp32 sum allreduce of 64 MiB per rank,
    out of place, P = 4 and 8, uncapped and under caps, ascending and arrival
    order. Device time per call (CUDA events over back-to-back calls), HBM
    fraction of 2 * P * S, sampled parity against the oracle. A fixed number
    of launches per line, so the command also serves ncu."""
    import numpy as np
    import torch
    import collective_communication_planner_gb300 as tccl
    import datagen
    import oracle

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    st = stream.cuda_stream
    peak, _ = measured_peak()
    n = (64 << 20) // 4
    for p in [int(x) for x in args.tma_reduce_ranks.split(",")]:
        xs = datagen.rank_buffers("uniform_f32", 2, p, n)
        sends = [torch.from_numpy(x).to(dev) for x in xs]
        recvs = [torch.empty_like(t) for t in sends]
        idx = np.sort(np.random.default_rng(9).choice(n, size=4096, replace=False))
        exp = oracle.allreduce([x[idx].copy() for x in xs], "f32", "sum")[0]
        g = tccl.Group(p)
        shapes = [tuple(int(v) for v in sh.split(":")) for sh in args.tma_reduce_shapes.split(",")] \
            if args.tma_reduce_shapes else [(0, 0)]
        runs = [(tccl.tcclEngineBulk, 0, 0, 0)]
        for slots, chunk in shapes:
            runs += [(tccl.tcclEngineTmaReduce, 0, slots, chunk), (tccl.tcclEngineTmaReduce, 1, slots, chunk)]
        for cap in [int(c) for c in args.tma_reduce_caps.split(",")]:
            for engine, order, slots, chunk in runs:
                c = tccl.tcclConfig_t()
                c.engine, c.reduce_order = engine, order
                c.reduce_slots, c.max_chunk_bytes = slots, chunk
                assert tccl.tcclGroupSetConfig(g.handle, c) == 0
                for t in recvs:
                    t.fill_(0)
                call = lambda: tccl.tcclAllReduce(g.handle, sends, recvs, n, tccl.tcclFloat32,
                                                  tccl.tcclSum, st, cap)
                for _ in range(3):
                    assert call() == 0
                stream.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(10):
                    assert call() == 0
                e1.record(stream)
                e1.synchronize()
                ms = e0.elapsed_time(e1) / 10
                info = g.last_launch()
                got = recvs[p - 1].cpu().numpy()[idx]
                exact = bool(np.array_equal(got.view(np.uint32), exp.view(np.uint32)))
                print(json.dumps({"mode": "tma_reduce", "P": p, "bytes_per_rank": n * 4, "cap": cap,
                                  "engine": "tma_reduce" if engine == tccl.tcclEngineTmaReduce else "bulk",
                                  "order": "arrival" if order else "ascending", "ctas": info["ctas"],
                                  "threads": info["threads"], "chunk_bytes": info["chunk_bytes"],
                                  "stages": info["stages"], "us": round(ms * 1e3, 2),
                                  "hbm_fraction": round(2 * p * n * 4 / (ms * 1e-3) / 1e9 / peak, 4),
                                  "sampled_exact": exact}), flush=True)
        assert g.query_error() == tccl.tcclSuccess
        g.close()
        del sends, recvs


# ------------------------------------------------------------------ copy-out mode
def copy_out_bench(args):
    """An allreduce workload (default C4: P=8, bf16, 128 MiB per rank) at CTA
    caps (default 8, 16 and 32) with the default engine choice (the copy-out
    engine) and other variants (the SM-only bulk engine, the TMA-fed fold,
    segment and copy-stream schedules): device time per call, HBM fraction of
    the 2*P*S bytes, segments and copies per call. Results checked against the
    oracle on sampled elements. A small, fixed number of launches, so the
    command also serves for an ncu launch list."""
    import numpy as np
    import torch
    import collective_communication_planner_gb300 as tccl

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.copy_out_workload]
    p, n = w["p"], w["count"]
    es = 2 if w["dtype"] == "bf16" else 4
    xs = make_inputs(w)
    sends = [host_to_torch(x).to(dev) for x in xs]
    recvs = [torch.empty_like(t) for t in sends]
    stream = torch.cuda.current_stream()
    st = stream.cuda_stream
    peak, _ = measured_peak()
    g = tccl.Group(p)
    alg = 2 * p * n * es

    def set_cfg(**kw):
        c = tccl.tcclConfig_t()
        for k, v in kw.items():
            setattr(c, k, v)
        assert tccl.tcclGroupSetConfig(g.handle, c) == 0

    import oracle
    idx = np.sort(np.random.default_rng(5).choice(n, size=4096, replace=False))
    exp = oracle.allreduce([x[idx].copy() for x in xs], w["dtype"], w["op"])[0]
    variants = {
        "auto": {},
        "sm_only": {"ce_auto_max_cap": -1},
        # the copy-out engine with its segments folded by the bulk engine's
        # TMA pipeline instead of register loads
        "tma_shared": {"ce_fold": 2},
        "tma_per_rank": {"ce_fold": 2, "stage_layout": 2},
        "tma_per_rank_8w": {"ce_fold": 2, "stage_layout": 2, "consumer_warps": 8},
        # the segment schedule: a shorter last segment (its copies overlap no
        # fold), more segments, fewer copy streams
        "tail30": {"ce_tail_percent": 30},
        "tail45": {"ce_tail_percent": 45},
        "tail60": {"ce_tail_percent": 60},
        "seg16": {"ce_segment_bytes": 16 << 20},
        "seg16_tail45": {"ce_segment_bytes": 16 << 20, "ce_tail_percent": 45},
        "streams1": {"ce_streams": 1},
        "streams2": {"ce_streams": 2},
        # allreduce copy streams: (each segment but the last, the last)
        "ar1_tail4": {"ce_ar_streams": 1, "ce_tail_streams": 4},
        "ar2_tail2": {"ce_ar_streams": 2, "ce_tail_streams": 2},
        "ar2_tail4": {"ce_ar_streams": 2, "ce_tail_streams": 4},
        "ar3_tail3": {"ce_ar_streams": 3, "ce_tail_streams": 3},
        "ar3_tail4": {"ce_ar_streams": 3, "ce_tail_streams": 4},
        "ar2_tail6": {"ce_streams": 6, "ce_ar_streams": 2, "ce_tail_streams": 6},
        "seg20": {"ce_segment_bytes": 20 << 20},
        "seg24": {"ce_segment_bytes": 24 << 20},
        "seg28": {"ce_segment_bytes": 28 << 20},
        "seg26": {"ce_segment_bytes": 26 << 20},
        "seg8": {"ce_segment_bytes": 8 << 20},
        "seg12": {"ce_segment_bytes": 12 << 20},
        "seg14": {"ce_segment_bytes": 14 << 20},
        "seg30": {"ce_segment_bytes": 30 << 20},
        "seg32": {"ce_segment_bytes": 32 << 20},
        "seg36": {"ce_segment_bytes": 36 << 20},
        # the copy-out engine whatever the cap (Auto stops at ce_auto_max_cap)
        "copy_out": {"engine": 5},
        # segments bulk-reduced into the anchor by the TMA-reduce engine (the
        # pairs it supports), Auto's cap rule / whatever the cap
        "tma_reduce_fold": {"ce_fold": 3},
        "copy_out_tma_reduce": {"engine": 5, "ce_fold": 3},
        "tma_reduce": {"engine": 4},
    }
    chosen = args.copy_out_variants.split(",") if args.copy_out_variants else ["auto", "sm_only"]
    caps = [int(c) for c in args.copy_out_caps.split(",")]
    for cap in caps:
        for variant in chosen:
            kw = variants[variant]
            set_cfg(**kw)
            call = lambda: tccl.tcclAllReduce(g.handle, sends, recvs, n, tccl.DTYPES[w["dtype"]],
                                              tccl.OPS[w["op"]], st, cap)
            for t in recvs:
                t.fill_(0)
            for _ in range(3):
                assert call() == 0
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(10):
                assert call() == 0
            e1.record(stream)
            e1.synchronize()
            ms = e0.elapsed_time(e1) / 10
            info = g.last_launch()
            got = recvs[p - 1].view(torch.int16 if es == 2 else recvs[0].dtype).cpu().numpy()[idx].view(exp.dtype)
            print(json.dumps({"mode": "copy_out", "workload": w["name"], "cap": cap, "variant": variant,
                              "engine": info["engine"], "ctas": info["ctas"], "threads": info["threads"],
                              "stages": info["stages"], "chunk_bytes": info["chunk_bytes"],
                              "stage_layout": info["stage_layout"],
                              "segments": info["ce_segments"], "copies": info["ce_copies"],
                              "us": round(ms * 1e3, 2), "hbm_fraction": round(alg / (ms * 1e-3) / 1e9 / peak, 4),
                              "sampled_exact": bool(np.array_equal(got, exp))}), flush=True)
    assert g.query_error() == tccl.tcclSuccess
    g.close()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="c4")
    ap.add_argument("--no-caps", action="store_true",
                    help="skip the capped points (CTA caps 8/16/32) and the C2 comparison")
    ap.add_argument("--cap", type=int, default=None, help="CTA cap (default: the workload's)")
    ap.add_argument("--soak", type=float, default=1.0, help="seconds of untimed load first")
    ap.add_argument("--cpu-seconds", type=float, default=2.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="measure every configuration point of C1..C5 (one JSON line each)")
    ap.add_argument("--sweep-configs", default="",
                    help="comma list, e.g. c3,c5 (default c1..c5); vs_p: allreduce over P = 2..64 at "
                         "64 MiB per rank, uncapped and at cap 16")
    ap.add_argument("--c3-bytes", default="",
                    help="C3 sizes per rank in bytes for --sweep, comma separated (default 4 KiB ... 256 MiB)")
    ap.add_argument("--overlap", action="store_true",
                    help="allreduce beside a concurrent cuBLAS GEMM, across CTA caps")
    ap.add_argument("--rmsnorm-tokens", default="1,8,64,512,4096",
                    help="token counts (rows of 8192) for --rmsnorm, comma separated")
    ap.add_argument("--e2e-pieces", type=int, default=2,
                    help="slices per end-to-end step (host copies overlap the other slices' reductions)")
    ap.add_argument("--reshard", action="store_true",
                    help="M-to-N reshard throughput on an 8192 x 8192 bf16 weight")
    ap.add_argument("--rmsnorm", action="store_true",
                    help="allreduce fused with RMSNorm vs the plain allreduce (C5 shapes)")
    ap.add_argument("--copy-out", action="store_true",
                    help="C4 at CTA caps 8/16/32: copy-out engine vs SM-only bulk engine")
    ap.add_argument("--copy-out-variants", default="",
                    help="for --copy-out: comma list of auto, sm_only, tma_shared, tma_per_rank, "
                         "tma_per_rank_8w, tail30, tail45, tail60, seg16, seg16_tail45, streams1, "
                         "streams2 (default auto,sm_only)")
    ap.add_argument("--copy-out-caps", default="8,16,32", help="for --copy-out: CTA caps")
    ap.add_argument("--copy-out-workload", choices=sorted(WORKLOADS), default="c4",
                    help="for --copy-out: the allreduce workload")
    ap.add_argument("--host-cost", action="store_true",
                    help="per-call host cost of tcclAllReduce from a C++ program (decode-sized messages)")
    ap.add_argument("--host-cost-batches", type=int, default=50)
    ap.add_argument("--tma-reduce", action="store_true",
                    help="TMA-reduce engine vs the bulk engine, fp32 sum, 64 MiB per rank")
    ap.add_argument("--tma-reduce-ranks", default="4,8")
    ap.add_argument("--tma-reduce-caps", default="0,32,16")
    ap.add_argument("--tma-reduce-shapes", default="",
                    help="TMA-reduce shapes slots:chunk_bytes, comma separated (default: the library's)")
    ap.add_argument("--gemm-n", type=int, default=8192)
    ap.add_argument("--overlap-engine", type=int, default=0,
                    help="engine for the overlap study (0 auto, 1 bulk, 4 TMA-reduce)")
    ap.add_argument("--overlap-reps", type=int, default=20)
    ap.add_argument("--overlap-caps", type=lambda v: [int(x) for x in v.split(",")],
                    default=[8, 16, 32, 64, 0])
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    w = WORKLOADS[args.workload]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist_mod.init_process_group("gloo")
        dist = dist_mod

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w)), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return

    import __graft_entry__
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if args.sweep:
        sweep(args)
        return
    if args.overlap:
        overlap(args)
        return
    if args.reshard:
        reshard_bench(args)
        return
    if args.rmsnorm:
        rmsnorm_bench(args)
        return
    if args.copy_out:
        copy_out_bench(args)
        return
    if args.host_cost:
        host_cost(args)
        return
    if args.tma_reduce:
        tma_reduce_bench(args)
        return
    if dist is not None:
        dist.barrier()
    out = run_ours(args, w, rank, world, dist)
    if out is not None:
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
