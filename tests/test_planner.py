"""Planner and lowering, checked on the host through tcclPlanInspect.

Invariants (no GPU needed):
  * every destination byte is written by exactly one window, and from the
    right source bytes (AR: same offset; RS: shard s of every send buffer;
    AG: rank k's send buffer into block k);
  * body windows are 16-byte co-aligned in every buffer they touch and a
    multiple of 16 bytes; edges and non co-aligned tasks run element-wise;
  * the bulk engine never uses more CTAs than the cap, windows are grouped by
    CTA, and the pipeline fits in shared memory;
  * logical tasks: AR = P shard-ins + P shard-outs (each after its shard-in),
    RS = P shard-ins, AG = P shard-outs;
  * argument validation matches the header.
"""
import itertools

import pytest

import collective_communication_planner_gb300 as tccl

AR, RS, AG = tccl.COLL_ALLREDUCE, tccl.COLL_REDUCE_SCATTER, tccl.COLL_ALLGATHER
ES = {tccl.tcclFloat32: 4, tccl.tcclBfloat16: 2, tccl.tcclInt32: 4}
BASE = 1 << 40  # fake device addresses, far apart


def bufs(p, nbytes_send, nbytes_recv, send_mis=0, recv_mis=0, in_place=None, coll=AR,
         shard_bytes=0):
    stride = 1 << 34
    send = [BASE + 2 * r * stride + (send_mis if isinstance(send_mis, int) else send_mis[r])
            for r in range(p)]
    recv = [BASE + (2 * r + 1) * stride + (recv_mis if isinstance(recv_mis, int) else recv_mis[r])
            for r in range(p)]
    if in_place:
        if coll == AR:
            recv = list(send)
        elif coll == RS:
            recv = [send[r] + r * shard_bytes for r in range(p)]
        else:
            send = [recv[r] + r * shard_bytes for r in range(p)]
    return send, recv


def cfg(engine=0, store=0, stage_bytes=0, stages=0, small_max_bytes=0):
    c = tccl.tcclConfig_t()
    c.engine = engine
    c.store_mode = store
    c.stage_bytes = stage_bytes
    c.stages = stages
    c.small_max_bytes = small_max_bytes
    return c


def inspect(coll, p, count, dt, send, recv, cap=0, engine=0, sm=152, smem=232448,
            max_windows=8192, **kw):
    r, wins, ntasks, info = tccl.tcclPlanInspect(coll, p, send, recv, count, dt, cap, sm, smem,
                                                 cfg(engine, **kw), max_windows=max_windows)
    return r, wins, ntasks, info


def check_cover(coll, p, count, es, send, recv, wins, info):
    """Exactly-once coverage of every destination byte with the right source."""
    if coll == AR:
        dst_len = count * es
    elif coll == RS:
        dst_len = count * es
    else:
        dst_len = p * count * es
    covered = {r: [] for r in range(p)}
    for w in wins:
        assert w["bytes"] > 0 and w["bytes"] % es == 0
        dranks = range(p) if w["dst_sel"] < 0 else [w["dst_sel"]]
        sranks = range(p) if w["src_sel"] < 0 else [w["src_sel"]]
        for d in dranks:
            covered[d].append((w["dst_off"], w["dst_off"] + w["bytes"]))
        if coll == AR:
            assert w["src_sel"] == -1 and w["dst_sel"] == -1 or p == 1
            assert w["src_off"] == w["dst_off"]
        elif coll == RS:
            s = w["dst_sel"] if p > 1 else 0
            assert w["src_sel"] == -1 or p == 1
            assert w["src_off"] == s * count * es + w["dst_off"]
        else:
            k = w["src_sel"] if p > 1 else 0
            assert w["dst_sel"] == -1 or p == 1
            assert w["dst_off"] == k * count * es + w["src_off"]
        if not w["scalar"]:
            assert w["bytes"] % 16 == 0
            for s in sranks:
                assert (send[s] + w["src_off"]) % 16 == 0
            for d in dranks:
                assert (recv[d] + w["dst_off"]) % 16 == 0
    for r in range(p):
        iv = sorted(covered[r])
        pos = 0
        for b, e in iv:
            assert b == pos, (r, b, pos)
            pos = e
        assert pos == dst_len
    if info.engine == tccl.tcclEngineBulk:
        # body windows first (shared chunk sequence), then element-wise
        # windows grouped by the CTA that runs them
        body = [w for w in wins if not w["scalar"]]
        assert wins[:len(body)] == body and all(w["cta"] == -1 for w in body)
        ctas = [w["cta"] for w in wins[len(body):]]
        assert ctas == sorted(ctas)
        assert all(0 <= c < info.ctas for c in ctas)
        assert info.total_chunks == sum(-(-w["bytes"] // info.chunk_bytes) for w in body)
        assert info.smem_bytes <= 232448
        assert info.stages >= 2 and info.chunk_bytes % 16 == 0
        assert info.ctas >= 1


CASES = list(itertools.product([AR, RS, AG], [1, 2, 3, 4, 8, 64],
                               [0, 1, 7, 8, 1000, 4096 + 3, 1 << 20],
                               [tccl.tcclFloat32, tccl.tcclBfloat16]))


@pytest.mark.parametrize("coll,p,count,dt", CASES)
@pytest.mark.parametrize("engine", [tccl.tcclEngineBulk, tccl.tcclEngineWarp, tccl.tcclEngineVec])
def test_exact_cover_aligned(coll, p, count, dt, engine):
    es = ES[dt]
    send, recv = bufs(p, 0, 0)
    r, wins, ntasks, info = inspect(coll, p, count, dt, send, recv, engine=engine)
    assert r == tccl.tcclSuccess
    if count == 0:
        assert wins == [] and ntasks == 0
        return
    check_cover(coll, p, count, es, send, recv, wins, info)


@pytest.mark.parametrize("coll", [AR, RS, AG])
@pytest.mark.parametrize("mis", [(4, 4), (8, 8), (4, 12), (2, 2), (6, 6), "mixed"])
@pytest.mark.parametrize("engine", [tccl.tcclEngineBulk, tccl.tcclEngineVec])
def test_exact_cover_misaligned(coll, mis, engine):
    p, count, dt = 4, 10_001, tccl.tcclBfloat16
    if mis == "mixed":
        send, recv = bufs(p, 0, 0, send_mis=[0, 2, 4, 6], recv_mis=[2, 2, 2, 2])
    else:
        send, recv = bufs(p, 0, 0, send_mis=mis[0], recv_mis=mis[1])
    r, wins, _, info = inspect(coll, p, count, dt, send, recv, engine=engine)
    assert r == tccl.tcclSuccess
    check_cover(coll, p, count, 2, send, recv, wins, info)
    if mis != "mixed" and mis[0] == mis[1] and coll == AR:
        # co-aligned: at most a scalar head and tail per shard
        assert sum(w["bytes"] for w in wins if w["scalar"]) <= 2 * 16 * p
    if mis == (4, 12) and coll == AR:
        assert all(w["scalar"] for w in wins)


@pytest.mark.parametrize("coll", [AR, RS, AG])
def test_exact_cover_in_place(coll):
    p, count, dt = 8, 33_333, tccl.tcclFloat32
    send, recv = bufs(p, 0, 0, in_place=True, coll=coll, shard_bytes=count * 4)
    r, wins, _, info = inspect(coll, p, count, dt, send, recv, engine=tccl.tcclEngineBulk)
    assert r == tccl.tcclSuccess
    check_cover(coll, p, count, 4, send, recv, wins, info)


@pytest.mark.parametrize("cap", [1, 2, 8, 9, 16, 32, 151, 152, 1000])
def test_cta_cap_bounds_the_grid(cap):
    p, count = 8, 64 << 20
    send, recv = bufs(p, 0, 0)
    for engine in (tccl.tcclEngineBulk, tccl.tcclEngineVec, tccl.tcclEngineWarp):
        r, wins, _, info = inspect(AR, p, count, tccl.tcclBfloat16, send, recv, cap=cap,
                                   engine=engine, max_windows=4096)
        assert r == tccl.tcclSuccess
        assert 1 <= info.ctas <= min(cap, 152 * 8)
        if engine == tccl.tcclEngineBulk:
            assert info.ctas == min(cap, 152)
            check_cover(AR, p, count, 2, send, recv, wins, info)


def chunk_owners(total, grid, order):
    """Which CTA runs each chunk, as the kernel's chunk cursor walks them."""
    owner = [None] * total
    per = -(-total // grid)
    for j in range(grid):
        seq = range(j, total, grid) if order == tccl.tcclOrderCyclic else \
            range(j * per, min((j + 1) * per, total))
        for c in seq:
            assert owner[c] is None
            owner[c] = j
    return owner


@pytest.mark.parametrize("order", [tccl.tcclOrderCyclic, tccl.tcclOrderBlocked])
@pytest.mark.parametrize("count", [1000, 1 << 20, 64 << 20, (64 << 20) + 7])
@pytest.mark.parametrize("cap", [0, 16])
def test_bulk_chunk_sequence_is_covered_once_and_balanced(order, count, cap):
    p = 8
    send, recv = bufs(p, 0, 0)
    c = cfg(tccl.tcclEngineBulk)
    c.chunk_order = order
    r, wins, _, info = tccl.tcclPlanInspect(AR, p, send, recv, count, tccl.tcclBfloat16, cap, 152,
                                            232448, c)
    assert r == 0 and info.chunk_order == order
    body = [w for w in wins if not w["scalar"]]
    assert len(body) == 1  # co-aligned allreduce: the shard bodies merge into one window
    owner = chunk_owners(info.total_chunks, info.ctas, order)
    assert None not in owner
    loads = [owner.count(j) for j in range(info.ctas)]
    assert max(loads) - min(loads) <= (1 if order == tccl.tcclOrderCyclic else max(loads))
    assert info.ctas <= (cap or 152)


def test_task_structure():
    p = 4
    send, recv = bufs(p, 0, 0)
    for coll, exp in ((AR, 2 * p), (RS, p), (AG, p)):
        r, _, ntasks, info = inspect(coll, p, 1000, tccl.tcclFloat32, send, recv)
        assert r == 0 and ntasks == exp and info.tasks == exp
    # allreduce with fewer elements than ranks: empty shards get no tasks
    r, wins, ntasks, _ = inspect(AR, 8, 3, tccl.tcclFloat32, *bufs(8, 0, 0))
    assert r == 0 and ntasks == 2


def test_auto_engine_choice():
    p = 8
    send, recv = bufs(p, 0, 0)
    r, _, _, info = inspect(AR, p, 8192, tccl.tcclBfloat16, send, send)  # 16 KiB per rank, in place
    assert info.engine == tccl.tcclEngineWarp
    r, _, _, info = inspect(AR, p, 1 << 20, tccl.tcclBfloat16, send, recv)  # 2 MiB per rank
    assert info.engine == tccl.tcclEngineVec
    r, _, _, info = inspect(AR, p, 1 << 20, tccl.tcclBfloat16, send, recv, cap=16)
    assert info.engine == tccl.tcclEngineBulk  # capped mid-size calls keep the TMA pipeline
    r, _, _, info = inspect(AR, p, 64 << 20, tccl.tcclBfloat16, send, recv)
    assert info.engine == tccl.tcclEngineBulk
    assert info.chunk_order == tccl.tcclOrderDynamic and info.store_mode == tccl.tcclStoreBulk
    r, _, _, info = inspect(AR, p, 64 << 20, tccl.tcclBfloat16, send, recv, cap=16)
    assert info.chunk_order == tccl.tcclOrderCyclic and info.store_mode == tccl.tcclStoreVec
    r, _, _, info = inspect(AR, 40, 1024, tccl.tcclFloat32, *bufs(40, 0, 0),
                            engine=tccl.tcclEngineWarp)
    assert info.engine == tccl.tcclEngineVec  # more ranks than lanes


def test_small_engine_switch_by_rank_count():
    # the warp engine up to 64 KiB per rank at P >= 5 and up to 128 KiB below;
    # the vec engine above, up to 192 lanes per SM in one CTA per SM of the
    # lanes / SMs rounded up to a warp, else in CTAs of 256
    sms = 152
    for p, kib, exp in ((9, 64, tccl.tcclEngineWarp), (8, 96, tccl.tcclEngineVec),
                        (8, 128, tccl.tcclEngineVec), (16, 128, tccl.tcclEngineVec),
                        (4, 128, tccl.tcclEngineWarp), (6, 128, tccl.tcclEngineVec),
                        (6, 64, tccl.tcclEngineWarp), (3, 128, tccl.tcclEngineWarp),
                        (4, 192, tccl.tcclEngineVec), (8, 256, tccl.tcclEngineVec),
                        (8, 384, tccl.tcclEngineVec), (8, 512, tccl.tcclEngineVec),
                        (8, 2048, tccl.tcclEngineVec)):
        send, recv = bufs(p, 0, 0)
        r, _, _, info = inspect(AR, p, kib * 512, tccl.tcclBfloat16, send, recv, sm=sms)
        assert r == 0 and info.engine == exp, (p, kib, info.engine)
        lanes = kib * 1024 // 16
        if exp == tccl.tcclEngineVec and lanes <= sms * 192:
            per_sm = -(-lanes // sms)
            threads = max(32, -(-per_sm // 32) * 32)
            assert info.threads == threads and info.ctas == -(-lanes // threads) <= sms, (p, kib, info.threads)
        elif exp == tccl.tcclEngineVec:
            assert info.threads == 256 and info.ctas == min(-(-lanes // 256), 8 * sms), (p, kib, info.ctas)
        else:
            assert info.threads == 256
    send, recv = bufs(8, 0, 0)
    r, _, _, info = inspect(AR, 8, 1 << 16, tccl.tcclBfloat16, send, recv)  # 128 KiB: 8192 lanes
    assert info.engine == tccl.tcclEngineVec and info.threads == 64 and info.ctas == 128
    r, _, _, info = inspect(AR, 8, 1 << 18, tccl.tcclBfloat16, send, recv)  # 512 KiB
    assert info.engine == tccl.tcclEngineVec and info.threads == 256 and info.ctas == 128
    r, _, _, info = inspect(AR, 8, 1 << 20, tccl.tcclBfloat16, send, recv)  # 2 MiB
    assert info.engine == tccl.tcclEngineVec and info.threads == 256 and info.ctas == 512
    # an explicit threshold wins over the rank-count default
    r, _, _, info = inspect(AR, 8, 1 << 16, tccl.tcclBfloat16, send, recv, small_max_bytes=128 << 10)
    assert info.engine == tccl.tcclEngineWarp


def test_out_of_place_allreduce_over_8_ranks_takes_the_vec_engine():
    # at P = 8 an out-of-place allreduce goes to the vec engine at every small size;
    # in place, other collectives, other rank counts and an explicit threshold keep the warp engine
    for kib in (1, 4, 16, 64):
        r, _, _, info = inspect(AR, 8, kib * 512, tccl.tcclBfloat16, *bufs(8, 0, 0))
        assert r == 0 and info.engine == tccl.tcclEngineVec, kib
        r, _, _, info = inspect(AR, 8, kib * 512, tccl.tcclBfloat16, *bufs(8, 0, 0, in_place=True))
        assert r == 0 and info.engine == tccl.tcclEngineWarp, kib
    r, _, _, info = inspect(AR, 7, 8192, tccl.tcclBfloat16, *bufs(7, 0, 0))
    assert info.engine == tccl.tcclEngineWarp
    r, _, _, info = inspect(RS, 8, 1024, tccl.tcclBfloat16, *bufs(8, 0, 0))
    assert info.engine == tccl.tcclEngineWarp
    r, _, _, info = inspect(AR, 8, 8192, tccl.tcclBfloat16, *bufs(8, 0, 0), small_max_bytes=64 << 10)
    assert info.engine == tccl.tcclEngineWarp


def test_small_engine_switch_edges():
    # the default switch-over follows the rank count: P = 4 keeps 128 KiB, P = 5 and 9 take 64 KiB
    for p, kib, exp in ((4, 128, tccl.tcclEngineWarp), (4, 129, tccl.tcclEngineVec),
                        (5, 64, tccl.tcclEngineWarp), (5, 65, tccl.tcclEngineVec),
                        (9, 64, tccl.tcclEngineWarp), (9, 65, tccl.tcclEngineVec)):
        send, recv = bufs(p, 0, 0)
        r, _, _, info = inspect(AR, p, kib * 256, tccl.tcclFloat32, send, recv)
        assert r == 0 and info.engine == exp, (p, kib, info.engine)
    # a capped call of any size keeps off the vec engine
    send, recv = bufs(8, 0, 0)
    r, _, _, info = inspect(AR, 8, 1 << 16, tccl.tcclBfloat16, send, recv, cap=16)
    assert info.engine == tccl.tcclEngineBulk


@pytest.mark.parametrize("sms", [132, 152, 160])
def test_vec_grid_follows_sm_count(sms):
    # one CTA per SM up to 192 lanes per SM of this device, CTAs of 256 above
    send, recv = bufs(8, 0, 0)
    for lanes in (sms * 192, sms * 192 + 32):
        r, _, _, info = inspect(AR, 8, lanes * 4, tccl.tcclFloat32, send, recv, sm=sms,
                                engine=tccl.tcclEngineVec)
        assert r == 0 and info.engine == tccl.tcclEngineVec
        if lanes <= sms * 192:
            assert info.threads == 192 and info.ctas == sms, (sms, lanes, info.threads, info.ctas)
        else:
            assert info.threads == 256 and info.ctas == -(-lanes // 256), (sms, lanes, info.threads)


def test_pipeline_shape_follows_shared_memory():
    send, recv = bufs(8, 0, 0)
    r, _, _, info = inspect(AR, 8, 1 << 24, tccl.tcclBfloat16, send, recv,
                            engine=tccl.tcclEngineBulk, stage_bytes=32768, stages=32)
    # uncapped allreduce: bulk stores, so two 4 KiB result slots share the budget
    assert info.chunk_bytes == 4096 and info.stages == (232448 - 1024 - 2 * 4096) // 32768
    r, _, _, small = inspect(AR, 8, 1 << 24, tccl.tcclBfloat16, send, recv,
                             engine=tccl.tcclEngineBulk, smem=48 * 1024)
    assert small.smem_bytes <= 48 * 1024 and small.stages >= 2


@pytest.mark.parametrize("p,chunk,stages", [(1, 16384, 6), (2, 16384, 3), (3, 16384, 2), (4, 12288, 2),
                                             (8, 6144, 2), (16, 6144, 2), (32, 3072, 2)])
def test_uncapped_allreduce_default_shape(p, chunk, stages):
    """With the default shape a large out-of-place allreduce (2 * P * S of
    512 MiB or more) sizes its ring for about 96 KiB of loads per CTA, in
    6 KiB chunks or more: stages * P * chunk stays within 96 KiB unless two
    stages need more."""
    send, recv = bufs(p, 0, 0)
    count = -(-(512 << 20) // (2 * p * 2))  # bf16: exactly at the threshold
    r, wins, _, info = inspect(AR, p, count, tccl.tcclBfloat16, send, recv, engine=tccl.tcclEngineBulk)
    assert r == 0 and info.stage_layout == tccl.tcclLayoutShared
    assert (info.chunk_bytes, info.stages) == (chunk, stages)
    assert stages == 2 or stages * p * chunk <= 96 * 1024
    check_cover(AR, p, count, 2, send, recv, wins, info)


@pytest.mark.parametrize("p", [2, 4, 8])
def test_other_calls_keep_the_full_ring(p):
    """The 96 KiB rule is for large, uncapped, out-of-place allreduce only: a
    reduce-scatter, a capped or in-place or smaller allreduce and an
    explicitly set shape fill shared memory."""
    send, recv = bufs(p, 0, 0)
    big = (512 << 20) // (2 * p * 2)
    full = lambda info: info.smem_bytes > 150 * 1024
    ring = lambda info: info.chunk_bytes == min(16384, 65536 // p)
    r, _, _, rs = inspect(RS, p, big, tccl.tcclBfloat16, send, recv, engine=tccl.tcclEngineBulk)
    assert r == 0 and full(rs) and ring(rs)
    r, _, _, capped = inspect(AR, p, big, tccl.tcclBfloat16, send, recv, cap=16,
                              engine=tccl.tcclEngineBulk)
    assert r == 0 and full(capped)
    r, _, _, explicit = inspect(AR, p, big, tccl.tcclBfloat16, send, recv, engine=tccl.tcclEngineBulk,
                                stage_bytes=65536, stages=7)
    assert r == 0 and full(explicit) and ring(explicit)
    r, _, _, small = inspect(AR, p, big - 8, tccl.tcclBfloat16, send, recv, engine=tccl.tcclEngineBulk)
    assert r == 0 and full(small) and ring(small)
    r, _, _, inpl = inspect(AR, p, big, tccl.tcclBfloat16, send, list(send), engine=tccl.tcclEngineBulk)
    assert r == 0 and full(inpl) and ring(inpl)
    mixed = list(send)
    mixed[-1] = recv[-1]  # one rank out of place: the call is not in place
    r, _, _, part = inspect(AR, p, big, tccl.tcclBfloat16, send, mixed, engine=tccl.tcclEngineBulk)
    assert r == 0 and not full(part)


@pytest.mark.parametrize("p", [2, 8, 64])
@pytest.mark.parametrize("cw", [8, 16])
def test_per_rank_stage_layout_shape(p, cw):
    send, recv = bufs(p, 0, 0)
    c = cfg(tccl.tcclEngineBulk)
    c.stage_layout = tccl.tcclLayoutPerRank
    c.consumer_warps = cw
    r, wins, _, info = tccl.tcclPlanInspect(AR, p, send, recv, 1 << 22, tccl.tcclBfloat16, 0,
                                            152, 232448, c)
    assert r == 0 and info.stage_layout == tccl.tcclLayoutPerRank
    # a stage is one rank's chunk: 4 vectors per consumer thread, whatever P is
    assert info.chunk_bytes == 16 * 4 * 32 * cw
    assert info.store_mode == tccl.tcclStoreVec
    assert info.smem_bytes == 1024 + info.stages * info.chunk_bytes <= 232448
    check_cover(AR, p, 1 << 22, 2, send, recv, wins, info)
    # all-gather keeps the shared layout (a single source)
    r, _, _, info = tccl.tcclPlanInspect(AG, p, send, recv, 1 << 16, tccl.tcclBfloat16, 0, 152,
                                         232448, c)
    assert info.stage_layout == tccl.tcclLayoutShared


def test_auto_layout_switches_to_per_rank_for_many_ranks():
    for p, exp in ((8, tccl.tcclLayoutShared), (16, tccl.tcclLayoutShared),
                   (32, tccl.tcclLayoutShared), (33, tccl.tcclLayoutPerRank),
                   (64, tccl.tcclLayoutPerRank)):
        send, recv = bufs(p, 0, 0)
        r, _, _, info = tccl.tcclPlanInspect(AR, p, send, recv, 1 << 22, tccl.tcclBfloat16, 0,
                                             152, 232448, cfg(tccl.tcclEngineBulk))
        assert r == 0 and info.stage_layout == exp, p


@pytest.mark.parametrize("coll", [AR, RS])
@pytest.mark.parametrize("p", [1, 2, 8])
def test_tma_reduce_engine_shape(coll, p):
    send, recv = bufs(p, 0, 0)
    r, wins, _, info = inspect(coll, p, 1_000_003, tccl.tcclFloat32, send, recv,
                               engine=tccl.tcclEngineTmaReduce)
    assert r == 0 and info.engine == tccl.tcclEngineTmaReduce
    lanes = info.threads // 32
    # default shape: 8 KiB chunks, 4 slots per issuing thread, two buffers per
    # slot (three for a reduce-scatter), within the shared memory and the
    # head's 120 barriers
    bufs_per_slot = 3 if coll == RS else 2
    assert info.chunk_bytes == 8192 and info.stages == 4
    assert info.smem_bytes == 1024 + lanes * 4 * bufs_per_slot * 8192 <= 232448
    assert lanes * 4 * bufs_per_slot <= 120
    assert info.ctas <= -(-info.total_chunks // (lanes * 4))
    check_cover(coll, p, 1_000_003, 4, send, recv, wins, info)


@pytest.mark.parametrize("slots,chunk", [(1, 8192), (2, 8192), (8, 2048), (4, 12288)])
def test_tma_reduce_engine_shape_knobs(slots, chunk):
    """reduce_slots and max_chunk_bytes set the TMA-reduce shape; the lanes
    fill what the shared memory and the barrier head allow."""
    p = 8
    send, recv = bufs(p, 0, 0)
    c = cfg(tccl.tcclEngineTmaReduce)
    c.reduce_slots = slots
    c.max_chunk_bytes = chunk
    r, wins, _, info = tccl.tcclPlanInspect(AR, p, send, recv, 3_000_001, tccl.tcclFloat32, 0, 152,
                                            232448, c)
    assert r == 0 and info.stages == slots and info.chunk_bytes == chunk
    lanes = info.threads // 32
    assert 1 <= lanes <= 16 and lanes * slots * 2 <= 120
    assert info.smem_bytes == 1024 + lanes * slots * 2 * chunk <= 232448


@pytest.mark.parametrize("slots", [1, 2, 4, 8])
def test_tma_reduce_slot_walk_covers_every_chunk(slots):
    """The TMA-reduce kernel's chunk walk: lane w of CTA b starts at
    b * lanes + w, takes `slots` chunks `step = grid * lanes` apart, then
    moves on by step * slots. Every chunk is taken exactly once."""
    for total in (1, 5, 100, 1000, 4097):
        for grid in (1, 3, 152):
            for lanes in (1, 7, 16):
                seen = set()
                step = grid * lanes
                for b in range(grid):
                    for w in range(lanes):
                        base = b * lanes + w
                        while base < total:
                            for j in range(slots):
                                c = base + j * step
                                if c >= total:
                                    break
                                assert c not in seen
                                seen.add(c)
                            base += step * slots
                assert seen == set(range(total)), (total, grid, lanes, slots)


def test_tma_reduce_engine_rejects_allgather():
    send, recv = bufs(4, 0, 0)
    r, *_ = inspect(AG, 4, 1000, tccl.tcclFloat32, send, recv, engine=tccl.tcclEngineTmaReduce)
    assert r == tccl.tcclInvalidUsage


def test_consumer_warps_are_capped_at_sixteen():
    send, recv = bufs(4, 0, 0)
    c = cfg(tccl.tcclEngineBulk)
    c.consumer_warps = 31
    r, _, _, info = tccl.tcclPlanInspect(AR, 4, send, recv, 1 << 22, tccl.tcclBfloat16, 0, 152,
                                         232448, c)
    assert info.threads == 32 * 17


# ------------------------------------------------------------------ validation
def test_rejects_null_and_misaligned_pointers():
    p = 2
    send, recv = bufs(p, 0, 0)
    for coll in (AR, RS, AG):
        r, *_ = inspect(coll, p, 16, tccl.tcclFloat32, [send[0], 0], recv)
        assert r == tccl.tcclInvalidArgument
        r, *_ = inspect(coll, p, 16, tccl.tcclFloat32, send, [recv[0] + 2, recv[1]])
        assert r == tccl.tcclInvalidArgument
        r, *_ = inspect(coll, p, 16, tccl.tcclBfloat16, send, [recv[0] + 2, recv[1]])
        assert r == tccl.tcclSuccess


def test_rejects_bad_enums_and_rank_counts():
    send, recv = bufs(2, 0, 0)
    r, *_ = inspect(AR, 2, 16, 7, send, recv)
    assert r == tccl.tcclInvalidArgument
    r, *_ = tccl.tcclPlanInspect(3, 2, send, recv, 16, 0)
    assert r == tccl.tcclInvalidArgument
    r, *_ = tccl.tcclPlanInspect(AR, 0, [], [], 16, 0)
    assert r == tccl.tcclInvalidArgument
    r, *_ = tccl.tcclPlanInspect(AR, 65, [BASE] * 65, [BASE] * 65, 16, 0)
    assert r == tccl.tcclInvalidArgument


def test_overlap_rules():
    p, count, es = 4, 1000, 4
    send, recv = bufs(p, 0, 0)
    # recv overlapping another rank's recv
    bad = list(recv)
    bad[1] = recv[0] + 64
    assert inspect(AR, p, count, 0, send, bad)[0] == tccl.tcclInvalidArgument
    # recv partially overlapping its own send (not the in-place form)
    bad = list(recv)
    bad[2] = send[2] + 16
    assert inspect(AR, p, count, 0, send, bad)[0] == tccl.tcclInvalidArgument
    # recv overlapping another rank's send
    bad = list(recv)
    bad[0] = send[1]
    assert inspect(AR, p, count, 0, send, bad)[0] == tccl.tcclInvalidArgument
    # send buffers may alias each other (read only)
    assert inspect(AR, p, count, 0, [send[0]] * p, recv)[0] == tccl.tcclSuccess
    # in-place forms are accepted; mixing in-place and out-of-place too
    mixed = list(recv)
    mixed[1] = send[1]
    assert inspect(AR, p, count, 0, send, mixed)[0] == tccl.tcclSuccess
    s, r_ = bufs(p, 0, 0, in_place=True, coll=RS, shard_bytes=count * es)
    assert inspect(RS, p, count, 0, s, r_)[0] == tccl.tcclSuccess
    r_bad = list(r_)
    r_bad[1] = s[1]  # shard 0 of rank 1's send, not shard 1
    assert inspect(RS, p, count, 0, s, r_bad)[0] == tccl.tcclInvalidArgument
    s, r_ = bufs(p, 0, 0, in_place=True, coll=AG, shard_bytes=count * es)
    assert inspect(AG, p, count, 0, s, r_)[0] == tccl.tcclSuccess
    s_bad = list(s)
    s_bad[0] = r_[0] + 4
    assert inspect(AG, p, count, 0, s_bad, r_)[0] == tccl.tcclInvalidArgument


def test_count_zero_is_success_without_work():
    send, recv = bufs(4, 0, 0)
    r, wins, nt, info = inspect(AR, 4, 0, 0, send, recv)
    assert r == tccl.tcclSuccess and wins == [] and nt == 0 and info.ctas == 0


def test_count_overflow_rejected():
    send, recv = bufs(8, 0, 0)
    r, *_ = inspect(RS, 8, (1 << 62), 0, send, recv)
    assert r == tccl.tcclInvalidArgument
