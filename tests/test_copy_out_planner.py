"""The copy-out engine's host decisions, checked through tcclCopyOutInspect
(no GPU needed): when Auto picks the engine, how an allreduce is cut into
segments, and when the register-load fold takes the shard-in."""
import itertools

import pytest

import collective_communication_planner_gb300 as tccl

AR, RS, AG = tccl.COLL_ALLREDUCE, tccl.COLL_REDUCE_SCATTER, tccl.COLL_ALLGATHER
BF16, F32 = tccl.tcclBfloat16, tccl.tcclFloat32
ES = {BF16: 2, F32: 4}
MiB = 1 << 20
BASE = 1 << 40
SMS = 152


def bufs(p, send_mis=0, recv_mis=0):
    stride = 1 << 36
    send = [BASE + 2 * r * stride + (send_mis[r] if isinstance(send_mis, list) else send_mis) for r in range(p)]
    recv = [BASE + (2 * r + 1) * stride + (recv_mis[r] if isinstance(recv_mis, list) else recv_mis)
            for r in range(p)]
    return send, recv


def inspect(coll, p, count, dt=BF16, cap=0, cfg=None, send_mis=0, recv_mis=0, sm_count=SMS):
    return inspect_wide(coll, p, count, dt, cap, cfg, send_mis, recv_mis, sm_count)[:4]


def inspect_wide(coll, p, count, dt=BF16, cap=0, cfg=None, send_mis=0, recv_mis=0, sm_count=SMS):
    send, recv = bufs(p, send_mis, recv_mis)
    r, co, rf, ns, se, wf = tccl.tcclCopyOutInspect(coll, p, send, recv, count, dt, cap, sm_count, cfg)
    assert r == tccl.tcclSuccess, tccl.tcclGetErrorString(r)
    return co, rf, ns, se, wf


def config(**kw):
    c = tccl.tcclConfig_t()
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def per_rank_bytes(coll, p, count, es):
    return count * es * (1 if coll == AR else p)


def auto_max_cap(p):
    return SMS * 4 // 7 if p <= 2 else (SMS * 5 // 12 if p <= 4 else SMS * 7 // 16)


@pytest.mark.parametrize("coll,p,mib,cap", list(itertools.product(
    [AR, RS, AG], [1, 2, 3, 4, 5, 8], [2, 4, 64], [0, 8, 47, 63, 64, 66, 67, 86, 87])))
def test_auto_choice(coll, p, mib, cap):
    """Auto's rule: P >= 2 and at least 4 MiB per rank buffer; allreduce and
    all-gather under a cap of at most 4/7 of the SMs for P <= 2 (86 of 152),
    5/12 for P = 3 and 4 (63), 7/16 for P >= 5 (66); reduce-scatter under any
    cap, or uncapped for P <= 4."""
    es = 2
    count = mib * MiB // es // (1 if coll == AR else p)
    co, rf, ns, se = inspect(coll, p, count, cap=cap)
    big = per_rank_bytes(coll, p, count, es) >= 4 * MiB
    if p < 2 or not big:
        want = False
    elif coll == RS:
        # the register fold takes a reduce-scatter whose shards are whole 16-byte vectors
        want = (cap > 0 or p <= 4) and count * es % 16 == 0
    else:
        want = 0 < cap <= auto_max_cap(p)
    assert bool(co) == want, (coll, p, mib, cap, co)
    if not co:
        assert (rf, ns, se) == (0, 0, 0)


def test_engine_setting_and_auto_limit():
    p, count = 8, 64 * MiB // 2
    # copy-out chosen explicitly: every allreduce / all-gather with P >= 2
    assert inspect(AR, p, 1000, cfg=config(engine=tccl.tcclEngineCopyOut))[0] == 1
    assert inspect(AG, p, 1000, cfg=config(engine=tccl.tcclEngineCopyOut))[0] == 1
    assert inspect(AR, 1, count, cfg=config(engine=tccl.tcclEngineCopyOut))[0] == 0
    # another explicit engine: never
    assert inspect(AR, p, count, cap=16, cfg=config(engine=tccl.tcclEngineBulk))[0] == 0
    # Auto switched off, or with a wider limit
    assert inspect(AR, p, count, cap=16, cfg=config(ce_auto_max_cap=-1))[0] == 0
    assert inspect(RS, p, count // p, cap=16, cfg=config(ce_auto_max_cap=-1))[0] == 0
    assert inspect(AR, p, count, cap=100, cfg=config(ce_auto_max_cap=100))[0] == 1
    assert inspect(AR, p, count, cap=101, cfg=config(ce_auto_max_cap=100))[0] == 0
    # the limit scales with the device: 132 SMs -> 132 * 7 // 16 = 57 for P = 8
    assert inspect(AR, p, count, cap=57, sm_count=132)[0] == 1
    assert inspect(AR, p, count, cap=58, sm_count=132)[0] == 0


@pytest.mark.parametrize("dt", [BF16, F32])
@pytest.mark.parametrize("count_bytes", [4 * MiB + 16, 16 * MiB, 64 * MiB, 128 * MiB + 512,
                                         1024 * MiB, 3 * 1024 * MiB + 256])
@pytest.mark.parametrize("seg_cfg", [0, 8 * MiB, 4096])
def test_segments(dt, count_bytes, seg_cfg):
    """Segments cover the call, start at multiples of 256 bytes, are at most
    ce_segment_bytes (28 MiB by default) unless that would need more than 64
    of them, and number at least four while each stays >= 4 MiB."""
    es = ES[dt]
    count = count_bytes // es
    cfg = config(engine=tccl.tcclEngineCopyOut, ce_segment_bytes=seg_cfg)
    co, rf, ns, se = inspect(AR, 4, count, dt=dt, cfg=cfg)
    assert co == 1 and rf == 1
    assert (se * es) % 256 == 0 and se > 0
    assert ns == -(-count // se) and 1 <= ns <= 64
    cap_bytes = seg_cfg or 28 * MiB
    if ns < 64:  # not grown to respect the 64-segment bound
        assert se * es == 256 or se * es <= min(cap_bytes, max(4 * MiB, -(-count_bytes // 4)))
    if cap_bytes >= 4 * MiB and count_bytes >= 16 * MiB:
        assert ns >= 4 and se * es >= min(4 * MiB, cap_bytes)


def test_segment_count_bound_grows_segments():
    co, rf, ns, se = inspect(AR, 2, (1 << 30), dt=F32, cfg=config(engine=tccl.tcclEngineCopyOut,
                                                                   ce_segment_bytes=4096))
    assert ns == 64 and se * 4 >= (1 << 32) // 64


@pytest.mark.parametrize("send_mis,recv_mis,fold", [
    (0, 0, True), (4, 4, True), (6, 6, True), (4, 0, False), (0, 2, False),
    ([0, 0, 0, 4], 0, False), (0, [0, 4, 4, 4], True)])
def test_register_fold_for_allreduce(send_mis, recv_mis, fold):
    """The allreduce's fold needs every send buffer co-aligned (mod 16) with
    rank 0's receive buffer, the anchor; the other receive buffers are only
    written by the copy engines, so their alignment does not matter."""
    co, rf, ns, se = inspect(AR, 4, 8 * MiB, cap=16, send_mis=send_mis, recv_mis=recv_mis)
    assert co == 1 and rf == int(fold)


@pytest.mark.parametrize("ce_fold,fold", [(0, True), (1, True), (2, False), (3, False)])
def test_fold_choice_follows_the_config(ce_fold, fold):
    """ce_fold = 2 asks for the TMA pipeline and 3 for the TMA-reduce engine
    even where the register fold could run; 0 and 1 keep the register fold
    for co-aligned buffers."""
    co, rf, ns, se = inspect(AR, 8, 64 * MiB, cap=16, cfg=config(ce_fold=ce_fold))
    assert co == 1 and rf == int(fold)
    assert tccl.tcclCopyOutInspect(AR, 8, *bufs(8), 1 << 20, BF16, 16, SMS,
                                   config(ce_fold=4))[0] == tccl.tcclInvalidArgument


@pytest.mark.parametrize("rc_bytes,send_mis,recv_mis,fold", [
    (1 * MiB, 0, 0, True), (1 * MiB, 6, 6, True), (1 * MiB + 2, 0, 0, False),
    (1 * MiB, 4, 0, False), (1 * MiB, 0, [0, 0, 8, 0], False)])
def test_register_fold_for_reduce_scatter(rc_bytes, send_mis, recv_mis, fold):
    """Reduce-scatter's fold writes every rank, so every buffer must be
    co-aligned and a shard a multiple of 16 bytes; otherwise the bulk engine
    runs it and the inspect reports no copy-out at all."""
    co, rf, ns, se = inspect(RS, 4, rc_bytes // 2, cap=8, send_mis=send_mis, recv_mis=recv_mis)
    assert (co, rf) == ((1, 1) if fold else (0, 0))
    assert (ns, se) == ((1, rc_bytes // 2) if fold else (0, 0))


def test_all_gather_is_copies_only():
    co, rf, ns, se = inspect(AG, 8, 1 * MiB, cap=8)
    assert (co, rf, ns, se) == (1, 0, 0, 0)


def test_errors_and_empty_calls():
    send, recv = bufs(4)
    r = tccl.tcclCopyOutInspect(AR, 4, send, recv, 0, BF16, 8, SMS)
    assert r[0] == tccl.tcclSuccess and r[1:] == (0, 0, 0, 0, 0)
    # overlapping receive buffers are rejected exactly as the call would be
    r = tccl.tcclCopyOutInspect(AR, 4, send, [recv[0]] * 4, 1 << 20, BF16, 8, SMS)
    assert r[0] == tccl.tcclInvalidArgument
    assert tccl.tcclCopyOutInspect(AR, 4, send, recv, 1 << 20, BF16, 8, 0)[0] == tccl.tcclInvalidArgument
    assert tccl.tcclCopyOutInspect(AR, 4, send, recv, 1 << 20, 7, 8, SMS)[0] == tccl.tcclInvalidArgument


@pytest.mark.parametrize("pct", [30, 45, 60, 100])
@pytest.mark.parametrize("mib", [16, 128, 1000])
def test_short_last_segment(pct, mib):
    """ce_tail_percent keeps the number of segments and cuts the last one to
    about that share of the others (which grow to cover the rest)."""
    es = 2
    count = mib * MiB // es
    _, _, ns0, se0 = inspect(AR, 8, count, cap=16)
    co, rf, ns, se = inspect(AR, 8, count, cap=16, cfg=config(ce_tail_percent=pct))
    assert co == 1 and ns == ns0
    last = count - (ns - 1) * se
    assert se * es % 256 == 0 and 0 < last <= se
    last0 = count - (ns0 - 1) * se0
    if pct == 100 or last0 <= pct / 100 * se0:
        # equal segments, or the equal split's ragged last one is short enough already
        assert se == se0
    else:
        assert se >= se0
        # the last segment is pct % of the others, to within the 256-byte rounding of each
        assert abs(last - pct / 100 * se) <= ns * 256 // es, (last, se)


@pytest.mark.parametrize("p", [2, 3, 5, 8, 9, 12, 16, 17])
@pytest.mark.parametrize("mis", [0, 2, 18])
def test_wide_folds_allreduce(p, mis):
    """The fold reads with 256-bit loads for P = 2 to 8 and multiples of 4,
    when every source and the anchor's destination is 32-byte aligned past
    the head. bf16 buffers 2 bytes past a 32-byte boundary have a 14-byte
    head that ends 16 bytes short of one (128-bit loads); 18 bytes past it,
    the head ends on one. Segments of 28 MiB keep that for every segment."""
    co, rf, ns, se, wf = inspect_wide(AR, p, 64 * MiB, cap=16, send_mis=mis, recv_mis=mis)
    assert co == 1 and rf == 1 and ns >= 4
    rank_ok = 2 <= p <= 8 or p % 4 == 0
    assert wf == (ns if rank_ok and mis in (0, 18) else 0), (p, mis, ns, wf)


def test_wide_folds_follow_each_segment():
    """Segments are whole multiples of 256 bytes (a requested 4 MiB + 16 is
    rounded down), so every segment starts as aligned as the buffers and
    all of them take the 256-bit loads."""
    seg_bytes = 4 * MiB + 16
    co, rf, ns, se, wf = inspect_wide(AR, 8, 8 * seg_bytes // 2, cap=8,
                                      cfg=config(ce_segment_bytes=seg_bytes))
    assert co == 1 and rf == 1 and se * 2 == 4 * MiB and ns == 9
    assert wf == ns


@pytest.mark.parametrize("p,rc_bytes,wide", [(4, 1 * MiB, 1), (4, 1 * MiB + 16, 0), (9, 1 * MiB, 0),
                                             (16, 64 * 1024, 1), (3, 32, 1)])
def test_wide_folds_reduce_scatter(p, rc_bytes, wide):
    """Reduce-scatter: every job (shard j of each send buffer) must stay
    32-byte aligned, so the shard size must be a multiple of 32 bytes."""
    co, rf, ns, se, wf = inspect_wide(RS, p, rc_bytes // 2, cap=8,
                                      cfg=config(engine=tccl.tcclEngineCopyOut))
    assert co == 1 and rf == 1 and wf == wide

