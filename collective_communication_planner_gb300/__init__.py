"""Python binding of libtccl: NCCL-semantics collectives over P logical ranks
held as separate buffers in one GB300's memory.

Argument marshalling only. Every step of a collective runs in the library's
own kernels; there is no Python or CPU fallback, and importing this module on
a machine where ``libtccl.so`` has not been built raises ``ImportError``.

The functions named like the C entry points (``tcclGroupCreate``,
``tcclAllReduce``, ...) take and return the same things as ``include/tccl.h``
(device pointers as ints, a ``cudaStream_t`` as an int) and return the
``tcclResult_t`` code. ``Group`` wraps them for torch tensors.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

_HERE = Path(__file__).resolve().parent
LIB_PATH = _HERE / "libtccl.so"

tcclSuccess, tcclInvalidArgument, tcclInvalidUsage = 0, 1, 2
tcclCudaError, tcclDeviceTimeout, tcclInternalError = 3, 4, 5
tcclFloat32, tcclBfloat16, tcclInt32 = 0, 1, 2
tcclSum, tcclMin, tcclMax = 0, 1, 2
tcclEngineAuto, tcclEngineBulk, tcclEngineWarp, tcclEngineVec, tcclEngineTmaReduce = 0, 1, 2, 3, 4
tcclEngineCopyOut = 5
tcclStoreAuto, tcclStoreBulk, tcclStoreVec = 0, 1, 2
tcclOrderAuto, tcclOrderBlocked, tcclOrderCyclic, tcclOrderDynamic = 0, 1, 2, 3
tcclReduceAscending, tcclReduceArrival = 0, 1
tcclLayoutAuto, tcclLayoutShared, tcclLayoutPerRank = 0, 1, 2
TCCL_MAX_RANKS = 64

COLL_ALLREDUCE, COLL_REDUCE_SCATTER, COLL_ALLGATHER = 0, 1, 2

DTYPES = {"f32": tcclFloat32, "bf16": tcclBfloat16, "i32": tcclInt32}
OPS = {"sum": tcclSum, "min": tcclMin, "max": tcclMax}


class tcclConfig_t(ctypes.Structure):
    _fields_ = [("engine", ctypes.c_int), ("small_max_bytes", ctypes.c_size_t),
                ("vec_max_bytes", ctypes.c_size_t),
                ("stage_bytes", ctypes.c_int), ("stages", ctypes.c_int),
                ("store_mode", ctypes.c_int), ("consumer_warps", ctypes.c_int),
                ("ctas_per_sm", ctypes.c_int), ("wait_timeout_ms", ctypes.c_double),
                ("chunk_order", ctypes.c_int), ("prefetch_chunks", ctypes.c_int),
                ("load_policy", ctypes.c_int), ("max_chunk_bytes", ctypes.c_size_t),
                ("stage_layout", ctypes.c_int), ("ce_streams", ctypes.c_int),
                ("ce_segment_bytes", ctypes.c_size_t), ("ce_auto_max_cap", ctypes.c_int),
                ("reduce_order", ctypes.c_int), ("ce_fold", ctypes.c_int),
                ("ce_tail_percent", ctypes.c_int), ("reduce_slots", ctypes.c_int),
                ("ce_ar_streams", ctypes.c_int), ("ce_tail_streams", ctypes.c_int)]


class tcclLaunchInfo_t(ctypes.Structure):
    _fields_ = [("engine", ctypes.c_int), ("store_mode", ctypes.c_int), ("ctas", ctypes.c_int),
                ("threads", ctypes.c_int), ("stages", ctypes.c_int),
                ("chunk_bytes", ctypes.c_int), ("windows", ctypes.c_int),
                ("tasks", ctypes.c_int), ("smem_bytes", ctypes.c_size_t),
                ("chunk_order", ctypes.c_int), ("total_chunks", ctypes.c_uint64),
                ("stage_layout", ctypes.c_int), ("ce_segments", ctypes.c_int),
                ("ce_copies", ctypes.c_int),
                ("ce_wide_folds", ctypes.c_int)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


TCCL_REPLICATE = -1


class tcclLayout_t(ctypes.Structure):
    _fields_ = [("ndims", ctypes.c_int), ("dims", ctypes.c_int * 4),
                ("start_rank", ctypes.c_int), ("placements", ctypes.c_int * 4)]


def make_layout(dims, placements, start_rank=0) -> tcclLayout_t:
    """A mesh of `dims` (row-major rank order) from `start_rank`, one placement
    per mesh axis: TCCL_REPLICATE or the tensor dimension that axis shards."""
    lay = tcclLayout_t()
    lay.ndims = len(dims)
    for i, v in enumerate(dims):
        lay.dims[i] = v
    for i in range(4):
        lay.placements[i] = placements[i] if i < len(placements) else TCCL_REPLICATE
    lay.start_rank = start_rank
    return lay


def _open():
    if not LIB_PATH.exists():
        raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                          "(the collectives have no fallback implementation)")
    lib = ctypes.CDLL(str(LIB_PATH))
    vp, pvp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)
    i, sz = ctypes.c_int, ctypes.c_size_t
    sig = {
        "tcclGetErrorString": (ctypes.c_char_p, [i]),
        "tcclGetVersion": (i, [ctypes.POINTER(i)]),
        "tcclGroupCreate": (i, [i, pvp]),
        "tcclGroupDestroy": (i, [vp]),
        "tcclGroupGetConfig": (i, [vp, ctypes.POINTER(tcclConfig_t)]),
        "tcclGroupSetConfig": (i, [vp, ctypes.POINTER(tcclConfig_t)]),
        "tcclAllReduce": (i, [vp, pvp, pvp, sz, i, i, vp, i]),
        "tcclReduceScatter": (i, [vp, pvp, pvp, sz, i, i, vp, i]),
        "tcclAllGather": (i, [vp, pvp, pvp, sz, i, vp, i]),
        "tcclGroupQueryError": (i, [vp, ctypes.POINTER(i)]),
        "tcclGetLastLaunchInfo": (i, [vp, ctypes.POINTER(tcclLaunchInfo_t)]),
        "tcclGroupRecordSms": (i, [vp, i]),
        "tcclGroupReadSmRecord": (i, [vp, ctypes.POINTER(i)]),
        "tcclGroupReadSmRecordLaunches": (i, [vp, ctypes.POINTER(i), i, ctypes.POINTER(i),
                                              ctypes.POINTER(i)]),
        "tcclPlanInspect": (i, [i, i, pvp, pvp, sz, i, i, i, i, ctypes.POINTER(tcclConfig_t),
                                ctypes.POINTER(ctypes.c_int64), i, ctypes.POINTER(i),
                                ctypes.POINTER(i), ctypes.POINTER(tcclLaunchInfo_t)]),
        "tcclGroupInjectWaitTimeout": (i, [vp, i, ctypes.c_double]),
        "tcclCopyOutInspect": (i, [i, i, pvp, pvp, sz, i, i, i, ctypes.POINTER(tcclConfig_t),
                                   ctypes.POINTER(i), ctypes.POINTER(i), ctypes.POINTER(i),
                                   ctypes.POINTER(sz), ctypes.POINTER(i)]),
        "tcclAllReduceNoAlloc": (i, [i, pvp, pvp, sz, i, i, vp, i]),
        "tcclAllReduceRMSNorm": (i, [vp, pvp, pvp, sz, sz, vp, ctypes.c_float, i, vp, i]),
        "tcclReshard": (i, [vp, pvp, ctypes.POINTER(tcclLayout_t), pvp,
                            ctypes.POINTER(tcclLayout_t), i, ctypes.POINTER(sz), i, vp, i]),
        "tcclReshardInspect": (i, [ctypes.POINTER(tcclLayout_t), ctypes.POINTER(tcclLayout_t), i,
                                   ctypes.POINTER(sz), i, pvp, pvp, i, i,
                                   ctypes.POINTER(ctypes.c_int64), i, ctypes.POINTER(i),
                                   ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64),
                                   ctypes.POINTER(i)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _open()

EXPORTED = ("tcclGetErrorString", "tcclGetVersion", "tcclGroupCreate", "tcclGroupDestroy",
            "tcclGroupGetConfig", "tcclGroupSetConfig", "tcclAllReduce", "tcclReduceScatter",
            "tcclAllGather", "tcclGroupQueryError", "tcclGetLastLaunchInfo",
            "tcclGroupRecordSms", "tcclGroupReadSmRecord", "tcclGroupReadSmRecordLaunches",
            "tcclPlanInspect", "tcclCopyOutInspect",
            "tcclGroupInjectWaitTimeout", "tcclAllReduceNoAlloc", "tcclReshard",
            "tcclReshardInspect", "tcclAllReduceRMSNorm")


def _ptr(x) -> int:
    if isinstance(x, int):
        return x
    if x is None:
        return 0
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return int(x)


def _ptr_array(bufs):
    arr = (ctypes.c_void_p * len(bufs))(*[_ptr(b) for b in bufs])
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), arr


def _stream(s) -> int:
    if s is None:
        return 0
    if isinstance(s, int):
        return s
    return s.cuda_stream


# ---------------------------------------------------------------- same-name calls
def tcclGetErrorString(r: int) -> str:
    return _lib.tcclGetErrorString(r).decode()


def tcclGetVersion() -> int:
    v = ctypes.c_int()
    _check(_lib.tcclGetVersion(ctypes.byref(v)))
    return v.value


def tcclGroupCreate(nranks: int):
    """Returns (result, handle)."""
    h = ctypes.c_void_p()
    r = _lib.tcclGroupCreate(nranks, ctypes.byref(h))
    return r, h


def tcclGroupDestroy(group) -> int:
    return _lib.tcclGroupDestroy(group)


def tcclGroupGetConfig(group):
    c = tcclConfig_t()
    r = _lib.tcclGroupGetConfig(group, ctypes.byref(c))
    return r, c


def tcclGroupSetConfig(group, cfg: tcclConfig_t) -> int:
    return _lib.tcclGroupSetConfig(group, ctypes.byref(cfg))


def tcclAllReduce(group, sendbufs, recvbufs, count, datatype, op, stream=None, cta_cap=0) -> int:
    sp, _k1 = _ptr_array(sendbufs)
    rp, _k2 = _ptr_array(recvbufs)
    return _lib.tcclAllReduce(group, sp, rp, count, datatype, op, _stream(stream), cta_cap)


def tcclReduceScatter(group, sendbufs, recvbufs, recvcount, datatype, op, stream=None,
                      cta_cap=0) -> int:
    sp, _k1 = _ptr_array(sendbufs)
    rp, _k2 = _ptr_array(recvbufs)
    return _lib.tcclReduceScatter(group, sp, rp, recvcount, datatype, op, _stream(stream),
                                  cta_cap)


def tcclAllGather(group, sendbufs, recvbufs, sendcount, datatype, stream=None, cta_cap=0) -> int:
    sp, _k1 = _ptr_array(sendbufs)
    rp, _k2 = _ptr_array(recvbufs)
    return _lib.tcclAllGather(group, sp, rp, sendcount, datatype, _stream(stream), cta_cap)


def tcclGroupQueryError(group):
    s = ctypes.c_int()
    r = _lib.tcclGroupQueryError(group, ctypes.byref(s))
    return r, s.value


def tcclGetLastLaunchInfo(group):
    info = tcclLaunchInfo_t()
    r = _lib.tcclGetLastLaunchInfo(group, ctypes.byref(info))
    return r, info


def tcclAllReduceNoAlloc(nranks, sendbufs, recvbufs, count, datatype, op, stream=None,
                         cta_cap=0) -> int:
    """Allreduce without a group, for callers that cannot allocate GPU memory
    (its scratch is a static device array; see include/tccl.h)."""
    sp, _k1 = _ptr_array(sendbufs)
    rp, _k2 = _ptr_array(recvbufs)
    return _lib.tcclAllReduceNoAlloc(nranks, sp, rp, count, datatype, op, _stream(stream), cta_cap)


def tcclAllReduceRMSNorm(group, sendbufs, recvbufs, rows, hidden, gamma, eps, datatype,
                         stream=None, cta_cap=0) -> int:
    sp, _k1 = _ptr_array(sendbufs)
    rp, _k2 = _ptr_array(recvbufs)
    return _lib.tcclAllReduceRMSNorm(group, sp, rp, rows, hidden, _ptr(gamma), float(eps),
                                     datatype, _stream(stream), cta_cap)


def _shape(shape):
    return (ctypes.c_size_t * len(shape))(*shape)


def tcclReshard(group, srcbufs, src_layout, dstbufs, dst_layout, shape, datatype, stream=None,
                cta_cap=0) -> int:
    sp, _k1 = _ptr_array(srcbufs)
    dp, _k2 = _ptr_array(dstbufs)
    return _lib.tcclReshard(group, sp, ctypes.byref(src_layout), dp, ctypes.byref(dst_layout),
                            len(shape), _shape(shape), datatype, _stream(stream), cta_cap)


def tcclReshardInspect(src_layout, dst_layout, shape, datatype, srcbufs, dstbufs, sm_count=152,
                       cta_cap=0, max_transfers=4096):
    """Host-only plan view: (result, transfers, bytes_read, bytes_written, windows) with
    transfers a list of dicts (src, dst_mask, lo, hi)."""
    sp, _k1 = _ptr_array(srcbufs)
    dp, _k2 = _ptr_array(dstbufs)
    buf = (ctypes.c_int64 * (10 * max_transfers))()
    nt, nw = ctypes.c_int(), ctypes.c_int()
    br, bw = ctypes.c_int64(), ctypes.c_int64()
    r = _lib.tcclReshardInspect(ctypes.byref(src_layout), ctypes.byref(dst_layout), len(shape),
                                _shape(shape), datatype, sp, dp, sm_count, cta_cap, buf,
                                max_transfers, ctypes.byref(nt), ctypes.byref(br),
                                ctypes.byref(bw), ctypes.byref(nw))
    nd = len(shape)
    tr = [dict(src=buf[10 * i], dst_mask=buf[10 * i + 1] & ((1 << 64) - 1),
               lo=list(buf[10 * i + 2:10 * i + 2 + nd]), hi=list(buf[10 * i + 6:10 * i + 6 + nd]))
          for i in range(min(nt.value, max_transfers))]
    return r, tr, br.value, bw.value, nw.value


def tcclGroupRecordSms(group, enable: bool) -> int:
    return _lib.tcclGroupRecordSms(group, int(bool(enable)))


def tcclGroupReadSmRecord(group):
    n = ctypes.c_int()
    r = _lib.tcclGroupReadSmRecord(group, ctypes.byref(n))
    return r, n.value


def tcclGroupReadSmRecordLaunches(group, max_launches: int = 64):
    """(result, distinct SMs per recorded launch, distinct SMs of all of them)."""
    buf = (ctypes.c_int * max(1, max_launches))()
    n, total = ctypes.c_int(), ctypes.c_int()
    r = _lib.tcclGroupReadSmRecordLaunches(group, buf, max_launches, ctypes.byref(n),
                                           ctypes.byref(total))
    return r, list(buf[:min(n.value, max_launches)]), total.value


def tcclGroupInjectWaitTimeout(group, enable: bool, timeout_ms: float = 0.0) -> int:
    return _lib.tcclGroupInjectWaitTimeout(group, int(bool(enable)), float(timeout_ms))


def tcclPlanInspect(coll, nranks, sendbufs, recvbufs, count, datatype, cta_cap=0,
                    sm_count=152, smem_per_block=232448, cfg=None, max_windows=4096):
    """Plans and lowers on the host only. Returns (result, windows, ntasks, info)
    with windows a list of dicts (cta, src_sel, src_off, dst_sel, dst_off,
    bytes, scalar, task)."""
    sp, _k1 = _ptr_array(sendbufs)
    rp, _k2 = _ptr_array(recvbufs)
    buf = (ctypes.c_int64 * (8 * max_windows))()
    nw, nt = ctypes.c_int(), ctypes.c_int()
    info = tcclLaunchInfo_t()
    r = _lib.tcclPlanInspect(coll, nranks, sp, rp, count, datatype, cta_cap, sm_count,
                             smem_per_block, ctypes.byref(cfg) if cfg is not None else None,
                             buf, max_windows, ctypes.byref(nw), ctypes.byref(nt),
                             ctypes.byref(info))
    keys = ("cta", "src_sel", "src_off", "dst_sel", "dst_off", "bytes", "scalar", "task")
    wins = [dict(zip(keys, buf[8 * i:8 * i + 8])) for i in range(min(nw.value, max_windows))]
    return r, wins, nt.value, info


def tcclCopyOutInspect(coll, nranks, sendbufs, recvbufs, count, datatype, cta_cap=0,
                       sm_count=152, cfg=None):
    """The copy-out engine's decisions on the host only. Returns (result,
    copy_out, register_fold, segments, segment_elems, wide_folds)."""
    sp, _k1 = _ptr_array(sendbufs)
    rp, _k2 = _ptr_array(recvbufs)
    co, rf, ns, wf = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    se = ctypes.c_size_t()
    r = _lib.tcclCopyOutInspect(coll, nranks, sp, rp, count, datatype, cta_cap, sm_count,
                                ctypes.byref(cfg) if cfg is not None else None, ctypes.byref(co),
                                ctypes.byref(rf), ctypes.byref(ns), ctypes.byref(se),
                                ctypes.byref(wf))
    return r, co.value, rf.value, ns.value, se.value, wf.value


# ---------------------------------------------------------------- torch-facing wrapper
class TcclError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        super().__init__(f"{what}: {tcclGetErrorString(code)} ({code})" if what else
                         f"{tcclGetErrorString(code)} ({code})")
        self.code = code


def _check(r: int, what: str = "") -> None:
    if r != tcclSuccess:
        raise TcclError(r, what)


_TORCH_DTYPE = None


def _dtype_code(t) -> int:
    global _TORCH_DTYPE
    if _TORCH_DTYPE is None:
        import torch
        _TORCH_DTYPE = {torch.float32: tcclFloat32, torch.bfloat16: tcclBfloat16,
                        torch.int32: tcclInt32}
    try:
        return _TORCH_DTYPE[t.dtype]
    except KeyError:
        raise TcclError(tcclInvalidArgument, f"unsupported dtype {t.dtype}") from None


def _current_stream():
    import torch
    return torch.cuda.current_stream().cuda_stream


class Group:
    """P logical ranks on the current CUDA device (``tcl::Group::create`` in
    single-process mode). Tensors are passed as lists, one per rank."""

    def __init__(self, nranks: int):
        r, h = tcclGroupCreate(nranks)
        _check(r, "tcclGroupCreate")
        self.handle = h
        self.nranks = nranks

    def close(self):
        if self.handle:
            _check(tcclGroupDestroy(self.handle), "tcclGroupDestroy")
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def config(self) -> tcclConfig_t:
        r, c = tcclGroupGetConfig(self.handle)
        _check(r, "tcclGroupGetConfig")
        return c

    def set_config(self, **kw) -> None:
        c = self.config
        for k, v in kw.items():
            setattr(c, k, v)
        _check(tcclGroupSetConfig(self.handle, c), "tcclGroupSetConfig")

    @staticmethod
    def _prepared(fn, args, name, keep):
        """A callable that makes the C call `fn(*args)` each time, with the
        arguments already marshalled; `keep` holds what they point into."""
        def call():
            r = fn(*args)
            if r != tcclSuccess:
                raise TcclError(r, name)

        call.keep = keep
        return call

    def prepare_all_reduce(self, sends, recvs=None, op="sum", cta_cap=0, stream=None):
        """A callable that issues this allreduce each time it is called, with
        its arguments marshalled once (pointer arrays, datatype, stream). For
        small messages the per-call marshalling is most of the host time. The
        tensors must stay alive, at the same addresses, while it is in use."""
        recvs = sends if recvs is None else recvs
        sp, keep_s = _ptr_array(sends)
        rp, keep_r = _ptr_array(recvs)
        args = (self.handle, sp, rp, sends[0].numel(), _dtype_code(sends[0]), OPS[op],
                _stream(stream) if stream is not None else _current_stream(), cta_cap)
        return self._prepared(_lib.tcclAllReduce, args, "tcclAllReduce", (keep_s, keep_r, sends, recvs))

    def prepare_reduce_scatter(self, sends, recvs, op="sum", cta_cap=0, stream=None):
        """prepare_all_reduce for reduce_scatter."""
        sp, keep_s = _ptr_array(sends)
        rp, keep_r = _ptr_array(recvs)
        args = (self.handle, sp, rp, recvs[0].numel(), _dtype_code(sends[0]), OPS[op],
                _stream(stream) if stream is not None else _current_stream(), cta_cap)
        return self._prepared(_lib.tcclReduceScatter, args, "tcclReduceScatter",
                              (keep_s, keep_r, sends, recvs))

    def prepare_all_gather(self, sends, recvs, cta_cap=0, stream=None):
        """prepare_all_reduce for all_gather."""
        sp, keep_s = _ptr_array(sends)
        rp, keep_r = _ptr_array(recvs)
        args = (self.handle, sp, rp, sends[0].numel(), _dtype_code(sends[0]),
                _stream(stream) if stream is not None else _current_stream(), cta_cap)
        return self._prepared(_lib.tcclAllGather, args, "tcclAllGather", (keep_s, keep_r, sends, recvs))

    def prepare_all_reduce_rmsnorm(self, sends, recvs, gamma, eps=1e-6, cta_cap=0, stream=None):
        """prepare_all_reduce for all_reduce_rmsnorm."""
        rows, hidden = sends[0].shape
        sp, keep_s = _ptr_array(sends)
        rp, keep_r = _ptr_array(recvs)
        args = (self.handle, sp, rp, rows, hidden, _ptr(gamma), eps, _dtype_code(sends[0]),
                _stream(stream) if stream is not None else _current_stream(), cta_cap)
        return self._prepared(_lib.tcclAllReduceRMSNorm, args, "tcclAllReduceRMSNorm",
                              (keep_s, keep_r, sends, recvs, gamma))

    def all_reduce(self, sends, recvs=None, op="sum", cta_cap=0, stream=None):
        """recvs[r] = fold over ranks of sends (ascending rank order). With
        recvs=None the reduction is in place."""
        recvs = sends if recvs is None else recvs
        dt = _dtype_code(sends[0])
        _check(tcclAllReduce(self.handle, sends, recvs, sends[0].numel(), dt, OPS[op],
                             stream if stream is not None else _current_stream(), cta_cap),
               "tcclAllReduce")
        return recvs

    def reduce_scatter(self, sends, recvs, op="sum", cta_cap=0, stream=None):
        dt = _dtype_code(sends[0])
        _check(tcclReduceScatter(self.handle, sends, recvs, recvs[0].numel(), dt, OPS[op],
                                 stream if stream is not None else _current_stream(), cta_cap),
               "tcclReduceScatter")
        return recvs

    def all_gather(self, sends, recvs, cta_cap=0, stream=None):
        dt = _dtype_code(sends[0])
        _check(tcclAllGather(self.handle, sends, recvs, sends[0].numel(), dt,
                             stream if stream is not None else _current_stream(), cta_cap),
               "tcclAllGather")
        return recvs

    def all_reduce_rmsnorm(self, sends, recvs, gamma, eps=1e-6, cta_cap=0, stream=None):
        """recvs[r][t, :] = RMSNorm(sum over ranks of sends[.][t, :]) * gamma, with
        every tensor [rows, hidden] (see tcclAllReduceRMSNorm)."""
        rows, hidden = sends[0].shape
        dt = _dtype_code(sends[0])
        _check(tcclAllReduceRMSNorm(self.handle, sends, recvs, rows, hidden, gamma, eps, dt,
                                    stream if stream is not None else _current_stream(), cta_cap),
               "tcclAllReduceRMSNorm")
        return recvs

    def reshard(self, srcs, src_layout, dsts, dst_layout, shape, cta_cap=0, stream=None):
        """Every destination rank gets its block of the tensor (see tcclReshard)."""
        dt = _dtype_code(srcs[0])
        _check(tcclReshard(self.handle, srcs, src_layout, dsts, dst_layout, list(shape), dt,
                           stream if stream is not None else _current_stream(), cta_cap),
               "tcclReshard")
        return dsts

    def query_error(self) -> int:
        r, s = tcclGroupQueryError(self.handle)
        _check(r, "tcclGroupQueryError")
        return s

    def last_launch(self) -> dict:
        r, info = tcclGetLastLaunchInfo(self.handle)
        _check(r, "tcclGetLastLaunchInfo")
        return info.as_dict()

    def record_sms(self, enable: bool = True) -> None:
        _check(tcclGroupRecordSms(self.handle, enable), "tcclGroupRecordSms")

    def read_sm_record(self) -> int:
        r, n = tcclGroupReadSmRecord(self.handle)
        _check(r, "tcclGroupReadSmRecord")
        return n

    def read_sm_record_launches(self):
        """(distinct SMs of each recorded launch, distinct SMs of all of them)."""
        r, per, total = tcclGroupReadSmRecordLaunches(self.handle)
        _check(r, "tcclGroupReadSmRecordLaunches")
        return per, total
