"""CPU oracle for allreduce / reduce-scatter / all-gather over P rank buffers.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline (and ``--impl reference``) leg may import this
package. The library under ``collective_communication_planner_gb300`` never
does, and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, built with gcc, no fast-math,
no FMA contraction); this module only marshals numpy arrays. What each call
computes, and which passage of the T-CCL description ("NCCL M2N vs T-CCL"
article, sections 2.1-2.4) it follows, is stated in ``oracle.c``'s header.

bf16 arrays are carried as ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_LIB_PATH = _HERE / "liboracle.so"
_lib = None

F32, BF16, I32 = 0, 1, 2
SUM, MIN, MAX = 0, 1, 2

DTYPES = {"f32": F32, "bf16": BF16, "i32": I32}
OPS = {"sum": SUM, "min": MIN, "max": MAX}
NP_DTYPE = {F32: np.float32, BF16: np.uint16, I32: np.int32}


def build(force: bool = False) -> Path:
    """Compile oracle.c into liboracle.so beside it."""
    src = _HERE / "oracle.c"
    if force or not _LIB_PATH.exists() or _LIB_PATH.stat().st_mtime < src.stat().st_mtime:
        tmp = _LIB_PATH.with_suffix(f".{os.getpid()}.tmp")
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
             "-ffp-contract=off", "-o", str(tmp), str(src)])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        _lib = _open(build())
    return _lib


def use_library(path) -> None:
    """Point this module at another build of oracle.c (the pin tests use it to
    show that deliberately broken copies fail them); ``None`` restores it."""
    global _lib
    _lib = None if path is None else _open(Path(path))


def _open(path: Path):
    lib = ctypes.CDLL(str(path))
    pp = ctypes.POINTER(ctypes.c_void_p)
    for name in ("oracle_allreduce", "oracle_reduce_scatter"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_uint64, pp, pp]
        f = getattr(lib, name + "_mt")
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_uint64, pp, pp,
                      ctypes.c_int]
    lib.oracle_allgather.restype = ctypes.c_int
    lib.oracle_allgather.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_uint64, pp, pp]
    lib.oracle_allgather_mt.restype = ctypes.c_int
    lib.oracle_allgather_mt.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_uint64, pp, pp,
                                        ctypes.c_int]
    return lib


def _ptrs(arrays):
    arr = (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), arr


def _code(v, table):
    return table[v] if isinstance(v, str) else int(v)


def _threads(nthreads):
    return nthreads if nthreads else max(1, os.cpu_count() or 1)


def allreduce(sends, dtype="f32", op="sum", recvs=None, nthreads: int = 1):
    """recv[r][i] = fold over ranks of send[.][i], for every rank r.

    ``nthreads`` > 1 (or 0 = all cores) runs the threaded variant, whose
    bits equal the single-threaded one. Returns the list of recv arrays.
    """
    dt, o = _code(dtype, DTYPES), _code(op, OPS)
    p = len(sends)
    count = sends[0].size
    for s in sends:
        assert s.dtype == NP_DTYPE[dt] and s.size == count and s.flags.c_contiguous
    if recvs is None:
        recvs = [np.empty(count, dtype=NP_DTYPE[dt]) for _ in range(p)]
    sp, _k1 = _ptrs(sends)
    rp, _k2 = _ptrs(recvs)
    lib = _load()
    rc = (lib.oracle_allreduce(dt, o, p, count, sp, rp) if nthreads == 1 else
          lib.oracle_allreduce_mt(dt, o, p, count, sp, rp, _threads(nthreads)))
    if rc < 0:
        raise ValueError("oracle_allreduce rejected its arguments")
    return recvs


def reduce_scatter(sends, dtype="f32", op="sum", recvs=None, nthreads: int = 1):
    """recv[r][j] = fold over ranks of send[.][r*rc + j]; rc = count / P."""
    dt, o = _code(dtype, DTYPES), _code(op, OPS)
    p = len(sends)
    total = sends[0].size
    assert total % p == 0
    rc = total // p
    if recvs is None:
        recvs = [np.empty(rc, dtype=NP_DTYPE[dt]) for _ in range(p)]
    sp, _k1 = _ptrs(sends)
    rp, _k2 = _ptrs(recvs)
    lib = _load()
    r = (lib.oracle_reduce_scatter(dt, o, p, rc, sp, rp) if nthreads == 1 else
         lib.oracle_reduce_scatter_mt(dt, o, p, rc, sp, rp, _threads(nthreads)))
    if r < 0:
        raise ValueError("oracle_reduce_scatter rejected its arguments")
    return recvs


def allgather(sends, recvs=None, nthreads: int = 1):
    """recv[r][k*sc + j] = send[k][j] for every r; sc = per-rank send count."""
    p = len(sends)
    sc = sends[0].size
    es = sends[0].dtype.itemsize
    if recvs is None:
        recvs = [np.empty(p * sc, dtype=sends[0].dtype) for _ in range(p)]
    sp, _k1 = _ptrs(sends)
    rp, _k2 = _ptrs(recvs)
    lib = _load()
    r = (lib.oracle_allgather(es, p, sc, sp, rp) if nthreads == 1 else
         lib.oracle_allgather_mt(es, p, sc, sp, rp, _threads(nthreads)))
    if r < 0:
        raise ValueError("oracle_allgather rejected its arguments")
    return recvs


def allreduce_ptrs(dtype, op, nranks, count, send_ptrs, recv_ptrs, nthreads=1):
    """Pointer form (addresses of host arrays), for in-place aliasing tests."""
    lib = _load()
    sp, _k1 = _ptrs_raw(send_ptrs)
    rp, _k2 = _ptrs_raw(recv_ptrs)
    dt, o = _code(dtype, DTYPES), _code(op, OPS)
    r = (lib.oracle_allreduce(dt, o, nranks, count, sp, rp) if nthreads == 1 else
         lib.oracle_allreduce_mt(dt, o, nranks, count, sp, rp, _threads(nthreads)))
    if r < 0:
        raise ValueError("oracle_allreduce rejected its arguments")


def reduce_scatter_ptrs(dtype, op, nranks, recvcount, send_ptrs, recv_ptrs, nthreads=1):
    lib = _load()
    sp, _k1 = _ptrs_raw(send_ptrs)
    rp, _k2 = _ptrs_raw(recv_ptrs)
    dt, o = _code(dtype, DTYPES), _code(op, OPS)
    r = (lib.oracle_reduce_scatter(dt, o, nranks, recvcount, sp, rp) if nthreads == 1 else
         lib.oracle_reduce_scatter_mt(dt, o, nranks, recvcount, sp, rp, _threads(nthreads)))
    if r < 0:
        raise ValueError("oracle_reduce_scatter rejected its arguments")


def allgather_ptrs(elem_size, nranks, sendcount, send_ptrs, recv_ptrs, nthreads=1):
    lib = _load()
    sp, _k1 = _ptrs_raw(send_ptrs)
    rp, _k2 = _ptrs_raw(recv_ptrs)
    r = (lib.oracle_allgather(elem_size, nranks, sendcount, sp, rp) if nthreads == 1 else
         lib.oracle_allgather_mt(elem_size, nranks, sendcount, sp, rp, _threads(nthreads)))
    if r < 0:
        raise ValueError("oracle_allgather rejected its arguments")


def _ptrs_raw(addrs):
    arr = (ctypes.c_void_p * len(addrs))(*addrs)
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), arr
