"""Seeded synthetic rank buffers (SplitMix64 streams), shared by both sides.

The recipe is stated in ``gen.c``. This module draws numbers only: it holds
none of the collective's arithmetic, so the oracle and the CUDA path can both
take its arrays as inputs without sharing any code of the method.

Workload shapes (rank count, element count, value law, seed) come from the
T-CCL description of NCCL-semantics collectives over P equal-length rank
buffers ("NCCL M2N vs T-CCL" article, section 2.3 programming model).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_LIB_PATH = _HERE / "libtccl_datagen.so"
_lib = None

UNIFORM_F32, INT32, NORMAL_F32, NORMAL_BF16 = 0, 1, 2, 3


def build(force: bool = False) -> Path:
    """Compile gen.c into a shared library next to it (gcc, no fast-math)."""
    src = _HERE / "gen.c"
    if force or not _LIB_PATH.exists() or _LIB_PATH.stat().st_mtime < src.stat().st_mtime:
        tmp = _LIB_PATH.with_suffix(f".{os.getpid()}.tmp")
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
             "-ffp-contract=off", "-o", str(tmp), str(src), "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(str(_LIB_PATH))
        lib.gen_fill.restype = ctypes.c_int
        lib.gen_fill.argtypes = [ctypes.c_int, ctypes.c_uint64, ctypes.c_int, ctypes.c_uint64,
                                 ctypes.c_void_p, ctypes.c_double, ctypes.c_double,
                                 ctypes.c_int32, ctypes.c_int32, ctypes.c_int]
        lib.gen_stream_state.restype = ctypes.c_uint64
        lib.gen_stream_state.argtypes = [ctypes.c_uint64, ctypes.c_int]
        lib.gen_raw.restype = None
        lib.gen_raw.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                ctypes.c_void_p]
        _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def stream_state(seed: int, rank: int) -> int:
    return int(_load().gen_stream_state(seed, rank))


def raw(state0: int, first: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().gen_raw(state0, first, n, out.ctypes.data)
    return out


def _fill(kind, seed, rank, n, dtype, mu=0.0, sigma=1.0, lo=0, hi=0, out=None, nthreads=0):
    if out is None:
        out = np.empty(n, dtype=dtype)
    assert out.dtype == dtype and out.size == n and out.flags.c_contiguous
    rc = _load().gen_fill(kind, seed, rank, n, out.ctypes.data, mu, sigma, lo, hi,
                            nthreads or _threads())
    if rc != 0:
        raise ValueError("gen_fill rejected its arguments")
    return out


def uniform_f32(seed: int, rank: int, n: int, out=None, nthreads: int = 0) -> np.ndarray:
    """Uniform values in [-1, 1), multiples of 2^-23."""
    return _fill(UNIFORM_F32, seed, rank, n, np.float32, out=out, nthreads=nthreads)


def int32(seed: int, rank: int, n: int, lo: int = -1000, hi: int = 1000, out=None,
          nthreads: int = 0) -> np.ndarray:
    """Integers uniform in [lo, hi]."""
    return _fill(INT32, seed, rank, n, np.int32, lo=lo, hi=hi, out=out, nthreads=nthreads)


def normal_f32(seed: int, rank: int, n: int, mu: float = 0.0, sigma: float = 1.0,
               out=None, nthreads: int = 0) -> np.ndarray:
    return _fill(NORMAL_F32, seed, rank, n, np.float32, mu=mu, sigma=sigma, out=out,
                 nthreads=nthreads)


def normal_bf16(seed: int, rank: int, n: int, mu: float = 0.0, sigma: float = 1.0,
                out=None, nthreads: int = 0) -> np.ndarray:
    """N(mu, sigma) rounded to bf16; returned as the uint16 bit patterns."""
    return _fill(NORMAL_BF16, seed, rank, n, np.uint16, mu=mu, sigma=sigma, out=out,
                 nthreads=nthreads)


def rank_buffers(kind: str, seed: int, nranks: int, n: int, **kw) -> list[np.ndarray]:
    """One array per logical rank, stream (seed, rank) each."""
    fn = {"uniform_f32": uniform_f32, "int32": int32, "normal_f32": normal_f32,
          "normal_bf16": normal_bf16}[kind]
    return [fn(seed, r, n, **kw) for r in range(nranks)]
