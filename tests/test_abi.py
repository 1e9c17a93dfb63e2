"""The C-ABI library loads and exports every entry point include/tccl.h declares.
No compute calls: these run without a GPU."""
import ctypes
import re
from pathlib import Path

import pytest

import collective_communication_planner_gb300 as tccl

HEADER = Path(__file__).resolve().parents[1] / "include" / "tccl.h"


def declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tccl[A-Z]\w*)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("tcclGroupCreate", "tcclGroupDestroy", "tcclAllReduce", "tcclReduceScatter",
              "tcclAllGather", "tcclGroupQueryError", "tcclGetErrorString",
              "tcclGetLastLaunchInfo"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(str(tccl.LIB_PATH))
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(tccl.EXPORTED)


def test_version_and_error_strings():
    assert tccl.tcclGetVersion() == 1000
    for code in range(6):
        s = tccl.tcclGetErrorString(code)
        assert s and "unknown" not in s
    assert "unknown" in tccl.tcclGetErrorString(99)


def test_group_calls_reject_null_group():
    null = ctypes.c_void_p()
    assert tccl.tcclGroupDestroy(null) == tccl.tcclInvalidArgument
    assert tccl.tcclAllReduce(null, [1], [2], 4, 0, 0) == tccl.tcclInvalidArgument
    assert tccl.tcclReduceScatter(null, [1], [2], 4, 0, 0) == tccl.tcclInvalidArgument
    assert tccl.tcclAllGather(null, [1], [2], 4, 0) == tccl.tcclInvalidArgument
    r, _ = tccl.tcclGroupQueryError(null)
    assert r == tccl.tcclInvalidArgument
    r, _ = tccl.tcclGetLastLaunchInfo(null)
    assert r == tccl.tcclInvalidArgument


def test_group_create_argument_checks():
    r, _ = tccl.tcclGroupCreate(0)
    assert r == tccl.tcclInvalidArgument
    r, _ = tccl.tcclGroupCreate(65)
    assert r == tccl.tcclInvalidArgument


def test_group_create_without_device_reports_cuda_error():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    r, h = tccl.tcclGroupCreate(4)
    assert r == tccl.tcclCudaError and not h.value


def test_library_does_not_load_the_oracle():
    # the product library links no oracle code
    lib_bytes = Path(tccl.LIB_PATH).read_bytes()
    assert b"oracle_allreduce" not in lib_bytes
