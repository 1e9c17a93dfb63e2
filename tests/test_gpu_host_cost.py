"""The C ABI driven from C++ (tests/host_cost.cu, no Python between the caller
and the library): decode-sized allreduces give exact results, and the host
side of a call stays within a few microseconds of an empty kernel launch."""
import json
import subprocess
import sys
from pathlib import Path

import pytest

pytestmark = pytest.mark.gpu
ROOT = Path(__file__).resolve().parents[1]


def test_cpp_caller_results_and_host_cost():
    sys.path.insert(0, str(ROOT))
    import bench

    exe = bench.build_host_cost()
    r = subprocess.run([str(exe), "10"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    rows = [json.loads(ln) for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(rows) == 5
    for row in rows:
        print(row)
        assert row["ok"], row
        # the library's own host work (validation, plan-cache lookup, launch
        # arguments) on top of the launch itself: a loose bound that catches a
        # regression such as a per-call allocation or synchronisation
        assert row["host_us"] < row["launch_early_us"] + 10.0, row
