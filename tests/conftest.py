import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size parity case")


@pytest.fixture(scope="session")
def golden_dir():
    return ROOT / "tests" / "golden"


def _build_everything():
    import __graft_entry__

    __graft_entry__.build()


_build_everything()
