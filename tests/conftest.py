import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")


def read_golden(name):
    """Rows of a golden fixture: (left fields, right fields), comments stripped."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            left, right = line.split(":")
            rows.append((left.split(), right.split()))
    return rows


@pytest.fixture
def golden():
    return read_golden


@pytest.fixture(autouse=True)
def _tag_parity_records(request):
    """Label the parity records a test makes with the test's id (see tests/gpu_util.py)."""
    yield
    mod = sys.modules.get("tests.gpu_util")
    if mod is not None:
        for rec in mod.OBSERVED:
            rec.setdefault("test", request.node.nodeid)


def pytest_sessionfinish(session, exitstatus):
    """With LL_PARITY_LOG set, write every GPU parity comparison (test, check, errors) as JSON."""
    path = os.environ.get("LL_PARITY_LOG")
    mod = sys.modules.get("tests.gpu_util")
    if not path or mod is None:
        return
    import json

    with open(path, "w") as f:
        json.dump(mod.OBSERVED, f)
