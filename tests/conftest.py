import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running case")


@pytest.fixture(scope="session")
def golden():
    import json
    with open(os.path.join(ROOT, "tests", "golden", "worked_examples.json")) as f:
        return json.load(f)


@pytest.fixture(scope="session", autouse=True)
def _library_variant():
    """With ATTN_LIBRARY=checked every test runs on the checked debug build: make sure
    that is the library that loaded."""
    if os.environ.get("ATTN_LIBRARY") == "checked":
        import ring_attention_online_gb300 as ra
        assert ra.attn_build_checked(), "ATTN_LIBRARY=checked loaded a library without checks"
    yield
