import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libhc")
    config.addinivalue_line("markers", "slow: CPU test that takes more than a few seconds")


@pytest.fixture(scope="session")
def golden_constants():
    import json
    with open(os.path.join(ROOT, "tests", "golden", "v41_hc_constants.json")) as fh:
        return {k: v["value"] for k, v in json.load(fh).items() if not k.startswith("_")}
