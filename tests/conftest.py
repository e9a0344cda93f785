import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running case")


def pytest_sessionfinish(session, exitstatus):
    """Write the parity margins the GPU tests recorded (largest error per named
    workload and output, beside its tolerance) when ORTHROS_PARITY_JSON names a file."""
    path = os.environ.get("ORTHROS_PARITY_JSON")
    if not path:
        return
    from tests.parity_util import MARGINS

    if MARGINS:
        import json

        merged = {}
        if os.path.exists(path):  # entries of earlier sessions stay unless measured again
            with open(path) as f:
                merged = json.load(f)
        merged.update(MARGINS)
        with open(path, "w") as f:
            json.dump(merged, f, indent=1, sort_keys=True)
            f.write("\n")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle

    oracle.build()
    return oracle
