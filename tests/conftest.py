import os
import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parent.parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


import json

import pytest


@pytest.fixture(scope="session")
def parity_record():
    """Per-workload parity counts gathered by the GPU parity tests.  When the environment variable
    EAGLE_PARITY_RECORD names a file, the counts are written there as JSON at the end of the
    session (merged with what the file already holds), so a run leaves a record of how many
    requests and decisions were compared and how many fell inside each exemption window."""
    rec = {}
    yield rec
    path = os.environ.get("EAGLE_PARITY_RECORD")
    if path and rec:
        old = {}
        if os.path.exists(path):
            try:
                with open(path) as f:
                    old = json.load(f)
            except (OSError, ValueError):
                old = {}
        old.update(rec)
        with open(path, "w") as f:
            json.dump(old, f, indent=1, sort_keys=True)
