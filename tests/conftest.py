import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 GPU and the built CUDA library")


@pytest.fixture(scope="session")
def facts():
    with open(os.path.join(GOLDEN, "pages_facts.json")) as f:
        return json.load(f)


@pytest.fixture(scope="session")
def oracle():
    import oracle as o
    o.build()
    return o
