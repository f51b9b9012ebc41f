"""Test configuration: the `gpu` marker and shared fixtures.

Tests marked `gpu` need a GB300 (sm_103) and the in-tree CUDA library; every
other test runs on a machine without a GPU.
"""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 GPU and the CUDA library")
    # build the CUDA library and the oracle in-tree if missing or stale (no-op otherwise)
    import __graft_entry__
    __graft_entry__.build()


@pytest.fixture(scope="session")
def golden():
    with open(os.path.join(ROOT, "tests", "golden", "page_constants.json")) as f:
        return json.load(f)
