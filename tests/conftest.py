"""Shared pytest setup: repo root on sys.path, the `gpu` marker, golden-fixture loading."""

import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def load_golden(name):
    """Golden fixtures are '#'-comment headers (the citation) followed by one JSON document."""
    with open(os.path.join(GOLDEN, name)) as f:
        body = "".join(line for line in f if not line.lstrip().startswith("#"))
    return json.loads(body)


@pytest.fixture(scope="session")
def orc():
    import oracle

    oracle.build()
    return oracle
