import json
import math
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def load_golden(name):
    """Load a fixture; the strings "-inf"/"inf" become floats."""
    def fix(x):
        if isinstance(x, list):
            return [fix(v) for v in x]
        if isinstance(x, str) and x in ("-inf", "inf"):
            return float(x)
        return x
    with open(os.path.join(GOLDEN, name)) as f:
        raw = json.load(f)
    return {k: fix(v) for k, v in raw.items()}


@pytest.fixture(scope="session")
def golden():
    return load_golden


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped, not failed, when no GPU is visible and they were
    # not explicitly selected with -m gpu.
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device visible")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)
