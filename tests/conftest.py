import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running check")


def pytest_collection_modifyitems(config, items):
    # GPU tests skip (rather than fail) only when no CUDA device is present at all;
    # with a device present, a missing or unloadable library is an error.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(scope="session")
def paper_facts():
    with open(os.path.join(ROOT, "tests", "golden", "paper_facts.json")) as f:
        return {k: v["value"] for k, v in json.load(f).items() if not k.startswith("_")}
