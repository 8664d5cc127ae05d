import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")


def pytest_collection_modifyitems(config, items):
    import torch
    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture
def set_option():
    """Set library options (moe_set_option) for one test; their old values come back afterwards."""
    import moe_expert_layer_routing_gb300 as mb
    saved = {}

    def _set(name, value):
        if name not in saved:
            saved[name] = mb.get_option(name)
        mb.set_option(name, value)

    yield _set
    for name, value in saved.items():
        mb.set_option(name, value)
