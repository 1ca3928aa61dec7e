import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# per-test limit when pytest-timeout is installed and no --timeout is given: device-side waits
# are bounded in the kernels, this bounds the host side (a deadlock would otherwise hang the run)
DEFAULT_TEST_TIMEOUT_S = 900


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    if not config.pluginmanager.hasplugin("timeout") or config.getoption("timeout", None):
        return
    for item in items:
        if item.get_closest_marker("timeout") is None:
            item.add_marker(pytest.mark.timeout(DEFAULT_TEST_TIMEOUT_S))
