import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


# KDA_TEST_CHECKED=1 runs the tests against the bounds-checked build of the
# library (tests/test_bounds_check.py starts such a run): every device-error
# read then also fails the test if a kernel recorded an out-of-buffer index,
# even where the test expects another device error.
CHECKED = os.environ.get("KDA_TEST_CHECKED") == "1"
BOUNDS_MESSAGE = "outside its buffer"


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    if CHECKED:
        from gated_delta_rule_48_gb300 import binding as kb
        kb.build(checked=True)
        kb.use_checked(True)
        plain = kb.kda_get_device_error

        def checked_device_error(stream=None):
            st = plain(stream)
            if st != 0:
                msg = kb.load().kda_last_error_message().decode(errors="replace")
                assert BOUNDS_MESSAGE not in msg, msg
            return st

        kb.kda_get_device_error = checked_device_error


@pytest.fixture(autouse=True)
def _no_bounds_violation_left():
    """In a checked run, a test that never reads the device error word still
    leaves nothing recorded."""
    yield
    if CHECKED:
        import torch
        if torch.cuda.is_available():
            from gated_delta_rule_48_gb300 import binding as kb
            kb.kda_get_device_error()


def pytest_collection_modifyitems(config, items):
    import torch
    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
