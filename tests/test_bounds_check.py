"""The bounds-checked build of the library (-DKDA_BOUNDS_CHECK): every plain
global load and store of the kernels checks its index against the extent of
the buffer it addresses and records a violation instead of making the access.

The self-test tells the two builds apart, and the parity tests of the main
paths then run again on the checked build in a child pytest
(KDA_TEST_CHECKED=1, see conftest.py).  There every device-error read also
fails if a kernel recorded an out-of-buffer index, so a pass shows that no
kernel indexed outside its buffers on those inputs: prefill (uniform, packed
varlen with empty sequences, split, d = 64 and 128, checkpoints, fused
preparation, the intermediate dump, the no-allocation entry point) and decode
(one token and several, with commits)."""
import os
import subprocess
import sys

import pytest

from gated_delta_rule_48_gb300 import binding as kb

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _device_error_message():
    st = kb.kda_get_device_error()
    return st, kb.load().kda_last_error_message().decode(errors="replace") if st else ""


def test_selftest_tells_the_builds_apart():
    if os.environ.get("KDA_TEST_CHECKED") == "1":
        pytest.skip("the child run tests only the checked build")
    kb.build(checked=True)
    try:
        kb.use_checked(True)
        assert kb.kda_bounds_checked()
        assert kb.kda_get_device_error() == 0
        kb.kda_selftest_bounds_check()
        st, msg = _device_error_message()
        assert st == 5 and "outside its buffer" in msg
        assert kb.kda_get_device_error() == 0  # read once, cleared
    finally:
        kb.use_checked(False)
    assert not kb.kda_bounds_checked()
    kb.kda_selftest_bounds_check()
    assert kb.kda_get_device_error() == 0  # compiled out: nothing recorded


CHILD_TESTS = [
    "tests/test_parity.py::test_workload0_tiny",
    "tests/test_parity.py::test_lengths_and_head_sizes",
    "tests/test_parity.py::test_varlen_short_and_long_with_empty",
    "tests/test_parity.py::test_segment_split_matches_oracle",
    "tests/test_parity.py::test_uniform_split_matches_oracle",
    "tests/test_parity.py::test_segment_split_d64_and_no_split_agree",
    "tests/test_parity.py::test_automatic_split_is_the_documented_length",
    "tests/test_parity.py::test_automatic_uniform_split_is_the_documented_length",
    "tests/test_parity.py::test_thousands_of_sequences",
    "tests/test_parity.py::test_state_aliasing_continuation",
    "tests/test_parity.py::test_decode_steps_equal_prefill_of_same_tokens",
    "tests/test_parity.py::test_empty_sequences_hand_state_through",
    "tests/test_parity.py::test_malformed_cu_seqlens_sets_device_error",
    "tests/test_fused.py",
    "tests/test_checkpoints.py",
    "tests/test_decode_tokens.py",
    "tests/test_intermediates.py",
    "tests/test_zz_no_alloc.py",
]


def test_main_paths_on_the_checked_build():
    if os.environ.get("KDA_TEST_CHECKED") == "1":
        pytest.skip("already the checked run")
    kb.build(checked=True)
    env = dict(os.environ, KDA_TEST_CHECKED="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "-m", "gpu", *CHILD_TESTS], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
