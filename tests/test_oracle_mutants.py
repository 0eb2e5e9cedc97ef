"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in a copy of the C oracle (a changed line of
kda_oracle.c), builds it into a temporary library, points the oracle binding
at it, and runs the pins of test_oracle.py: at least one pin must fail.  This
is evidence that the pins constrain the oracle, not just re-run it.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

MUTANTS = {
    "delta write subtracted": ("S[c * dv + j] += w->k[c] * w->u[j];",
                               "S[c * dv + j] -= w->k[c] * w->u[j];"),
    "error term sign flipped": ("w->u[j] = b * (w->v[j] - acc);",
                                "w->u[j] = b * (w->v[j] + acc);"),
    "beta ignored": ("w->u[j] = b * (w->v[j] - acc);",
                     "w->u[j] = 1.0 * (w->v[j] - acc);"),
    "clamp at -5 dropped": ("if (la < -5.0) la = -5.0;", ""),
    "decay exponent halved": ("w->alpha[c] = exp(la);", "w->alpha[c] = exp(0.5 * la);"),
    "decay on the wrong channel": ("S[c * dv + j] *= w->alpha[c];",
                                   "S[c * dv + j] *= w->alpha[(c + 1) % dk];"),
    "read out with k instead of q": ("acc += S[c * dv + j] * w->q[c];",
                                     "acc += S[c * dv + j] * w->k[c];"),
    "read out before the write": ("        /* S = S' + k u^T */",
                                  "        for (int64_t j = 0; j < dv; ++j) { double acc = 0.0;"
                                  " for (int64_t c = 0; c < dk; ++c) acc += S[c * dv + j] * w->q[c];"
                                  " job->out[(t * nh + hs) * dv + j] = acc; }\n        continue;"),
}

PINS = [
    lambda: pins.test_unit_key_beta_one_writes_value(8, 5),
    lambda: pins.test_beta_zero_from_zero_state_is_zero(),
    lambda: pins.test_single_token_closed_form(6, 4),
    lambda: pins.test_clamped_floor_decay(-7.5),
    lambda: pins.test_per_channel_decay_axis_and_time_index(),
    lambda: pins.test_orthonormal_keys_reduce_to_linear_attention(16, 8, 16),
    lambda: pins.test_chunked_ut_form_matches_recurrence(16, 70),
    lambda: pins.test_scalar_decay_is_rescaled_ungated_delta_rule(),
    lambda: pins.test_state_norm_never_grows_without_writes(),
]


def _build(tmp_path, src_text, name):
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(src_text)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", str(c),
                           "-o", str(so), "-lm"])
    lib = ctypes.CDLL(str(so))
    ref = oracle._load()
    lib.kda_oracle_forward.restype = ref.kda_oracle_forward.restype
    lib.kda_oracle_forward.argtypes = ref.kda_oracle_forward.argtypes
    return lib


def _failing_pins(lib):
    saved = oracle._lib
    oracle._lib = lib
    failed = 0
    try:
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                failed += 1
    finally:
        oracle._lib = saved
    return failed


def test_unmutated_copy_passes_every_pin(tmp_path):
    lib = _build(tmp_path, open(SRC).read(), "same")
    assert _failing_pins(lib) == 0


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_each_planted_mistake_fails_a_pin(tmp_path, name):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor for '{name}' not found once"
    lib = _build(tmp_path, text.replace(old, new), "mutant")
    assert _failing_pins(lib) >= 1, f"no pin caught: {name}"
