"""Pins for the oracle's input preparation of the fused entry points (CPU only).

``oracle.prep`` forms log alpha = -5 sigmoid(gate), L2-normalises q and k per
(token, head) and rounds them to bfloat16.  Each pin checks it against
something other than itself: a library routine (scipy's logistic function,
torch's float32 -> bfloat16 conversion), closed values, the invariants of a
normalisation (unit norm, scale invariance, the axis it acts on), and the
floor of the norm.  A wrong sign in the gate, normalising over the wrong
axis, a dropped rounding or rounding the wrong way fails one of them.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import prep
from gated_delta_rule_48_gb300 import inputs as kin


def _bits(x):
    """bfloat16 bit patterns of float values that bfloat16 represents exactly."""
    t = torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.tensor(np.asarray(x, dtype=np.float32)))
    return kin.bf16_bits(t)


def test_round_bf16_matches_torch_on_float32_values():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32),
                        (rng.standard_normal(2000) * 1e-3).astype(np.float32),
                        (rng.standard_normal(2000) * 1e3).astype(np.float32)])
    ref = torch.tensor(x).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(prep.round_bf16(x.astype(np.float64)), ref)


def test_round_bf16_ties_go_to_even():
    # bf16 spacing just above 1 is 2^-7; halfway points round to the even mantissa
    assert prep.round_bf16(np.array(1.0 + 2.0 ** -8)) == 1.0
    assert prep.round_bf16(np.array(1.0 + 3 * 2.0 ** -8)) == 1.0 + 2.0 ** -6
    assert prep.round_bf16(np.array(-(1.0 + 2.0 ** -8))) == -1.0
    assert prep.round_bf16(np.array(1.0 + 2.0 ** -8 + 2.0 ** -30)) == 1.0 + 2.0 ** -7
    assert prep.round_bf16(np.array(0.0)) == 0.0


def test_gate_curve_is_minus_five_logistic():
    special = pytest.importorskip("scipy.special")
    x = np.linspace(-30.0, 30.0, 2001)
    np.testing.assert_allclose(prep.gate_log_alpha(x), -5.0 * special.expit(x), rtol=1e-14,
                               atol=1e-300)
    assert prep.gate_log_alpha(np.array(0.0)) == -2.5
    # bounded below at -5 (large logits forget the most), zero decay for very negative logits
    assert -5.0 <= prep.gate_log_alpha(np.array(40.0)) < -5.0 + 1e-15
    assert -1e-15 < prep.gate_log_alpha(np.array(-40.0)) <= 0.0
    assert np.all(np.diff(prep.gate_log_alpha(x)) < 0)


def test_normalise_unit_norm_per_token_head():
    rng = np.random.default_rng(1)
    # heads with very different scales: a wrong axis would mix them
    x = rng.standard_normal((7, 3, 64)) * np.array([1e-3, 1.0, 50.0])[None, :, None]
    y = prep.l2_normalise(x)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), 1.0, rtol=1e-14)
    # same direction as the input
    np.testing.assert_allclose(y * np.linalg.norm(x, axis=-1, keepdims=True), x, rtol=1e-13)


def test_prepare_scale_invariant_and_unit_vectors_unchanged():
    rng = np.random.default_rng(2)
    q = torch.from_numpy(rng.standard_normal((5, 2, 128)).astype(np.float32)).to(torch.bfloat16)
    qb, qb8 = kin.bf16_bits(q), kin.bf16_bits(q * 8)  # exact power-of-two scaling in bf16
    g = kin.bf16_bits(torch.zeros((5, 2, 128), dtype=torch.bfloat16))
    a, _, _ = prep.prepare(qb, qb, g)
    b, _, _ = prep.prepare(qb8, qb8, g)
    np.testing.assert_array_equal(a, b)
    # rounding after normalising: every component is a bfloat16 value, the norm is 1 to bf16 precision
    np.testing.assert_array_equal(prep.round_bf16(a), a)
    assert np.all(np.abs(np.linalg.norm(a, axis=-1) - 1.0) < 2.0 ** -7)
    # a unit vector that bfloat16 holds exactly comes back unchanged
    u = np.zeros((1, 1, 128))
    u[0, 0, [3, 17, 64, 127]] = [0.5, -0.5, 0.5, 0.5]
    pu, _, _ = prep.prepare(_bits(u), _bits(u), _bits(np.zeros_like(u)))
    np.testing.assert_array_equal(pu, u)


def test_normalise_floor_zero_and_tiny_vectors():
    z = np.zeros((1, 1, 8))
    np.testing.assert_array_equal(prep.l2_normalise(z), z)
    t = np.zeros((1, 1, 8))
    t[0, 0, 2] = 1e-15                   # norm below the 1e-12 floor: divided by the floor
    np.testing.assert_allclose(prep.l2_normalise(t)[0, 0, 2], 1e-3, rtol=1e-15)


def test_fused_forward_is_forward_of_prepared_inputs():
    p = kin.make_prefill_raw([40, 25], 2, 16, seed=7, s0_std=0.05)
    args = (kin.bf16_bits(p.q_raw), kin.bf16_bits(p.k_raw), kin.bf16_bits(p.v),
            kin.bf16_bits(p.gate), p.beta.numpy(), p.S0.numpy(), p.cu_seqlens)
    out, S = prep.forward_fused(*args)
    q, k, la = prep.prepare(args[0], args[1], args[3])
    out2, S2 = oracle.forward(q, k, prep.bf16_bits_to_f64(args[2]), la,
                              p.beta.numpy().astype(np.float64), p.S0.numpy().astype(np.float64),
                              p.cu_seqlens)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(S, S2)
    # the layer is blind to the scale of the raw q and k projections
    p8 = kin.make_prefill_raw([40, 25], 2, 16, seed=7, s0_std=0.05, q_scale=8.0)
    out8, S8 = prep.forward_fused(kin.bf16_bits(p8.q_raw), kin.bf16_bits(p8.k_raw), *args[2:])
    np.testing.assert_array_equal(out8, out)
    np.testing.assert_array_equal(S8, S)


def test_fused_decode_matches_fused_prefill():
    d = kin.make_decode_raw(3, 2, 16, steps=5, seed=9)
    bits = [kin.bf16_bits(t) for t in (d.q_raw, d.k_raw, d.v, d.gate)]
    out, S = prep.decode_steps_fused(*bits, d.beta.numpy(), d.S.numpy())
    steps, N = 5, 3

    def pack(a):
        return np.ascontiguousarray(np.swapaxes(a, 0, 1)).reshape((N * steps,) + a.shape[2:])

    cu = np.arange(N + 1) * steps
    out_p, S_p = prep.forward_fused(*[pack(b) for b in bits], pack(d.beta.numpy()), d.S.numpy(), cu)
    np.testing.assert_allclose(S, S_p, rtol=0, atol=0)
    np.testing.assert_allclose(np.swapaxes(out, 0, 1).reshape(out_p.shape), out_p, rtol=0, atol=0)


# ---------------------------------------------------------------- planted mistakes
# Each case replaces one step of oracle.prep with a plausible slip and runs the
# pins above against the modified module: at least one must fail.
import types


def _pins(mod):
    saved = {}
    failed = 0
    pins = [test_round_bf16_matches_torch_on_float32_values, test_round_bf16_ties_go_to_even,
            test_gate_curve_is_minus_five_logistic, test_normalise_unit_norm_per_token_head,
            test_prepare_scale_invariant_and_unit_vectors_unchanged,
            test_normalise_floor_zero_and_tiny_vectors]
    for name in ("round_bf16", "gate_log_alpha", "l2_normalise", "prepare"):
        saved[name] = getattr(prep, name)
        setattr(prep, name, getattr(mod, name))
    try:
        for pin in pins:
            try:
                pin()
            except (AssertionError, ValueError):
                failed += 1
    finally:
        for name, fn in saved.items():
            setattr(prep, name, fn)
    return failed


def _mutant(**overrides):
    mod = types.SimpleNamespace(round_bf16=prep.round_bf16, gate_log_alpha=prep.gate_log_alpha,
                                l2_normalise=prep.l2_normalise)
    for k, v in overrides.items():
        setattr(mod, k, v)

    def prepare(q_raw_bits, k_raw_bits, gate_bits):
        q = mod.round_bf16(mod.l2_normalise(prep.bf16_bits_to_f64(q_raw_bits)))
        k = mod.round_bf16(mod.l2_normalise(prep.bf16_bits_to_f64(k_raw_bits)))
        return q, k, mod.gate_log_alpha(prep.bf16_bits_to_f64(gate_bits))
    mod.prepare = prepare
    return mod


MUTANTS = {
    "gate sign flipped": dict(gate_log_alpha=lambda g: -5.0 / (1.0 + np.exp(np.asarray(g, float)))),
    "gate scale 4 instead of 5": dict(gate_log_alpha=lambda g: -4.0 / (1.0 + np.exp(-np.asarray(g, float)))),
    "normalised over heads": dict(l2_normalise=lambda x: np.asarray(x, float) / np.maximum(
        np.sqrt(np.sum(np.asarray(x, float) ** 2, axis=-2, keepdims=True)), 1e-12)),
    "no floor on the norm": dict(l2_normalise=lambda x: np.asarray(x, float) / np.sqrt(
        np.sum(np.asarray(x, float) ** 2, axis=-1, keepdims=True))),
    "rounded by truncation": dict(round_bf16=lambda x: np.ldexp(np.trunc(np.ldexp(
        np.frexp(np.asarray(x, float))[0], 8)), np.frexp(np.asarray(x, float))[1] - 8)),
    "no rounding": dict(round_bf16=lambda x: np.asarray(x, float)),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_each_planted_prep_mistake_fails_a_pin(name):
    with np.errstate(all="ignore"):
        assert _pins(_mutant(**MUTANTS[name])) >= 1, f"no pin caught: {name}"


def test_unmodified_prep_passes_every_pin():
    assert _pins(_mutant()) == 0
