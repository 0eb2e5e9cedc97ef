"""Pins for the fp64 oracle (CPU only).

Each test checks the oracle against something other than itself: a closed
form the mathematics fixes, a special case that reduces to a textbook
routine, an invariant of the recurrence, a second independently derived
algorithm (the chunked UT-transform form), or a numeric fact the pages print.
They are chosen so that a plausible slip -- wrong sign in (I - beta k k^T),
decay applied after the write, readout before the update, decay on the wrong
axis or at the wrong time index, a dropped clamp, a transposed state --
fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import naive_chunked
from gated_delta_rule_48_gb300 import inputs as kin

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, T, H, dk, dv, *, la_lo=-5.0, la_hi=0.0, beta=None, unit_k=True,
          unit_q=False, s0=0.5, n_seqs=1):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    if unit_q:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    la = rng.uniform(la_lo, la_hi, size=(T, H, dk))
    b = rng.uniform(0.0, 1.0, size=(T, H)) if beta is None else np.full((T, H), float(beta))
    S0 = None if s0 is None else s0 * rng.standard_normal((n_seqs, H, dk, dv))
    return q, k, v, la, b, S0


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("dk,dv", [(8, 5), (16, 16)])
def test_unit_key_beta_one_writes_value(dk, dv):
    """beta = 1 and |k| = 1: (I - k k^T) annihilates k, so S_t^T k_t = v_t
    whatever alpha and the previous state are.  Reading with q = k gives v."""
    rng = np.random.default_rng(1)
    q, k, v, la, b, S0 = _rand(rng, 40, 2, dk, dv, la_lo=-9.0, la_hi=1.0, beta=1.0, s0=1.0)
    out, _ = oracle.forward(k.copy(), k, v, la, b, S0)
    np.testing.assert_allclose(out, v, rtol=0, atol=1e-12)


def test_beta_zero_from_zero_state_is_zero():
    rng = np.random.default_rng(2)
    q, k, v, la, b, _ = _rand(rng, 33, 3, 8, 8, beta=0.0)
    out, S = oracle.forward(q, k, v, la, b, None)
    assert np.all(out == 0.0) and np.all(S == 0.0)


@pytest.mark.parametrize("dk,dv", [(6, 4), (8, 8)])
def test_single_token_closed_form(dk, dv):
    """T = 1 from a zero state: S_1 = beta k v^T and o = beta (q.k) v."""
    rng = np.random.default_rng(3)
    q, k, v, la, b, _ = _rand(rng, 1, 4, dk, dv, unit_k=False)
    out, S = oracle.forward(q, k, v, la, b, None)
    for h in range(4):
        np.testing.assert_allclose(out[0, h], b[0, h] * (q[0, h] @ k[0, h]) * v[0, h],
                                   rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(S[0, h], b[0, h] * np.outer(k[0, h], v[0, h]),
                                   rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("la_value", [-5.0, -7.5, -1e6])
def test_clamped_floor_decay(la_value):
    """log_alpha at or below the floor acts as exactly -5 per step; with beta = 0
    the state is only decayed: S_t = e^{-5t} S0 and o_t = e^{-5t} S0^T q_t."""
    rng = np.random.default_rng(4)
    T, H, dk, dv = 12, 2, 5, 7
    q, k, v, _, _, S0 = _rand(rng, T, H, dk, dv, s0=1.0)
    la = np.full((T, H, dk), la_value)
    b = np.zeros((T, H))
    out, S = oracle.forward(q, k, v, la, b, S0)
    for t in range(T):
        for h in range(H):
            want = math.exp(-5.0 * (t + 1)) * (S0[0, h].T @ q[t, h])
            np.testing.assert_allclose(out[t, h], want, rtol=1e-12, atol=0)
    np.testing.assert_allclose(S, math.exp(-5.0 * T) * S0, rtol=1e-12, atol=0)


def test_positive_log_alpha_clamped_to_no_decay():
    rng = np.random.default_rng(5)
    q, k, v, _, _, S0 = _rand(rng, 9, 1, 4, 3, s0=1.0)
    la = np.full((9, 1, 4), 0.7)
    out, S = oracle.forward(q, k, v, la, np.zeros((9, 1)), S0)
    np.testing.assert_allclose(S, S0, rtol=0, atol=0)


def test_per_channel_decay_axis_and_time_index():
    """beta = 0, time- and channel-varying log_alpha: S_t = Diag(exp(sum_{s<=t} la_s)) S0.
    Row c of S (key channel c) decays with channel c; the gate of token t acts
    at step t (not t-1).  dk != dv so a transposed state cannot pass."""
    rng = np.random.default_rng(6)
    T, H, dk, dv = 10, 2, 6, 3
    q, k, v, la, _, S0 = _rand(rng, T, H, dk, dv, la_lo=-2.0, la_hi=0.0, s0=1.0)
    out, S = oracle.forward(q, k, v, la, np.zeros((T, H)), S0)
    G = np.cumsum(la, axis=0)  # [T, H, dk]
    for t in range(T):
        for h in range(H):
            St = np.exp(G[t, h])[:, None] * S0[0, h]
            np.testing.assert_allclose(out[t, h], St.T @ q[t, h], rtol=1e-12, atol=1e-15)
    for h in range(H):
        np.testing.assert_allclose(S[0, h], np.exp(G[-1, h])[:, None] * S0[0, h], rtol=1e-12)


@pytest.mark.parametrize("dk,dv,T", [(16, 8, 16), (12, 12, 7)])
def test_orthonormal_keys_reduce_to_linear_attention(dk, dv, T):
    """No decay, beta = 1, orthonormal keys, zero state: every delta write lands
    on a direction no earlier key touched, so the layer is plain causal linear
    attention: S_T = K^T V and o_t = sum_{i<=t} (q_t . k_i) v_i."""
    rng = np.random.default_rng(7)
    H = 2
    q = rng.standard_normal((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    k = np.empty((T, H, dk))
    for h in range(H):
        Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
        k[:, h] = Qm[:, :T].T
    la = np.zeros((T, H, dk))
    b = np.ones((T, H))
    out, S = oracle.forward(q, k, v, la, b, None)
    for h in range(H):
        scores = np.tril(q[:, h] @ k[:, h].T)
        np.testing.assert_allclose(out[:, h], scores @ v[:, h], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(S[0, h], k[:, h].T @ v[:, h], rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- second algorithm

@pytest.mark.parametrize("chunk", [1, 4, 16, 64])
@pytest.mark.parametrize("T", [1, 5, 17, 64, 70, 130])
def test_chunked_ut_form_matches_recurrence(chunk, T):
    rng = np.random.default_rng(100 + T + chunk)
    q, k, v, la, b, S0 = _rand(rng, T, 2, 8, 6, la_lo=-6.0, la_hi=0.5, s0=0.3)
    ref_o, ref_S = oracle.forward(q, k, v, la, b, S0)
    o, S = naive_chunked.forward(q, k, v, la, b, S0, chunk=chunk)
    assert _rel(o, ref_o) < 1e-10
    assert _rel(S, ref_S) < 1e-10


def test_chunked_ut_form_matches_recurrence_varlen_and_weak_decay():
    rng = np.random.default_rng(11)
    lens = [3, 64, 1, 90, 17]
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, la, b, S0 = _rand(rng, T, 2, 8, 8, la_lo=-0.05, la_hi=0.0, s0=0.3,
                               n_seqs=len(lens))
    ref_o, ref_S = oracle.forward(q, k, v, la, b, S0, cu)
    o, S = naive_chunked.forward(q, k, v, la, b, S0, cu, chunk=16)
    assert _rel(o, ref_o) < 1e-10
    assert _rel(S, ref_S) < 1e-10


def test_scalar_decay_is_rescaled_ungated_delta_rule():
    """All channels share one decay per token (the scalar-gated case).  Then
    Diag(alpha) commutes with (I - beta k k^T), so S_t = G_t R_t with
    G_t = prod_{s<=t} alpha_s and R the ungated delta rule driven by v_t / G_t."""
    rng = np.random.default_rng(12)
    T, H, dk, dv = 20, 2, 6, 5
    q, k, v, _, b, S0 = _rand(rng, T, H, dk, dv, s0=0.5)
    la_tok = rng.uniform(-0.3, 0.0, size=(T, H))
    la = np.repeat(la_tok[:, :, None], dk, axis=2)
    G = np.exp(np.cumsum(la_tok, axis=0))  # [T, H]
    out, S = oracle.forward(q, k, v, la, b, S0)
    outR, SR = oracle.forward(q, k, v / G[:, :, None], np.zeros_like(la), b, S0)
    np.testing.assert_allclose(out, outR * G[:, :, None], rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(S[0], SR[0] * G[-1][:, None, None], rtol=1e-10, atol=1e-13)


# ---------------------------------------------------------------- invariants

def test_linearity_in_values_and_state():
    rng = np.random.default_rng(13)
    q, k, v1, la, b, S01 = _rand(rng, 50, 2, 8, 8, s0=0.4)
    v2 = rng.standard_normal(v1.shape)
    S02 = rng.standard_normal(S01.shape)
    c = -1.7
    o1, s1 = oracle.forward(q, k, v1, la, b, S01)
    o2, s2 = oracle.forward(q, k, v2, la, b, S02)
    o3, s3 = oracle.forward(q, k, v1 + c * v2, la, b, S01 + c * S02)
    assert _rel(o3, o1 + c * o2) < 1e-12
    assert _rel(s3, s1 + c * s2) < 1e-12


def test_continuation_across_calls():
    rng = np.random.default_rng(14)
    q, k, v, la, b, S0 = _rand(rng, 77, 2, 8, 4, la_lo=-0.5, s0=0.4)
    o, S = oracle.forward(q, k, v, la, b, S0)
    cut = 31
    oa, Sa = oracle.forward(q[:cut], k[:cut], v[:cut], la[:cut], b[:cut], S0)
    ob, Sb = oracle.forward(q[cut:], k[cut:], v[cut:], la[cut:], b[cut:], Sa)
    np.testing.assert_allclose(np.concatenate([oa, ob]), o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(Sb, S, rtol=0, atol=1e-13)


def test_packed_sequences_equal_separate_calls():
    rng = np.random.default_rng(15)
    lens = [5, 0, 19, 1, 40]
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, la, b, S0 = _rand(rng, sum(lens), 3, 8, 8, s0=0.4, n_seqs=len(lens))
    o, S = oracle.forward(q, k, v, la, b, S0, cu)
    for n in range(len(lens)):
        t0, t1 = cu[n], cu[n + 1]
        on, Sn = oracle.forward(q[t0:t1], k[t0:t1], v[t0:t1], la[t0:t1], b[t0:t1],
                                S0[n:n + 1])
        assert np.array_equal(o[t0:t1], on)
        assert np.array_equal(S[n], Sn[0])
    # an empty sequence hands its initial state straight through
    assert np.array_equal(S[1], S0[1])


def test_segment_transition_and_increment_compose():
    """A segment maps its entry state affinely: S_end = M S_in + B, where B is
    the segment run from a zero state and M is the segment applied to the
    identity with v = 0 (the increment / transition pair used to split a long
    sequence)."""
    rng = np.random.default_rng(16)
    dk, dv, T = 8, 6, 45
    q, k, v, la, b, S_in = _rand(rng, T, 2, dk, dv, la_lo=-0.4, s0=0.7)
    _, B = oracle.forward(q, k, v, la, b, None)
    eye = np.broadcast_to(np.eye(dk), (1, 2, dk, dk)).copy()
    _, M = oracle.forward(q, k, np.zeros((T, 2, dk)), la, b, eye)
    _, S_end = oracle.forward(q, k, v, la, b, S_in)
    for h in range(2):
        assert _rel(M[0, h] @ S_in[0, h] + B[0, h], S_end[0, h]) < 1e-12


def test_state_norm_never_grows_without_writes():
    """With v = 0, beta in [0, 1] and unit keys, each step multiplies the state
    by Diag(alpha) (entries <= 1) and then by I - beta k k^T, whose spectrum is
    {1, 1 - beta}: column norms never grow.  (A flipped sign, I + beta k k^T,
    would grow them.)"""
    rng = np.random.default_rng(17)
    T, dk, dv = 30, 8, 3
    q, k, v, la, b, S0 = _rand(rng, T, 1, dk, dv, la_lo=-0.2, s0=1.0)
    v[:] = 0.0
    prev = np.linalg.norm(S0[0, 0], axis=0)
    for t in range(1, T + 1):
        _, S = oracle.forward(q[:t], k[:t], v[:t], la[:t], b[:t], S0)
        cur = np.linalg.norm(S[0, 0], axis=0)
        assert np.all(cur <= prev * (1 + 1e-14))
        prev = cur


# ---------------------------------------------------------------- encodings

def test_bf16_inputs_widen_exactly():
    """The bf16/f32 input encoding gives the same result as the same values
    passed in fp64 (torch's own bf16 -> fp64 conversion decodes them)."""
    p = kin.make_prefill([37, 5], 2, 16, 8, seed=9, s0_std=0.02)
    o1, S1 = oracle.forward(kin.bf16_bits(p.q), kin.bf16_bits(p.k), kin.bf16_bits(p.v),
                            p.log_alpha.numpy(), p.beta.numpy(), p.S0.numpy(), p.cu_seqlens)
    f = lambda t: t.to(torch.float64).numpy()
    o2, S2 = oracle.forward(f(p.q), f(p.k), f(p.v), f(p.log_alpha), f(p.beta), f(p.S0),
                            p.cu_seqlens)
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)


def test_head_subset_matches_full():
    p = kin.make_prefill([20, 11], 4, 8, seed=10, s0_std=0.02)
    args = (kin.bf16_bits(p.q), kin.bf16_bits(p.k), kin.bf16_bits(p.v),
            p.log_alpha.numpy(), p.beta.numpy(), p.S0.numpy(), p.cu_seqlens)
    o, S = oracle.forward(*args)
    o2, S2 = oracle.forward(*args, heads=(1, 3))
    assert np.array_equal(o[:, 1:3], o2) and np.array_equal(S[:, 1:3], S2)


def test_decode_steps_chain_single_token_calls():
    d = kin.make_decode(3, 2, 8, 4, steps=5, seed=21)
    out, S = oracle.decode_steps(kin.bf16_bits(d.q), kin.bf16_bits(d.k), kin.bf16_bits(d.v),
                                 d.log_alpha.numpy(), d.beta.numpy(), d.S.numpy())
    Sref = d.S.numpy().astype(np.float64)
    f = lambda t: t.to(torch.float64).numpy()
    for s in range(5):
        cu = np.arange(4, dtype=np.int64)
        o_s, Sref = oracle.forward(f(d.q[s]), f(d.k[s]), f(d.v[s]), f(d.log_alpha[s]),
                                   f(d.beta[s]), Sref, cu)
        np.testing.assert_allclose(out[s], o_s, rtol=0, atol=1e-15)
    np.testing.assert_allclose(S, Sref, rtol=0, atol=1e-15)


# ---------------------------------------------------------------- printed facts

def _golden_facts():
    facts = {}
    with open(os.path.join(GOLDEN, "decay_bound_facts.txt")) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                key, val = (s.strip() for s in line.split("="))
                facts[key] = float(val)
    return facts


def test_printed_decay_bound_facts():
    f = _golden_facts()
    floor = f["log_decay_floor"]
    # e^-5 kept per step, printed as 0.67 %
    assert round(100 * math.exp(floor), 2) == f["step_floor_percent"]
    # 16 steps at the floor accumulate exactly the printed tile bound
    assert f["tile_tokens"] * floor == f["tile_log_decay_bound"]
    # e^80 rounds to the printed 5.5e34 and sits below the printed bf16 range,
    # which is bf16's largest finite value to two figures
    assert float(f"{math.exp(-f['tile_log_decay_bound']):.1e}") == f["tile_reciprocal_bound"]
    bf16_max = torch.finfo(torch.bfloat16).max
    assert float(f"{bf16_max:.1e}") == f["bf16_max_approx"]
    assert math.exp(-f["tile_log_decay_bound"]) < bf16_max
    assert torch.isfinite(torch.tensor(math.exp(80.0), dtype=torch.bfloat16))


def test_oracle_decay_over_one_tile_matches_printed_bound():
    """The oracle's floor is the printed one: one tile of floor decays scales
    the state by exactly e^{tile bound}."""
    f = _golden_facts()
    n = int(f["tile_tokens"])
    rng = np.random.default_rng(22)
    q, k, v, _, _, S0 = _rand(rng, n, 1, 4, 4, s0=1.0)
    la = np.full((n, 1, 4), -100.0)  # far below the floor
    _, S = oracle.forward(q, k, v, la, np.zeros((n, 1)), S0)
    np.testing.assert_allclose(S, math.exp(f["tile_log_decay_bound"]) * S0, rtol=1e-12)
