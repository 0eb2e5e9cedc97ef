"""A numpy model of the prefill kernel's arithmetic plan, against the fp64 oracle.

The model is neither the oracle nor the CUDA path, and shares nothing with
either.  It restates the chunked form in fp32:
- 64-token chunks and the chunk-local cumulative log-decay g;
- two 32-token strips, each anchored at its 16th token G, for the intra-chunk
  products A_kk (times beta, strictly lower) and A_qk (lower, diagonal
  included);
- T = (I + A_kk)^{-1} Diag(beta);
- U = T V - T P, with P = (k e^g) S;
- O = (q e^g) S + A_qk U;
- S <- Diag(e^{g_last}) S + K'^T U, with K' = k e^{g_last - g}.

Each operand is rounded the way the kernel rounds it:
- the strip products take bf16 operands;
- T enters the product with V as a bf16 hi + lo pair;
- T against -P, and P, k e^g, q e^g, A_qk, U and K', are tf32 rounded to
  nearest;
- S is read by the tensor core as tf32 (modelled truncated; rounding it or
  keeping fp32 changes the results below in the fourth digit);
- out is rounded to bf16.

On the weak-decay input below, the model gives out rel-L2 2.70e-3 and state
rel-L2 5.28e-4, the errors the GPU kernel has on the same input.  The tests
check:
- the model's algebra, with every rounding off, for both paths;
- that the plan keeps the state within its tolerance;
- that the two cheaper plans the kernel avoids do not: bf16 T against V
  breaks the state tolerance, and truncated tf32 takes most of its margin;
- that splitting a sequence into segments adds no error to the plan.

Weak decay (log alpha = -0.03 on every channel) carries the state across
all 32 chunks of each sequence.  Under strong decay the final state forgets
state-path errors within a chunk or two.

The split path is modelled the same way, with three steps:
- the summary pass, per non-final segment, from a zero state (increment B)
  and from the identity (transition M), in the W form the summary kernel
  uses.  -W = -(T (k e^g)) is rounded to tf32; then U_B = U~ - W S_B,
  U_M = -W S_M, and S_B, S_M are updated like S;
- the fp32 scan S_in(j+1) = M_j S_in(j) + B_j;
- the replay of every segment from its entry state.
Its tests use slower decay (log alpha = -0.003, e^-1.5 over a 512-token
segment), so that the transition M carries the entry state.  At -0.03 a
segment scales it by e^-15, and M would hardly enter the result.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_48_gb300 import inputs as kin
from kda_testlib import OUT_REL_L2, STATE_REL_L2, rel_l2

F32 = np.float32
C = 64


def tf32_rn(x):
    """fp32 -> tf32, round to nearest (ties away): add half a tf32 ulp, clear 13 bits."""
    u = np.ascontiguousarray(x, dtype=F32).view(np.uint32).astype(np.uint64)
    return ((u + 0x1000) & 0xFFFFE000).astype(np.uint32).view(F32)


def tf32_trunc(x):
    u = np.ascontiguousarray(x, dtype=F32).view(np.uint32)
    return (u & np.uint32(0xFFFFE000)).view(F32)


def bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=F32)).to(torch.bfloat16).float().numpy()


def exact(x):
    return np.asarray(x, dtype=F32)


PLAN = dict(strip=bf16, t_p=tf32_rn, t_v="hi+lo", p=tf32_rn, kg=tf32_rn, u=tf32_rn,
            kp=tf32_rn, qg=tf32_rn, aqk=tf32_rn, s_op=tf32_trunc, out=bf16)
NO_ROUNDING = dict(strip=exact, t_p=exact, t_v="exact", p=exact, kg=exact, u=exact,
                   kp=exact, qg=exact, aqk=exact, s_op=exact, out=exact)


def chunked_head(q, k, v, log_alpha, beta, S0, r):
    """One (sequence, head) chain: q, k [T, dk], v [T, dv], log_alpha [T, dk],
    beta [T], S0 [dk, dv]; r = the rounding of each operand (PLAN's keys)."""
    T = q.shape[0]
    S = S0.astype(F32).copy()
    out = np.zeros((T, v.shape[1]), F32)
    for c0 in range(0, T, C):
        n = min(C, T - c0)
        qc, kc, vc = q[c0:c0 + n], k[c0:c0 + n], v[c0:c0 + n]
        b = beta[c0:c0 + n].astype(F32)
        g = np.cumsum(np.clip(log_alpha[c0:c0 + n], -5.0, 0.0).astype(F32), axis=0, dtype=F32)
        Akk = np.zeros((n, n), F32)
        Aqk = np.zeros((n, n), F32)
        for s in range(2):
            r0, r1 = 32 * s, min(32 * s + 32, n)
            if r0 >= n:
                continue
            G = g[min(32 * s + 15, n - 1)]
            with np.errstate(over="ignore", invalid="ignore"):  # masked entries only
                kb = r["strip"](kc[:r1] * np.exp(G - g[:r1]))
                Aqk[r0:r1, :r1] = r["strip"](qc[r0:r1] * np.exp(g[r0:r1] - G)) @ kb.T
                Akk[r0:r1, :r1] = r["strip"](kc[r0:r1] * np.exp(g[r0:r1] - G)) @ kb.T
        Akk = np.where(np.tri(n, k=-1, dtype=bool), Akk, 0).astype(F32) * b[:, None]
        Aqk = np.where(np.tri(n, dtype=bool), Aqk, 0).astype(F32)
        Tm = np.linalg.inv(np.eye(n) + Akk).astype(F32) * b[None, :]
        Sop = r["s_op"](S)
        P = r["kg"](kc * np.exp(g)) @ Sop
        if r["t_v"] == "hi+lo":
            hi = bf16(Tm)
            TV = hi @ vc + bf16(Tm - hi) @ vc
        elif r["t_v"] == "bf16":
            TV = bf16(Tm) @ vc
        else:
            TV = Tm @ vc
        U = r["u"](r["t_p"](Tm) @ (-r["p"](P)) + TV)
        out[c0:c0 + n] = r["out"](r["qg"](qc * np.exp(g)) @ Sop + r["aqk"](Aqk) @ U)
        S = S * np.exp(g[-1])[:, None] + r["kp"](kc * np.exp(g[-1] - g)).T @ U
    return out, S


def summary_head(k, v, log_alpha, beta, r):
    """Increment B and transition M of one segment of one head (S_end = M S_in + B)."""
    T, d = k.shape
    SB = np.zeros((d, v.shape[1]), F32)
    SM = np.eye(d, dtype=F32)
    for c0 in range(0, T, C):
        n = min(C, T - c0)
        kc, vc = k[c0:c0 + n], v[c0:c0 + n]
        b = beta[c0:c0 + n].astype(F32)
        g = np.cumsum(np.clip(log_alpha[c0:c0 + n], -5.0, 0.0).astype(F32), axis=0, dtype=F32)
        Akk = np.zeros((n, n), F32)
        for s in range(2):
            r0, r1 = 32 * s, min(32 * s + 32, n)
            if r0 >= n:
                continue
            G = g[min(32 * s + 15, n - 1)]
            with np.errstate(over="ignore", invalid="ignore"):  # masked entries only
                kb = r["strip"](kc[:r1] * np.exp(G - g[:r1]))
                Akk[r0:r1, :r1] = r["strip"](kc[r0:r1] * np.exp(g[r0:r1] - G)) @ kb.T
        Akk = np.where(np.tri(n, k=-1, dtype=bool), Akk, 0).astype(F32) * b[:, None]
        Tm = np.linalg.inv(np.eye(n) + Akk).astype(F32) * b[None, :]
        negW = r["p"](-(r["t_p"](Tm) @ r["kg"](kc * np.exp(g))))
        if r["t_v"] == "hi+lo":
            hi = bf16(Tm)
            TV = hi @ vc + bf16(Tm - hi) @ vc
        else:
            TV = Tm @ vc
        UB = r["u"](TV + negW @ r["s_op"](SB))
        UM = r["u"](negW @ r["s_op"](SM))
        Kp = r["kp"](kc * np.exp(g[-1] - g))
        SB = SB * np.exp(g[-1])[:, None] + Kp.T @ UB
        SM = SM * np.exp(g[-1])[:, None] + Kp.T @ UM
    return SB, SM


def split_head(q, k, v, log_alpha, beta, S0, seg, r):
    """One chain cut into segments of `seg` tokens: summary, scan, replay."""
    T = q.shape[0]
    bounds = list(range(0, T, seg)) + [T]
    entry = [S0.astype(F32)]
    for j in range(len(bounds) - 2):
        a, e = bounds[j], bounds[j + 1]
        B, M = summary_head(k[a:e], v[a:e], log_alpha[a:e], beta[a:e], r)
        entry.append((M @ entry[-1] + B).astype(F32))
    out = np.zeros((T, v.shape[1]), F32)
    S = entry[0]
    for j in range(len(bounds) - 1):
        a, e = bounds[j], bounds[j + 1]
        out[a:e], S = chunked_head(q[a:e], k[a:e], v[a:e], log_alpha[a:e], beta[a:e], entry[j], r)
    return out, S


@pytest.fixture(scope="module")
def weak_decay():
    p = kin.make_prefill([2048, 2048], 2, 128, seed=11, s0_std=0.05, log_alpha_fixed=-0.03)
    ref_o, ref_S = oracle.forward(kin.bf16_bits(p.q), kin.bf16_bits(p.k), kin.bf16_bits(p.v),
                                  p.log_alpha.numpy(), p.beta.numpy(), p.S0.numpy(),
                                  p.cu_seqlens)
    return p, ref_o, ref_S


@pytest.fixture(scope="module")
def slow_decay():
    p = kin.make_prefill([2048, 2048], 2, 128, seed=12, s0_std=0.05, log_alpha_fixed=-0.003)
    ref_o, ref_S = oracle.forward(kin.bf16_bits(p.q), kin.bf16_bits(p.k), kin.bf16_bits(p.v),
                                  p.log_alpha.numpy(), p.beta.numpy(), p.S0.numpy(),
                                  p.cu_seqlens)
    return p, ref_o, ref_S


def model_errors(case, rounding, seg=0):
    p, ref_o, ref_S = case
    q, k, v = (t.float().numpy() for t in (p.q, p.k, p.v))
    la, be, S0 = p.log_alpha.numpy(), p.beta.numpy(), p.S0.numpy()
    out = np.zeros_like(ref_o)
    S = np.zeros_like(ref_S)
    for n in range(p.n_seqs):
        a, e = p.cu_seqlens[n], p.cu_seqlens[n + 1]
        for h in range(p.H):
            if seg:
                out[a:e, h], S[n, h] = split_head(q[a:e, h], k[a:e, h], v[a:e, h], la[a:e, h],
                                                  be[a:e, h], S0[n, h], seg, rounding)
            else:
                out[a:e, h], S[n, h] = chunked_head(q[a:e, h], k[a:e, h], v[a:e, h],
                                                    la[a:e, h], be[a:e, h], S0[n, h], rounding)
    return rel_l2(out, ref_o), rel_l2(S, ref_S)


def test_model_without_roundings_matches_the_oracle(weak_decay):
    eo, es = model_errors(weak_decay, NO_ROUNDING)
    assert eo < 2e-5 and es < 2e-5, (eo, es)


def test_kernel_plan_keeps_out_and_state_within_tolerance(weak_decay):
    eo, es = model_errors(weak_decay, PLAN)
    assert eo < OUT_REL_L2 and es < 0.7 * STATE_REL_L2, (eo, es)


def test_bf16_T_against_V_breaks_the_state_tolerance(weak_decay):
    _, es = model_errors(weak_decay, dict(PLAN, t_v="bf16"))
    assert es > STATE_REL_L2, es


def test_truncated_tf32_takes_most_of_the_state_margin(weak_decay):
    _, es_plan = model_errors(weak_decay, PLAN)
    trunc = dict(PLAN, **{key: tf32_trunc for key in ("t_p", "p", "kg", "u", "kp", "qg", "aqk")})
    _, es = model_errors(weak_decay, trunc)
    assert es > 1.5 * es_plan and es > 0.8 * STATE_REL_L2, (es, es_plan)


def test_split_model_without_roundings_matches_the_oracle(slow_decay):
    eo, es = model_errors(slow_decay, NO_ROUNDING, seg=512)
    assert eo < 2e-5 and es < 2e-5, (eo, es)


def test_split_path_adds_no_error_to_the_plan(slow_decay):
    eo, es = model_errors(slow_decay, PLAN)
    eo_s, es_s = model_errors(slow_decay, PLAN, seg=512)
    assert es < STATE_REL_L2 and eo < OUT_REL_L2, (eo, es)
    assert abs(es_s - es) < 0.05 * es and abs(eo_s - eo) < 0.05 * eo, (eo, es, eo_s, es_s)
