"""The fused entry points (input preparation on load) vs the fp64 oracle.

kda_chunk_fwd_fused / kda_decode_step_fused take raw q, k and bf16 gate
logits; the oracle prepares the same raw values its own way (oracle.prep)
and runs the recurrence.  Same tolerances as the unfused path.
"""
import numpy as np
import pytest
import torch

from oracle import prep
from gated_delta_rule_48_gb300 import binding as kb
from gated_delta_rule_48_gb300 import inputs as kin
from kda_testlib import check_out, check_state

pytestmark = pytest.mark.gpu


def _dev(p, uniform=False):
    d = dict(q=p.q_raw.cuda(), k=p.k_raw.cuda(), v=p.v.cuda(), g=p.gate.cuda(),
             b=p.beta.cuda(), S0=None if p.S0 is None else p.S0.cuda())
    d["cu"] = None if uniform else torch.from_numpy(p.cu_seqlens.astype(np.int32)).cuda()
    return d


def run_fused(p, uniform=False):
    d = _dev(p, uniform)
    out, S = kb.kda_chunk_fwd_fused(d["q"], d["k"], d["v"], d["g"], d["b"], d["S0"], d["cu"],
                                    n_seqs=p.n_seqs)
    assert kb.kda_get_device_error() == 0
    return out.float().cpu().numpy(), S.cpu().numpy()


def oracle_fused(p, heads=None):
    return prep.forward_fused(kin.bf16_bits(p.q_raw), kin.bf16_bits(p.k_raw), kin.bf16_bits(p.v),
                              kin.bf16_bits(p.gate), p.beta.numpy(),
                              None if p.S0 is None else p.S0.numpy(), p.cu_seqlens, heads=heads)


@pytest.mark.parametrize("d", [64, 128])
def test_fused_prefill_varlen(d):
    p = kin.make_prefill_raw([1, 0, 63, 64, 65, 300, 17], 3, d, seed=31, s0_std=0.05)
    out, S = run_fused(p)
    ref_o, ref_S = oracle_fused(p)
    check_out(out, ref_o)
    check_state(S, ref_S)


def test_fused_prefill_batched_b4_h32_t4096():
    p = kin.make_prefill_raw([4096] * 4, 32, 128, seed=32, s0_std=0.02)
    out, S = run_fused(p, uniform=True)
    ref_o, ref_S = oracle_fused(p)
    check_out(out, ref_o)
    check_state(S, ref_S)


@pytest.mark.parametrize("d", [64, 128])
def test_fused_prefill_long_sequence_is_split(d):
    # 2 heads x 1 sequence cannot fill the GPU, so the summary / scan / replay path runs
    p = kin.make_prefill_raw([6000], 2, d, seed=33, s0_std=0.02)
    out, S = run_fused(p)
    ref_o, ref_S = oracle_fused(p)
    check_out(out, ref_o)
    check_state(S, ref_S)


def test_fused_prefill_blind_to_projection_scale():
    """Scaling q_raw, k_raw by 8 (exact in bf16) leaves every result bit-identical."""
    p = kin.make_prefill_raw([500, 200], 4, 128, seed=34, s0_std=0.02)
    a_out, a_S = run_fused(p)
    p.q_raw = p.q_raw * 8
    p.k_raw = p.k_raw * 8
    b_out, b_S = run_fused(p)
    np.testing.assert_array_equal(a_out, b_out)
    np.testing.assert_array_equal(a_S, b_S)


@pytest.mark.parametrize("d", [64, 128])
def test_fused_decode_steps(d):
    r = kin.make_decode_raw(64, 4, d, steps=8, seed=35)
    S = r.S.cuda()
    qs, ks, vs, gs, bs = (t.cuda() for t in (r.q_raw, r.k_raw, r.v, r.gate, r.beta))
    outs = [kb.kda_decode_step_fused(qs[s], ks[s], vs[s], gs[s], bs[s], S) for s in range(8)]
    out = torch.stack(outs).float().cpu().numpy()
    ref_o, ref_S = prep.decode_steps_fused(kin.bf16_bits(r.q_raw), kin.bf16_bits(r.k_raw),
                                           kin.bf16_bits(r.v), kin.bf16_bits(r.gate),
                                           r.beta.numpy(), r.S.numpy())
    check_out(out, ref_o)
    check_state(S.cpu().numpy(), ref_S)


def test_fused_decode_tokens_with_commit():
    """K raw tokens per call, partial commits: outputs of all K tokens and the
    committed states against the oracle's prepared recurrence."""
    r = kin.make_decode_raw(24, 2, 128, steps=5, seed=36)
    f = lambda t: t.transpose(0, 1).contiguous()
    q, k, v, g, b = (f(t) for t in (r.q_raw, r.k_raw, r.v, r.gate, r.beta))
    commit = np.array([5, 0, 2, 3] * 6, dtype=np.int32)
    S = r.S.cuda()
    out = kb.kda_decode_tokens_fused(q.cuda(), k.cuda(), v.cuda(), g.cuda(), b.cuda(), S,
                                     torch.from_numpy(commit).cuda())
    assert kb.kda_get_device_error() == 0
    N, K = 24, 5
    flat = lambda t: t.reshape((N * K,) + tuple(t.shape[2:]))
    bits = lambda t: kin.bf16_bits(flat(t))
    ref_o, _ = prep.forward_fused(bits(q), bits(k), bits(v), bits(g), flat(b).numpy(), r.S.numpy(),
                                  np.arange(N + 1) * K)
    check_out(out.float().cpu().numpy().reshape(ref_o.shape), ref_o)
    keep = np.concatenate([np.arange(n * K, n * K + c) for n, c in enumerate(commit)]).astype(int)
    _, ref_S = prep.forward_fused(bits(q)[keep], bits(k)[keep], bits(v)[keep], bits(g)[keep],
                                  flat(b).numpy()[keep], r.S.numpy(),
                                  np.concatenate([[0], np.cumsum(commit)]))
    check_state(S.cpu().numpy(), ref_S)


def test_fused_decode_tokens_several_batches():
    """Raw projections, K = 11 (two batches of the kernel's 8), partial commits."""
    K, N = 11, 16
    r = kin.make_decode_raw(N, 2, 128, steps=K, seed=37)
    f = lambda t: t.transpose(0, 1).contiguous()
    q, k, v, g, b = (f(t) for t in (r.q_raw, r.k_raw, r.v, r.gate, r.beta))
    commit = np.array([11, 0, 7, 8, 9, 3, 10, 1] * 2, dtype=np.int32)
    S = r.S.cuda()
    out = kb.kda_decode_tokens_fused(q.cuda(), k.cuda(), v.cuda(), g.cuda(), b.cuda(), S,
                                     torch.from_numpy(commit).cuda())
    assert kb.kda_get_device_error() == 0
    flat = lambda t: t.reshape((N * K,) + tuple(t.shape[2:]))
    bits = lambda t: kin.bf16_bits(flat(t))
    ref_o, _ = prep.forward_fused(bits(q), bits(k), bits(v), bits(g), flat(b).numpy(), r.S.numpy(),
                                  np.arange(N + 1) * K)
    check_out(out.float().cpu().numpy().reshape(ref_o.shape), ref_o)
    keep = np.concatenate([np.arange(n * K, n * K + c) for n, c in enumerate(commit)]).astype(int)
    _, ref_S = prep.forward_fused(bits(q)[keep], bits(k)[keep], bits(v)[keep], bits(g)[keep],
                                  flat(b).numpy()[keep], r.S.numpy(),
                                  np.concatenate([[0], np.cumsum(commit)]))
    check_state(S.cpu().numpy(), ref_S)
