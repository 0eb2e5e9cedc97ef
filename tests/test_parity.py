"""GPU path vs the fp64 oracle, element by element, on the same seeded inputs.

Tolerances (see kda_testlib): out max|err| <= 2e-2 and relative L2 <= 5e-3;
final state relative L2 <= 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_48_gb300 import binding as kb
from gated_delta_rule_48_gb300 import inputs as kin
from kda_testlib import (check_out, check_state, oracle_prefill, rel_l2, to_device)

pytestmark = pytest.mark.gpu


def run_gpu(p, segment_tokens=0):
    d = to_device(p)
    out, S = kb.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"],
                              d["cu_seqlens"], n_seqs=p.n_seqs, segment_tokens=segment_tokens)
    assert kb.kda_get_device_error() == 0
    return out.float().cpu().numpy(), S.cpu().numpy()


def compare(p, segment_tokens=0, heads=None):
    out, S = run_gpu(p, segment_tokens)
    ref_o, ref_S = oracle_prefill(p, heads=heads)
    if heads is not None:
        out, S = out[:, heads[0]:heads[1]], S[:, heads[0]:heads[1]]
    check_out(out, ref_o)
    check_state(S, ref_S)
    return out, S


# ---------------------------------------------------------------- named workloads

def test_workload0_tiny():
    compare(kin.workload(0))


def test_workload1_batched_prefill():
    compare(kin.workload(1))


def test_workload2_stress_bound():
    compare(kin.workload(2))


def test_workload3_million_token_varlen_heads01():
    compare(kin.workload(3), heads=(0, 2))


def test_workload4_batched_decode_64_steps():
    d = kin.decode_workload(steps=64)
    S = d.S.cuda()
    qs, ks, vs = d.q.cuda(), d.k.cuda(), d.v.cuda()
    las, bs = d.log_alpha.cuda(), d.beta.cuda()
    outs = []
    for s in range(64):
        outs.append(kb.kda_decode_step(qs[s], ks[s], vs[s], las[s], bs[s], S))
    out = torch.stack(outs).float().cpu().numpy()
    ref_o, ref_S = oracle.decode_steps(kin.bf16_bits(d.q), kin.bf16_bits(d.k),
                                       kin.bf16_bits(d.v), d.log_alpha.numpy(),
                                       d.beta.numpy(), d.S.numpy())
    check_out(out, ref_o)
    check_state(S.cpu().numpy(), ref_S)


# ---------------------------------------------------------------- shapes and edges

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("T", [1, 15, 16, 17, 63, 64, 65, 200])
def test_lengths_and_head_sizes(T, d):
    compare(kin.make_prefill([T, T], 2, d, seed=T + d, s0_std=0.02))


@pytest.mark.parametrize("d", [64, 128])
def test_varlen_short_and_long_with_empty(d):
    lens = [1, 0, 5, 64, 3, 700, 0, 17, 129]
    compare(kin.make_prefill(lens, 3, d, seed=31, s0_std=0.02))


@pytest.mark.parametrize("beta", [0.0, 1.0])
def test_beta_extremes(beta):
    compare(kin.make_prefill([300], 2, 128, seed=32, s0_std=0.02, beta_mode="const",
                             beta_value=beta))


@pytest.mark.parametrize("la", [-5.0, 0.0, -0.01])
def test_log_alpha_floor_and_no_decay(la):
    """-5 everywhere: every 16-token tile reaches the -80 bound exactly; 0 and
    -0.01: long memory, so the state hand-off across chunks is exercised."""
    compare(kin.make_prefill([333, 128], 2, 128, seed=33, s0_std=0.02, log_alpha_fixed=la))


def test_out_of_range_log_alpha_is_clamped():
    p = kin.make_prefill([150], 2, 64, seed=34, s0_std=0.02)
    la = p.log_alpha.numpy()
    la[::3] = -40.0
    la[1::7] = 3.0
    compare(p)


# ---------------------------------------------------------------- sequence split

@pytest.mark.parametrize("seg", [64, 128, 256])
@pytest.mark.parametrize("la", [None, 0.0, -0.02])
def test_segment_split_matches_oracle(seg, la):
    """Forced split of long sequences: summary (B, M) per segment, scan of the
    entry states, replay.  Weak decay makes the transitions matter."""
    lens = [700, 65, 0, 1000, 3]
    compare(kin.make_prefill(lens, 2, 128, seed=35, s0_std=0.05, log_alpha_fixed=la),
            segment_tokens=seg)


@pytest.mark.parametrize("seg,dk", [(64, 128), (192, 128), (128, 64)])
def test_uniform_split_matches_oracle(seg, dk):
    """Forced split of a uniform batch (cu_seqlens NULL): the first pass replays
    segment 0 of every sequence beside the middle segments' summaries, and the
    second pass replays the rest, every one but the last from the T records
    the first pass kept.  777 tokens per sequence end in a ragged chunk."""
    p = kin.make_prefill([777] * 3, 2, dk, seed=45, s0_std=0.05, log_alpha_fixed=-0.02)
    assert p.uniform
    compare(p, segment_tokens=seg)


def test_automatic_split_is_the_documented_length():
    """kda_chunk_fwd's automatic split is an explicit split at the length
    kda_auto_segment_tokens reports for this device: the same launches, so
    bit-identical results."""
    p = kin.make_prefill([3000, 1700], 2, 128, seed=38, s0_std=0.05, log_alpha_fixed=-0.02)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    L = kb.kda_auto_segment_tokens(p.total_T, p.n_seqs, p.H, sms, False)  # packed
    assert L > 0  # 4 chains on this part: the model splits
    d = to_device(p)
    auto = kb.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"],
                            d["cu_seqlens"], n_seqs=p.n_seqs, segment_tokens=0)
    expl = kb.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"],
                            d["cu_seqlens"], n_seqs=p.n_seqs, segment_tokens=L)
    assert kb.kda_get_device_error() == 0
    assert torch.equal(auto[0], expl[0]) and torch.equal(auto[1], expl[1])
    ref_o, ref_S = oracle_prefill(p)
    check_out(auto[0].float().cpu().numpy(), ref_o)
    check_state(auto[1].cpu().numpy(), ref_S)


def test_automatic_uniform_split_is_the_documented_length():
    """The same for a uniform batch (cu_seqlens NULL), where the first pass also
    replays segment 0 and the second pass loads the T records."""
    p = kin.make_prefill([4096] * 2, 2, 128, seed=46, s0_std=0.05, log_alpha_fixed=-0.02)
    assert p.uniform
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    L = kb.kda_auto_segment_tokens(p.total_T, p.n_seqs, p.H, sms, True)
    assert L > 0 and -(-4096 // L) >= 3  # 4 chains: several segments, so loaded replays run
    d = to_device(p)
    auto = kb.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"], None,
                            n_seqs=p.n_seqs, segment_tokens=0)
    expl = kb.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"], None,
                            n_seqs=p.n_seqs, segment_tokens=L)
    assert kb.kda_get_device_error() == 0
    assert torch.equal(auto[0], expl[0]) and torch.equal(auto[1], expl[1])
    ref_o, ref_S = oracle_prefill(p)
    check_out(auto[0].float().cpu().numpy(), ref_o)
    check_state(auto[1].cpu().numpy(), ref_S)


@pytest.mark.parametrize("seg", [0, 64])
def test_thousands_of_sequences(seg):
    """2,500 packed sequences of 0..199 tokens: the planner walks them in
    blocks of 1,024, and with 64-token segments it emits and orders some 5,000
    segments (several per chunk-count bucket)."""
    rng = np.random.default_rng(44)
    lens = [int(x) for x in rng.integers(0, 200, size=2500)]
    compare(kin.make_prefill(lens, 2, 64, seed=44, s0_std=0.05, log_alpha_fixed=-0.05),
            segment_tokens=seg)


def test_segment_split_d64_and_no_split_agree():
    p = kin.make_prefill([999, 257], 2, 64, seed=36, s0_std=0.05, log_alpha_fixed=-0.03)
    o1, S1 = compare(p, segment_tokens=128)
    o2, S2 = compare(p, segment_tokens=-1)
    assert rel_l2(o1, o2) < 5e-3 and rel_l2(S1, S2) < 1e-3


# ---------------------------------------------------------------- API contract

def test_state_aliasing_continuation():
    """S_final may alias S0: running T tokens in two calls equals one call."""
    p = kin.make_prefill([256], 2, 128, seed=37, s0_std=0.02, log_alpha_fixed=-0.05)
    d = to_device(p)
    full_o, full_S = kb.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                      d["S0"], None, n_seqs=1)
    S = d["S0"].clone()
    cut = 100
    o1, _ = kb.kda_chunk_fwd(d["q"][:cut], d["k"][:cut], d["v"][:cut], d["log_alpha"][:cut],
                             d["beta"][:cut], S, None, S_final=S, n_seqs=1)
    o2, _ = kb.kda_chunk_fwd(d["q"][cut:], d["k"][cut:], d["v"][cut:], d["log_alpha"][cut:],
                             d["beta"][cut:], S, None, S_final=S, n_seqs=1)
    o = torch.cat([o1, o2]).float().cpu().numpy()
    ref_o, ref_S = oracle_prefill(p)
    check_out(o, ref_o)
    check_state(S.cpu().numpy(), ref_S)


def test_decode_steps_equal_prefill_of_same_tokens():
    p = kin.make_prefill([64] * 4, 3, 128, seed=38, s0_std=0.02)
    d = to_device(p)
    out_p, S_p = kb.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"],
                                  None, n_seqs=4)
    S = d["S0"].clone()
    view = lambda t: t.view(4, 64, *t.shape[1:]).transpose(0, 1).contiguous()
    qs, ks, vs, las, bs = (view(d[x]) for x in ("q", "k", "v", "log_alpha", "beta"))
    outs = [kb.kda_decode_step(qs[t], ks[t], vs[t], las[t], bs[t], S) for t in range(64)]
    out_d = torch.stack(outs).transpose(0, 1).reshape(256, 3, 128)
    assert rel_l2(out_d.float().cpu().numpy(), out_p.float().cpu().numpy()) < 5e-3
    assert rel_l2(S.cpu().numpy(), S_p.cpu().numpy()) < 1e-3


def test_empty_sequences_hand_state_through():
    p = kin.make_prefill([0, 0, 0], 2, 64, seed=39, s0_std=0.1)
    d = to_device(p)
    S0 = torch.randn(3, 2, 64, 64, device="cuda")
    out, S = kb.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0,
                              d["cu_seqlens"], n_seqs=3)
    assert kb.kda_get_device_error() == 0
    assert torch.equal(S, S0)


def test_no_state_requested():
    p = kin.make_prefill([100], 2, 64, seed=40)
    d = to_device(p)
    out, S = kb.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], None, None,
                              n_seqs=1, want_state=False)
    assert S is None
    ref_o, _ = oracle_prefill(p)
    check_out(out.float().cpu().numpy(), ref_o)


@pytest.mark.parametrize("bad", ["first", "decreasing", "last"])
def test_malformed_cu_seqlens_sets_device_error(bad):
    p = kin.make_prefill([10, 20, 30], 2, 64, seed=41)
    d = to_device(p)
    cu = [0, 10, 30, 60]
    if bad == "first":
        cu[0] = 1
    elif bad == "decreasing":
        cu[2] = 5
    else:
        cu[3] = 59
    cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
    out = torch.full((60, 2, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    S = torch.full((3, 2, 64, 64), 7.0, dtype=torch.float32, device="cuda")
    kb.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], None, cu_t,
                     out=out, S_final=S)
    assert kb.kda_get_device_error() == 5  # KDA_ERR_DEVICE_INPUT
    assert kb.kda_get_device_error() == 0  # cleared
    assert bool((out == 7.0).all()) and bool((S == 7.0).all())
