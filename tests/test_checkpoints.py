"""kda_chunk_fwd_checkpoints: the state after every `interval` tokens of each
sequence, against the fp64 oracle run on the corresponding prefixes."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_48_gb300 import binding as kb
from gated_delta_rule_48_gb300 import inputs as kin
from kda_testlib import check_out, check_state, oracle_prefill

pytestmark = pytest.mark.gpu


def _oracle_checkpoints(p, interval):
    """State after j * interval tokens of each sequence = S_final of that prefix."""
    cu = p.cu_seqlens
    rows, lens, s0_idx = [], [], []
    for n in range(p.n_seqs):
        L = int(cu[n + 1] - cu[n])
        for j in range(1, L // interval + 1):
            rows.append(np.arange(cu[n], cu[n] + j * interval))
            lens.append(j * interval)
            s0_idx.append(n)
    if not rows:
        return np.zeros((0, p.H, p.dk, p.dv))
    idx = np.concatenate(rows)
    cu_p = np.concatenate([[0], np.cumsum(lens)])
    S0 = None if p.S0 is None else p.S0.numpy()[s0_idx]
    _, S = oracle.forward(kin.bf16_bits(p.q)[idx], kin.bf16_bits(p.k)[idx], kin.bf16_bits(p.v)[idx],
                          p.log_alpha.numpy()[idx], p.beta.numpy()[idx], S0, cu_p)
    return S


def _run(p, interval, max_ck):
    d = dict(q=p.q.cuda(), k=p.k.cuda(), v=p.v.cuda(), la=p.log_alpha.cuda(), b=p.beta.cuda())
    S0 = None if p.S0 is None else p.S0.cuda()
    cu = torch.from_numpy(p.cu_seqlens.astype(np.int32)).cuda()
    out, S, ck = kb.kda_chunk_fwd_checkpoints(d["q"], d["k"], d["v"], d["la"], d["b"], S0, cu,
                                              interval=interval, max_checkpoints=max_ck)
    return out, S, ck


@pytest.mark.parametrize("d", [64, 128])
def test_checkpoints_match_prefix_states(d):
    # lengths with and without a multiple of the interval, one shorter than it, an empty one
    p = kin.make_prefill([1024, 700, 0, 130, 1300], 2, d, seed=61, s0_std=0.05)
    interval = 256
    ref = _oracle_checkpoints(p, interval)            # 4 + 2 + 0 + 0 + 5 = 11
    assert ref.shape[0] == 11
    out, S, ck = _run(p, interval, ref.shape[0])
    assert kb.kda_get_device_error() == 0
    check_state(ck.cpu().numpy(), ref, "checkpoints")
    ref_o, ref_S = oracle_prefill(p)
    check_out(out.float().cpu().numpy(), ref_o)
    check_state(S.cpu().numpy(), ref_S)
    # a sequence whose length is a multiple of the interval: last checkpoint == S_final
    assert torch.equal(ck[3], S[0])


def test_checkpoints_through_the_split_path():
    # one long sequence, 2 heads: the automatic split runs summary / scan / replay
    p = kin.make_prefill([5000], 2, 128, seed=62, s0_std=0.02)
    ref = _oracle_checkpoints(p, 1024)
    out, S, ck = _run(p, 1024, ref.shape[0])
    assert kb.kda_get_device_error() == 0
    check_state(ck.cpu().numpy(), ref, "checkpoints")


def test_checkpoint_overflow_is_reported_and_results_still_written():
    p = kin.make_prefill([512, 512], 2, 64, seed=63, s0_std=0.05)
    ref = _oracle_checkpoints(p, 128)                 # 8 checkpoints, room for 5
    out, S, ck = _run(p, 128, 5)
    assert kb.kda_get_device_error() == 5
    assert b"checkpoints" in kb.load().kda_last_error_message()
    check_state(ck.cpu().numpy(), ref[:5], "kept checkpoints")
    ref_o, ref_S = oracle_prefill(p)
    check_out(out.float().cpu().numpy(), ref_o)
    check_state(S.cpu().numpy(), ref_S)
