"""kda_decode_tokens: K tokens per sequence per call with a commit count
(speculative decoding's verify / commit), against the fp64 oracle, against
K single decode steps, and across calls of different K."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_48_gb300 import binding as kb
from gated_delta_rule_48_gb300 import inputs as kin
from kda_testlib import check_out, check_state

pytestmark = pytest.mark.gpu


def _seq_major(d):
    """make_decode's [steps, N, ...] tensors as [N, steps, ...] (sequence n's tokens together)."""
    f = lambda t: t.transpose(0, 1).contiguous()
    return f(d.q), f(d.k), f(d.v), f(d.log_alpha), f(d.beta)


def _oracle(q, k, v, la, b, S, commit):
    """Outputs of all K tokens from S, and each sequence's state after its first commit[n]."""
    N, K = q.shape[:2]
    flat = lambda t: t.reshape((N * K,) + tuple(t.shape[2:]))
    bits = lambda t: kin.bf16_bits(flat(t))
    cu = np.arange(N + 1) * K
    out, _ = oracle.forward(bits(q), bits(k), bits(v), flat(la).numpy(), flat(b).numpy(),
                            S.numpy(), cu)
    # committed prefixes: a packed batch of the first commit[n] tokens of each sequence
    keep = np.concatenate([np.arange(n * K, n * K + c) for n, c in enumerate(commit)]).astype(int)
    cu_c = np.concatenate([[0], np.cumsum(commit)])
    _, S_c = oracle.forward(bits(q)[keep], bits(k)[keep], bits(v)[keep], flat(la).numpy()[keep],
                            flat(b).numpy()[keep], S.numpy(), cu_c)
    return out.reshape((N, K) + out.shape[1:]), S_c


@pytest.mark.parametrize("d", [64, 128])
def test_decode_tokens_commit_all_and_partial(d):
    dec = kin.make_decode(48, 4, d, steps=8, seed=41)
    q, k, v, la, b = _seq_major(dec)
    rng = np.random.default_rng(41)
    for commit in (np.full(48, 8), rng.integers(0, 9, size=48)):
        S = dec.S.cuda()
        out = kb.kda_decode_tokens(q.cuda(), k.cuda(), v.cuda(), la.cuda(), b.cuda(), S,
                                   torch.from_numpy(commit.astype(np.int32)).cuda())
        assert kb.kda_get_device_error() == 0
        ref_o, ref_S = _oracle(q, k, v, la, b, dec.S, commit)
        check_out(out.float().cpu().numpy(), ref_o)
        check_state(S.cpu().numpy(), ref_S)
        # commit 0 leaves the state bit-identical
        zero = commit == 0
        np.testing.assert_array_equal(S.cpu().numpy()[zero], dec.S.numpy()[zero])


@pytest.mark.parametrize("d", [64, 128])
def test_decode_tokens_several_batches(d):
    """K = 19 tokens: three batches of the kernel's 8, with commits before,
    at and after the batch boundaries (the state is carried across them)."""
    K = 19
    dec = kin.make_decode(24, 3, d, steps=K, seed=45)
    q, k, v, la, b = _seq_major(dec)
    commit = np.array([19, 0, 8, 9, 16, 17, 1, 12] * 3, dtype=np.int32)
    S = dec.S.cuda()
    out = kb.kda_decode_tokens(q.cuda(), k.cuda(), v.cuda(), la.cuda(), b.cuda(), S,
                               torch.from_numpy(commit).cuda())
    assert kb.kda_get_device_error() == 0
    ref_o, ref_S = _oracle(q, k, v, la, b, dec.S, commit)
    check_out(out.float().cpu().numpy(), ref_o)
    check_state(S.cpu().numpy(), ref_S)


def test_decode_tokens_two_tokens_strong_and_weak_decay():
    """K = 2 (the smallest multi-token call) with log alpha at the clamp (-5)
    on half the channels and 0 (no decay) on the rest."""
    dec = kin.make_decode(40, 2, 128, steps=2, seed=46)
    la = dec.log_alpha.clone()
    la[..., :64] = -5.0
    la[..., 64:] = 0.0
    dec.log_alpha = la
    q, k, v, la, b = _seq_major(dec)
    S = dec.S.cuda()
    out = kb.kda_decode_tokens(q.cuda(), k.cuda(), v.cuda(), la.cuda(), b.cuda(), S)
    ref_o, ref_S = _oracle(q, k, v, la, b, dec.S, np.full(40, 2))
    check_out(out.float().cpu().numpy(), ref_o)
    check_state(S.cpu().numpy(), ref_S)


def test_decode_tokens_verify_then_commit_is_exact():
    """Verify (commit 0), then commit the accepted prefix: the verify call
    writes no state, the outputs do not depend on the commit counts, and a
    sequence that accepts c tokens ends bit-identical to a call over only its
    first c tokens (the per-token arithmetic does not depend on K)."""
    dec = kin.make_decode(32, 4, 128, steps=6, seed=42)
    q, k, v, la, b = (t.cuda() for t in _seq_major(dec))
    accept = np.array([6, 0, 3, 2] * 8, dtype=np.int32)
    S = dec.S.cuda()
    out_v = kb.kda_decode_tokens(q, k, v, la, b, S, torch.zeros(32, dtype=torch.int32, device="cuda"))
    assert torch.equal(S, dec.S.cuda())                       # verify wrote no state
    out_c = kb.kda_decode_tokens(q, k, v, la, b, S, torch.from_numpy(accept).cuda())
    assert torch.equal(out_v, out_c)                          # outputs do not depend on commit
    for c in (6, 3, 2):
        Sc = dec.S.cuda()
        o = kb.kda_decode_tokens(q[:, :c].contiguous(), k[:, :c].contiguous(),
                                 v[:, :c].contiguous(), la[:, :c].contiguous(),
                                 b[:, :c].contiguous(), Sc)
        assert torch.equal(o, out_c[:, :c])
        sel = torch.from_numpy(accept == c).cuda()
        assert torch.equal(S[sel], Sc[sel])
    assert torch.equal(S[torch.from_numpy(accept == 0).cuda()],
                       dec.S.cuda()[torch.from_numpy(accept == 0).cuda()])


def test_decode_tokens_matches_single_steps():
    """K tokens in one call against K calls of the single step (a separate
    kernel): same outputs and state up to rounding."""
    dec = kin.make_decode(64, 8, 128, steps=5, seed=44)
    q, k, v, la, b = (t.cuda() for t in _seq_major(dec))
    S = dec.S.cuda()
    out = kb.kda_decode_tokens(q, k, v, la, b, S)
    S1 = dec.S.cuda()
    outs = [kb.kda_decode_step(q[:, t].contiguous(), k[:, t].contiguous(), v[:, t].contiguous(),
                               la[:, t].contiguous(), b[:, t].contiguous(), S1) for t in range(5)]
    check_out(out.float().cpu().numpy(), torch.stack(outs, 1).float().cpu().numpy())
    check_state(S.cpu().numpy(), S1.cpu().numpy())


def test_decode_tokens_rejects_commit_out_of_range():
    dec = kin.make_decode(4, 2, 64, steps=3, seed=43)
    q, k, v, la, b = (t.cuda() for t in _seq_major(dec))
    S = dec.S.cuda()
    out = torch.full((4, 3, 2, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    commit = torch.tensor([3, 4, 0, -1], dtype=torch.int32, device="cuda")
    kb.kda_decode_tokens(q, k, v, la, b, S, commit, out=out)
    assert kb.kda_get_device_error() == 5  # KDA_ERR_DEVICE_INPUT
    assert b"commit" in kb.load().kda_last_error_message()
    # the rejected sequences (1 and 3) are untouched, the others ran
    assert torch.equal(S[1], dec.S[1].cuda()) and torch.equal(S[3], dec.S[3].cuda())
    assert torch.isnan(out[1].float()).all() and torch.isnan(out[3].float()).all()
    assert not torch.isnan(out[0].float()).any() and not torch.isnan(out[2].float()).any()
    assert not torch.equal(S[0], dec.S[0].cuda())
