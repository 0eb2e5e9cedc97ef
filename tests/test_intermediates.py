"""Intermediate parity: the prefill's per-chunk steps against the fp64 chunked
evaluator (oracle/naive_chunked.py), one step at a time.

kda_debug_chunk_dump runs the prefill and also writes, for one chunk of one
(sequence, head): the cumulative log-decay g, the intra-chunk matrices A_kk
and A_qk, the UT transform T, U = T (V - k e^g S) and the state S entering
the chunk.  Each is compared with the evaluator's value for the same chunk,
fed the state the GPU dumped, so a wrong step shows at that step instead of
only in the final output.  The state itself is compared with the oracle's
state after the same prefix of tokens.

Tolerances follow the kernel's rounding plan, with margin over what GB300
gives: g is an fp32 cumulative sum (1e-5 relative); A_kk and A_qk come from
bf16 operands (1e-2 of the matrix scale, measured 2-3e-3); T is fp32 from
them, read as tf32 (5e-3, measured 4e-4); U = T (V - k e^g S) (relative L2
5e-3, measured 6e-4); the state is held to the state tolerance.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from oracle import naive_chunked
from gated_delta_rule_48_gb300 import binding as kb
from gated_delta_rule_48_gb300 import inputs as kin
from kda_testlib import check_out, check_state, oracle_prefill, rel_l2, to_device


def _close(x, ref, rel, what):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = max(np.max(np.abs(ref)), 1e-30)
    err = np.max(np.abs(x - ref)) / scale
    assert err <= rel, f"{what}: max|err| / max|ref| = {err:.3e} > {rel:.1e}"
    return err


CASES = [
    # (lengths, d, which (seq, head, chunk)): a chunk deep in a long sequence,
    # a ragged last chunk (44 of 64 tokens), the first chunk
    ([300, 200], 128, (1, 1, 2)),
    ([300, 200], 128, (0, 0, 4)),
    ([130, 64], 64, (0, 1, 0)),
]


@pytest.mark.gpu
@pytest.mark.parametrize("lens,d,which", CASES, ids=["deep", "ragged", "first_d64"])
def test_chunk_intermediates_match_the_chunked_evaluator(lens, d, which):
    seq, head, chunk = which
    p = kin.make_prefill(lens, 2, d, seed=71 + d, s0_std=0.05, log_alpha_fixed=-0.02)
    dd = to_device(p)
    out, S_fin, parts = kb.kda_debug_chunk_dump(dd["q"], dd["k"], dd["v"], dd["log_alpha"],
                                                dd["beta"], dd["S0"], dd["cu_seqlens"],
                                                n_seqs=p.n_seqs, seq=seq, head=head,
                                                chunk=chunk)
    assert kb.kda_get_device_error() == 0
    # the call is a full prefill as well
    ref_o, ref_S = oracle_prefill(p)
    check_out(out.float().cpu().numpy(), ref_o)
    check_state(S_fin.cpu().numpy(), ref_S)

    t0 = int(p.cu_seqlens[seq]) + 64 * chunk
    t1 = min(t0 + 64, int(p.cu_seqlens[seq + 1]))
    n = t1 - t0
    f64 = lambda t: t[t0:t1, head].double().numpy()
    q, k, v = f64(p.q), f64(p.k), f64(p.v)
    la, b = f64(p.log_alpha), p.beta[t0:t1, head].double().numpy()
    got = {key: val.cpu().numpy().astype(np.float64) for key, val in parts.items()}
    S_in = got["S"][:d, :d]

    # the state entering the chunk: the oracle's state after the same prefix
    cu = np.array([0, t0 - int(p.cu_seqlens[seq])])
    pre = slice(int(p.cu_seqlens[seq]), t0)
    S0 = None if p.S0 is None else p.S0[seq:seq + 1].numpy()
    if t0 > int(p.cu_seqlens[seq]):
        _, S_ref = oracle.forward(kin.bf16_bits(p.q[pre]), kin.bf16_bits(p.k[pre]),
                                  kin.bf16_bits(p.v[pre]), p.log_alpha[pre].numpy(),
                                  p.beta[pre].numpy(), S0, cu)
        S_ref = S_ref[0, head]
    else:
        S_ref = S0[0, head]
    assert rel_l2(S_in, S_ref) <= 1e-3

    # each step against the chunked evaluator from the dumped state
    _, _, mid = naive_chunked.chunk_step(q, k, v, la, b, S_in)
    # measured on GB300: g 2e-7, A 2-3e-3, T 3-4e-4, U 4-6e-4 (relative L2)
    assert np.max(np.abs(got["g"][:n, :d] - mid["g"])) <= 1e-5 * max(1.0, np.max(np.abs(mid["g"])))
    _close(got["A_kk"][:n, :n], mid["A_kk"], 1e-2, "A_kk")
    _close(got["A_qk"][:n, :n], mid["A_qk"], 1e-2, "A_qk")
    _close(got["T"][:n, :n], mid["T"], 5e-3, "T")
    assert rel_l2(got["U"][:n, :d], mid["U"]) <= 5e-3, rel_l2(got["U"][:n, :d], mid["U"])
    # rows past the sequence's end act as the identity: nothing in A or T
    if n < 64:
        assert np.all(got["A_kk"][n:, :] == 0) and np.all(got["T"][:, n:] == 0)


def test_dump_arguments_are_checked_on_the_host():
    lib = kb.load()
    P = lambda i: ctypes.c_void_p((1 << 40) + i * (1 << 32))
    args = [P(i) for i in range(9)]
    args[6] = None
    base = args + [256, 2, 2, 64, 64]
    assert lib.kda_debug_chunk_dump(*base, 0, 0, 0, None, None) == 1           # no dump buffer
    assert lib.kda_debug_chunk_dump(*base, 2, 0, 0, P(20), None) == 1          # seq out of range
    assert lib.kda_debug_chunk_dump(*base, 0, 2, 0, P(20), None) == 1          # head out of range
    assert lib.kda_debug_chunk_dump(*base, 0, 0, 0, P(0), None) == 1           # over q
    assert b"dump" in lib.kda_last_error_message()
