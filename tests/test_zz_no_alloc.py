"""kda_chunk_fwd_noalloc: the prefill entry point that allocates nothing.

It is meant for callers that cannot allocate device memory during a call
(their runtime hands all device memory to its own allocator up front, or they
must not touch a memory pool mid-step).  Its working data lives in a fixed
array inside the library, shared by every call.  These tests call it through
the C ABI and check it against kda_chunk_fwd on the same inputs, for two
calls in a row with different shapes, so a second call that saw the first
call's leftovers would fail.  This file sorts last so a stop-at-first-failure
run has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from gated_delta_rule_48_gb300 import binding as kb
from gated_delta_rule_48_gb300 import inputs as kin
from kda_testlib import check_out, check_state, to_device

MAX_SEQS = 8184  # the entry point's documented limit


def _noalloc(d, p, out, S_final):
    lib = kb.load()
    st = lib.kda_chunk_fwd_noalloc(
        ctypes.c_void_p(d["q"].data_ptr()), ctypes.c_void_p(d["k"].data_ptr()),
        ctypes.c_void_p(d["v"].data_ptr()), ctypes.c_void_p(d["log_alpha"].data_ptr()),
        ctypes.c_void_p(d["beta"].data_ptr()),
        None if d["S0"] is None else ctypes.c_void_p(d["S0"].data_ptr()),
        None if d["cu_seqlens"] is None else ctypes.c_void_p(d["cu_seqlens"].data_ptr()),
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(S_final.data_ptr()),
        p.total_T, p.n_seqs, p.H, p.dk, p.dv,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.kda_last_error_message()


@pytest.mark.gpu
def test_noalloc_matches_kda_chunk_fwd_on_two_calls_in_a_row():
    cases = [
        kin.make_prefill([700, 1, 0, 129, 64], 3, 128, seed=51, s0_std=0.05,
                         log_alpha_fixed=-0.02),
        kin.make_prefill([300, 77], 2, 64, seed=52, s0_std=0.05),
    ]
    for p in cases:
        d = to_device(p)
        ref_out, ref_S = kb.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                          d["S0"], d["cu_seqlens"], n_seqs=p.n_seqs)
        out = torch.full_like(ref_out, float("nan"))
        S = torch.full_like(ref_S, float("nan"))
        _noalloc(d, p, out, S)
        assert kb.kda_get_device_error() == 0
        check_out(out.float().cpu().numpy(), ref_out.float().cpu().numpy(), "noalloc out")
        check_state(S.cpu().numpy(), ref_S.cpu().numpy(), "noalloc S_final")


def test_noalloc_rejects_more_sequences_than_its_scratch_holds():
    """Checked on the host before any GPU work, so this needs no GPU."""
    lib = kb.load()
    base = 1 << 40
    ptr = lambda i: ctypes.c_void_p(base + i * (1 << 34))
    n = MAX_SEQS + 1
    st = lib.kda_chunk_fwd_noalloc(ptr(0), ptr(1), ptr(2), ptr(3), ptr(4), None, None,
                                   ptr(7), ptr(8), n, n, 1, 64, 64, None)
    assert st == 2  # KDA_ERR_UNSUPPORTED
    assert b"no-allocation scratch limit" in lib.kda_last_error_message()
