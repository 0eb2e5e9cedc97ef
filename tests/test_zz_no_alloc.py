"""kda_chunk_fwd_noalloc: the prefill entry point that allocates nothing.

It is meant for callers that cannot allocate device memory during a call:
their runtime hands all device memory to its own allocator up front, or they
must not touch a memory pool mid-step.  Its working data lives in a fixed
array inside the library, shared by every call.  These tests call it through
the C ABI and check its results against the fp64 oracle on two calls in a
row with different shapes (a packed batch, then a uniform batch with
cu_seqlens = NULL, which takes the planner's uniform path), so a second call
that saw the first call's leftovers would fail.  A fresh process checks that
when it is the first call on a device it creates no memory pool.  This file
sorts last so a stop-at-first-failure run has already run every other test.
"""
import ctypes
import os
import subprocess
import sys
import textwrap

import pytest
import torch

from gated_delta_rule_48_gb300 import binding as kb
from gated_delta_rule_48_gb300 import inputs as kin
from kda_testlib import check_out, check_state, oracle_prefill, to_device

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
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


CASES = [
    # packed batch: empty sequences, a single token, ragged tails, weak decay
    dict(lens=[700, 1, 0, 129, 64], H=3, d=128, seed=51, s0_std=0.05, log_alpha_fixed=-0.02),
    # uniform batch, cu_seqlens = NULL: the planner's uniform path
    dict(lens=[300, 300, 300], H=2, d=64, seed=52, s0_std=0.05),
]


def _case(c):
    p = kin.make_prefill(c["lens"], c["H"], c["d"], seed=c["seed"], s0_std=c["s0_std"],
                         log_alpha_fixed=c.get("log_alpha_fixed"))
    assert p.uniform == (len(set(c["lens"])) == 1)
    return p


@pytest.mark.gpu
def test_noalloc_matches_the_oracle_on_two_calls_in_a_row():
    for c in CASES:
        p = _case(c)
        d = to_device(p)
        out = torch.full((p.total_T, p.H, p.dv), float("nan"), dtype=torch.bfloat16,
                         device="cuda")
        S = torch.full((p.n_seqs, p.H, p.dk, p.dv), float("nan"), dtype=torch.float32,
                       device="cuda")
        _noalloc(d, p, out, S)
        assert kb.kda_get_device_error() == 0
        ref_o, ref_S = oracle_prefill(p)
        check_out(out.float().cpu().numpy(), ref_o, "noalloc out")
        check_state(S.cpu().numpy(), ref_S, "noalloc S_final")


@pytest.mark.gpu
def test_noalloc_as_first_call_creates_no_pool():
    """In a fresh process the no-allocation entry point is the first library
    call on the device; afterwards the library has still created no pool.
    A packed kda_chunk_fwd call, which takes a workspace, then creates it."""
    script = textwrap.dedent(f"""
        import sys
        sys.path.insert(0, {ROOT!r}); sys.path.insert(0, {os.path.join(ROOT, 'tests')!r})
        import torch
        from gated_delta_rule_48_gb300 import binding as kb
        import test_zz_no_alloc as t
        from kda_testlib import to_device
        torch.cuda.set_device(0)
        p = t._case(t.CASES[0]); d = to_device(p)
        out = torch.empty((p.total_T, p.H, p.dv), dtype=torch.bfloat16, device="cuda")
        S = torch.empty((p.n_seqs, p.H, p.dk, p.dv), dtype=torch.float32, device="cuda")
        t._noalloc(d, p, out, S)
        assert kb.kda_get_device_error() == 0
        assert kb.kda_workspace_pool_bytes() == -1, "the no-allocation call created a pool"
        kb.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"],
                         d["cu_seqlens"], n_seqs=p.n_seqs)
        torch.cuda.synchronize()
        assert kb.kda_workspace_pool_bytes() >= 0, "kda_chunk_fwd on a packed batch made no pool"
        print("fresh-process check ok")
    """)
    res = subprocess.run([sys.executable, "-c", script], cwd=ROOT, capture_output=True,
                         text=True, timeout=600)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-3000:]
    assert "fresh-process check ok" in res.stdout


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
