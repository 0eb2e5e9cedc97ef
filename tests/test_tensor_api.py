"""The descriptor form of the two layer calls (kda_chunk_fwd_t,
kda_decode_step_t): the library itself rejects a wrong dtype, a shape that
does not match q's, and a layout that is not dense row-major, before anything
is launched.  Those checks run on the host, so the rejection cases need no GPU
(the descriptors point at host tensors that are never read).  The GPU case
checks the descriptor call against the pointer call and the oracle."""
import numpy as np
import pytest
import torch

from gated_delta_rule_48_gb300 import binding as kb
from gated_delta_rule_48_gb300 import inputs as kin
from kda_testlib import check_out, check_state, oracle_prefill, to_device

INVALID = 1


def prefill_tensors(T=128, N=2, H=2, d=64, batched=False):
    if batched:
        lead = (N, T // N)
    else:
        lead = (T,)
    return dict(
        q=torch.zeros(*lead, H, d, dtype=torch.bfloat16),
        k=torch.zeros(*lead, H, d, dtype=torch.bfloat16),
        v=torch.zeros(*lead, H, d, dtype=torch.bfloat16),
        log_alpha=torch.zeros(*lead, H, d, dtype=torch.float32),
        beta=torch.zeros(*lead, H, dtype=torch.float32),
        S0=torch.zeros(N, H, d, d, dtype=torch.float32),
        cu_seqlens=None if batched else torch.tensor([0, T // 2, T], dtype=torch.int32),
        out=torch.zeros(*lead, H, d, dtype=torch.bfloat16),
        S_final=torch.zeros(N, H, d, d, dtype=torch.float32),
    )


def call_prefill(t):
    lib = kb.load()
    names = ["q", "k", "v", "log_alpha", "beta", "S0", "cu_seqlens", "out", "S_final"]
    descs = [kb.describe(t[n]) for n in names]
    st = lib.kda_chunk_fwd_t(*[kb._dref(d) for d in descs], None)
    return st, lib.kda_last_error_message().decode()


@pytest.mark.parametrize("name,dtype", [
    ("q", torch.float32), ("k", torch.float16), ("v", torch.float32),
    ("log_alpha", torch.bfloat16), ("beta", torch.bfloat16), ("S0", torch.bfloat16),
    ("cu_seqlens", torch.int64), ("out", torch.float32), ("S_final", torch.bfloat16)])
def test_wrong_dtype_is_rejected(name, dtype):
    t = prefill_tensors()
    t[name] = t[name].to(dtype)
    st, msg = call_prefill(t)
    assert st == INVALID and msg.startswith(name + ": dtype"), msg


@pytest.mark.parametrize("name", ["q", "k", "v", "log_alpha", "out", "S0", "S_final"])
def test_non_dense_layout_is_rejected(name):
    t = prefill_tensors()
    x = t[name]
    # the same extents, with the last two dimensions stored transposed
    t[name] = x.transpose(-1, -2).contiguous().transpose(-1, -2)
    assert t[name].shape == x.shape and not t[name].is_contiguous()
    st, msg = call_prefill(t)
    assert st == INVALID and msg.startswith(name + ": not dense"), msg


def test_strided_slice_is_rejected():
    t = prefill_tensors()
    big = torch.zeros(256, 2, 64, dtype=torch.bfloat16)
    t["q"] = big[::2]  # every other token: extents right, token stride doubled
    st, msg = call_prefill(t)
    assert st == INVALID and "q: not dense" in msg


@pytest.mark.parametrize("name,shape", [
    ("k", (128, 3, 64)), ("v", (127, 2, 64)), ("log_alpha", (128, 2, 32)),
    ("beta", (128, 2, 1)), ("S0", (2, 2, 64, 32)), ("cu_seqlens", (4,)),
    ("out", (128, 2, 32)), ("S_final", (3, 2, 64, 64))])
def test_shape_mismatch_is_rejected(name, shape):
    t = prefill_tensors()
    t[name] = torch.zeros(shape, dtype=t[name].dtype)
    st, msg = call_prefill(t)
    # a state whose sequence count disagrees with cu_seqlens may be reported
    # under either name
    names = (name, "cu_seqlens") if name in ("S0", "S_final") else (name,)
    assert st == INVALID and msg.split(":")[0] in names, msg


def test_batched_layout_takes_no_cu_seqlens():
    t = prefill_tensors(batched=True)
    t["cu_seqlens"] = torch.tensor([0, 64, 128], dtype=torch.int32)
    st, msg = call_prefill(t)
    assert st == INVALID and msg.startswith("cu_seqlens:"), msg


def test_pointer_rules_still_apply_after_the_descriptor_checks():
    t = prefill_tensors()
    t["out"] = t["q"]  # well-formed descriptors, but out aliases q
    st, msg = call_prefill(t)
    assert st == INVALID and "out overlaps q" in msg, msg
    t = prefill_tensors(d=96)
    st, msg = call_prefill(t)
    assert st == 2 and "dk" in msg  # KDA_ERR_UNSUPPORTED from the pointer form's checks


def test_decode_descriptors_are_checked():
    lib = kb.load()
    N, H, d = 4, 2, 64
    t = dict(q=torch.zeros(N, H, d, dtype=torch.bfloat16),
             k=torch.zeros(N, H, d, dtype=torch.bfloat16),
             v=torch.zeros(N, H, d, dtype=torch.bfloat16),
             log_alpha=torch.zeros(N, H, d), beta=torch.zeros(N, H),
             S_inout=torch.zeros(N, H, d, d), out=torch.zeros(N, H, d, dtype=torch.bfloat16))
    names = ["q", "k", "v", "log_alpha", "beta", "S_inout", "out"]

    def call(**over):
        tt = dict(t, **over)
        descs = [kb.describe(tt[n]) for n in names]
        st = lib.kda_decode_step_t(*[kb._dref(x) for x in descs], None)
        return st, lib.kda_last_error_message().decode()

    st, msg = call(S_inout=t["S_inout"].to(torch.bfloat16))
    assert st == INVALID and msg.startswith("S_inout: dtype")
    st, msg = call(S_inout=t["S_inout"].transpose(-1, -2).contiguous().transpose(-1, -2))
    assert st == INVALID and msg.startswith("S_inout: not dense")
    st, msg = call(beta=torch.zeros(N, H, 1))
    assert st == INVALID and msg.startswith("beta:")
    st, msg = call(q=torch.zeros(N, H, d))
    assert st == INVALID and msg.startswith("q: dtype")


@pytest.mark.gpu
def test_descriptor_calls_equal_the_pointer_calls():
    p = kin.make_prefill([300, 77, 0, 129], 2, 128, seed=61, s0_std=0.05)
    d = to_device(p)
    ref_o, ref_S = kb.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"],
                                    d["cu_seqlens"])
    out = torch.empty_like(ref_o)
    S = torch.empty_like(ref_S)
    kb.kda_chunk_fwd_t(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"],
                       d["cu_seqlens"], out, S)
    assert kb.kda_get_device_error() == 0
    assert torch.equal(out, ref_o) and torch.equal(S, ref_S)
    o_or, S_or = oracle_prefill(p)
    check_out(out.float().cpu().numpy(), o_or)
    check_state(S.cpu().numpy(), S_or)
    # a uniform batch as [B, T_b, H, d]
    pb = kin.make_prefill([128] * 3, 2, 64, seed=62, s0_std=0.05)
    db = to_device(pb)
    view = lambda x: x.view(3, 128, *x.shape[1:])
    ob = torch.empty(3, 128, 2, 64, dtype=torch.bfloat16, device="cuda")
    Sb = torch.empty(3, 2, 64, 64, device="cuda")
    kb.kda_chunk_fwd_t(view(db["q"]), view(db["k"]), view(db["v"]), view(db["log_alpha"]),
                       view(db["beta"]), db["S0"], None, ob, Sb)
    o_or, S_or = oracle_prefill(pb)
    check_out(ob.reshape(384, 2, 64).float().cpu().numpy(), o_or)
    check_state(Sb.cpu().numpy(), S_or)
    # decode
    dec = kin.make_decode(8, 2, 128, steps=1, seed=63)
    Sa, Sb2 = dec.S.cuda(), dec.S.cuda()
    args = [x[0].cuda() for x in (dec.q, dec.k, dec.v, dec.log_alpha, dec.beta)]
    o1 = kb.kda_decode_step(*args, Sa)
    o2 = torch.empty_like(o1)
    kb.kda_decode_step_t(*args, Sb2, o2)
    assert torch.equal(o1, o2) and torch.equal(Sa, Sb2)
