"""The entry points are stream-ordered and allocate only stream-ordered, so a
CUDA graph can capture them, and calls on different streams can overlap.
Both are checked against eager calls on the same inputs."""
import numpy as np
import pytest
import torch

from gated_delta_rule_48_gb300 import binding as kb
from gated_delta_rule_48_gb300 import inputs as kin
from kda_testlib import to_device

pytestmark = pytest.mark.gpu


def _eager(d, n_seqs):
    return kb.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"],
                            d["cu_seqlens"], n_seqs=n_seqs)


def test_prefill_and_decode_captured_in_a_cuda_graph():
    # varlen with a long sequence: the planner, the split path (summary, scan,
    # replay) and the workspace allocation all go into the graph
    p = kin.make_prefill([3000, 100, 700], 2, 128, seed=81, s0_std=0.05)
    d = to_device(p)
    ref_out, ref_S = _eager(d, p.n_seqs)
    dec = kin.make_decode(16, 2, 128, steps=3, seed=82)
    S_dec = dec.S.cuda()
    q, k, v, la, b = (t.cuda() for t in (dec.q, dec.k, dec.v, dec.log_alpha, dec.beta))
    S_ref = S_dec.clone()
    ref_dec = [kb.kda_decode_step(q[s], k[s], v[s], la[s], b[s], S_ref) for s in range(3)]

    out = torch.empty_like(ref_out)
    S = torch.empty_like(ref_S)
    S_g = S_dec.clone()
    dec_out = torch.empty((3,) + tuple(ref_dec[0].shape), dtype=torch.bfloat16, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up on the capture stream (allocator pools)
        kb.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"],
                         d["cu_seqlens"], out, S, n_seqs=p.n_seqs, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st = torch.cuda.current_stream()
        kb.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"],
                         d["cu_seqlens"], out, S, n_seqs=p.n_seqs, stream=st)
        for s in range(3):
            kb.kda_decode_step(q[s], k[s], v[s], la[s], b[s], S_g, dec_out[s], stream=st)
    for rep in range(2):
        out.zero_()
        S.zero_()
        S_g.copy_(S_dec)
        g.replay()
        torch.cuda.synchronize()
        assert kb.kda_get_device_error() == 0
        assert torch.equal(out, ref_out) and torch.equal(S, ref_S)
        assert torch.equal(S_g, S_ref)
        for s in range(3):
            assert torch.equal(dec_out[s], ref_dec[s])


def test_concurrent_calls_on_two_streams():
    ps = [kin.make_prefill([1500] * 2, 4, 128, seed=83 + i, s0_std=0.05) for i in range(2)]
    ds = [to_device(p) for p in ps]
    refs = [_eager(d, p.n_seqs) for d, p in zip(ds, ps)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in ps]
    outs = []
    for d, p, s in zip(ds, ps, streams):
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            outs.append(kb.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                         d["S0"], d["cu_seqlens"], n_seqs=p.n_seqs, stream=s))
    torch.cuda.synchronize()
    for (o, S), (ro, rS) in zip(outs, refs):
        assert torch.equal(o, ro) and torch.equal(S, rS)


def test_decode_tokens_captured_in_a_cuda_graph():
    """The persistent multi-token decode (with commit counts) inside a graph:
    two replays from the same starting state equal the eager call bit for bit."""
    dec = kin.make_decode(40, 4, 128, steps=5, seed=84)
    f = lambda t: t.transpose(0, 1).contiguous().cuda()
    q, k, v, la, b = f(dec.q), f(dec.k), f(dec.v), f(dec.log_alpha), f(dec.beta)
    commit = torch.tensor([5, 0, 3, 1] * 10, dtype=torch.int32, device="cuda")
    S_ref = dec.S.cuda()
    ref_out = kb.kda_decode_tokens(q, k, v, la, b, S_ref, commit)
    S_g = dec.S.cuda()
    out = torch.empty_like(ref_out)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up on the capture stream
        kb.kda_decode_tokens(q, k, v, la, b, S_g.clone(), commit, out, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        kb.kda_decode_tokens(q, k, v, la, b, S_g, commit, out, stream=torch.cuda.current_stream())
    for rep in range(2):
        out.zero_()
        S_g.copy_(dec.S.cuda())
        g.replay()
        torch.cuda.synchronize()
        assert kb.kda_get_device_error() == 0
        assert torch.equal(out, ref_out) and torch.equal(S_g, S_ref)
