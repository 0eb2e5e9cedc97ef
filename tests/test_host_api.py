"""kda_chunk_fwd_host: a uniform batch in host memory, sliced in time and
pipelined through the GPU, against the fp64 oracle and against the
device-resident call."""
import numpy as np
import pytest
import torch

from gated_delta_rule_48_gb300 import binding as kb
from gated_delta_rule_48_gb300 import inputs as kin
from kda_testlib import check_out, check_state, oracle_prefill, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,slice_tokens", [(128, 0), (128, 192), (64, 128)])
def test_host_pipeline_matches_oracle_and_device_call(d, slice_tokens):
    p = kin.make_prefill([1000] * 3, 4, d, seed=71, s0_std=0.05)   # 1000 = 5 x 192 + 40: a ragged last slice
    pin = lambda t: t.contiguous().pin_memory()
    out = torch.empty((p.total_T, p.H, p.dv), dtype=torch.bfloat16).pin_memory()
    S = torch.empty((p.n_seqs, p.H, p.dk, p.dv), dtype=torch.float32).pin_memory()
    kb.kda_chunk_fwd_host(pin(p.q), pin(p.k), pin(p.v), pin(p.log_alpha), pin(p.beta), pin(p.S0),
                          out, S, n_seqs=p.n_seqs, slice_tokens=slice_tokens)
    torch.cuda.synchronize()
    assert kb.kda_get_device_error() == 0
    ref_o, ref_S = oracle_prefill(p)
    check_out(out.float().numpy(), ref_o)
    check_state(S.numpy(), ref_S)
    dd = to_device(p)
    o2, S2 = kb.kda_chunk_fwd(dd["q"], dd["k"], dd["v"], dd["log_alpha"], dd["beta"], dd["S0"],
                              None, n_seqs=p.n_seqs)
    # slicing only moves the chunk boundaries' rounding: the two agree closely
    assert np.abs(out.float().numpy() - o2.float().cpu().numpy()).max() < 2e-2
    np.testing.assert_allclose(S.numpy(), S2.cpu().numpy(), rtol=0, atol=2e-3)


def test_host_pipeline_zero_state_and_no_state_out():
    p = kin.make_prefill([256] * 2, 2, 64, seed=72)
    out = torch.empty((p.total_T, p.H, p.dv), dtype=torch.bfloat16).pin_memory()
    kb.kda_chunk_fwd_host(p.q, p.k, p.v, p.log_alpha, p.beta, None, out, None, n_seqs=2)
    torch.cuda.synchronize()
    ref_o, _ = oracle_prefill(p)
    check_out(out.float().numpy(), ref_o)
