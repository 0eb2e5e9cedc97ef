"""The bounded waits every kernel makes on its own asynchronous work: a wait
that runs out reports a timeout through the device error word, and the
context stays usable.  The wait runs on an mbarrier nothing arrives on, with a
short poll limit, so nothing faults or hangs."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_48_gb300 import binding as kb
from gated_delta_rule_48_gb300 import inputs as kin
from kda_testlib import check_out, check_state

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_stays_usable():
    assert kb.kda_get_device_error() == 0
    kb.kda_selftest_bounded_wait(200)
    assert kb.kda_get_device_error() == 5  # KDA_ERR_DEVICE_INPUT
    assert b"timed out" in kb.load().kda_last_error_message()
    assert kb.kda_get_device_error() == 0  # the word was cleared
    # a normal prefill afterwards is exact
    p = kin.make_prefill([200, 77], 2, 128, seed=91, s0_std=0.05)
    cu = torch.from_numpy(p.cu_seqlens.astype(np.int32)).cuda()
    out, S = kb.kda_chunk_fwd(p.q.cuda(), p.k.cuda(), p.v.cuda(), p.log_alpha.cuda(),
                              p.beta.cuda(), p.S0.cuda(), cu)
    assert kb.kda_get_device_error() == 0
    ref_o, ref_S = oracle.forward(kin.bf16_bits(p.q), kin.bf16_bits(p.k), kin.bf16_bits(p.v),
                                  p.log_alpha.numpy(), p.beta.numpy(), p.S0.numpy(),
                                  p.cu_seqlens)
    check_out(out.float().cpu().numpy(), ref_o)
    check_state(S.cpu().numpy(), ref_S)
