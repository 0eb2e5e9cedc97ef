"""Shared helpers of the test suite: moving seeded inputs to the GPU, running
the oracle on the same values, and the parity metrics with their tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from gated_delta_rule_48_gb300 import inputs as kin

# GPU-vs-oracle tolerances on the same seeded inputs.
OUT_MAX_ABS = 2e-2     # max |out - oracle|
OUT_REL_L2 = 5e-3      # ||out - oracle|| / ||oracle||
STATE_REL_L2 = 1e-3    # ||S_final - oracle|| / ||oracle||


def rel_l2(x, ref):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(x - ref)
    if den == 0.0:
        return float(num)
    return float(num / den)


def max_abs(x, ref):
    if np.asarray(ref).size == 0:
        return 0.0
    return float(np.max(np.abs(np.asarray(x, np.float64) - np.asarray(ref, np.float64))))


def check_out(out, ref, what="out"):
    ma, rl = max_abs(out, ref), rel_l2(out, ref)
    assert ma <= OUT_MAX_ABS and rl <= OUT_REL_L2, f"{what}: max|err|={ma:.3e} relL2={rl:.3e}"
    return ma, rl


def check_state(S, ref, what="S_final"):
    rl = rel_l2(S, ref)
    assert rl <= STATE_REL_L2, f"{what}: relL2={rl:.3e}"
    return rl


def to_device(p: kin.PrefillInputs, device="cuda"):
    d = dict(q=p.q.to(device), k=p.k.to(device), v=p.v.to(device),
             log_alpha=p.log_alpha.to(device), beta=p.beta.to(device),
             S0=None if p.S0 is None else p.S0.to(device))
    d["cu_seqlens"] = (None if p.uniform else
                       torch.from_numpy(p.cu_seqlens.astype(np.int32)).to(device))
    return d


def oracle_prefill(p: kin.PrefillInputs, heads=None, threads=None):
    """Oracle on exactly the values the GPU receives (bf16 q/k/v, f32 gates)."""
    return oracle.forward(kin.bf16_bits(p.q), kin.bf16_bits(p.k), kin.bf16_bits(p.v),
                          p.log_alpha.numpy(), p.beta.numpy(),
                          None if p.S0 is None else p.S0.numpy(), p.cu_seqlens,
                          heads=heads, threads=threads)
