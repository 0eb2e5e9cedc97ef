"""Input preparation of the fused entry points -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` may import this
module; it shares no code with the CUDA library.

``kda_chunk_fwd_fused`` / ``kda_decode_step_fused`` take raw projections and
prepare them on load.  The pages bound the forget gate's log-decay below at
-5 by changing the decay curve itself (lecture "Inside Kimi K3: Architecture
of an Open Frontier Model", sequence paragraph; orkas.ai close read, section
"A lower bound that deleted a GPU code path").  The reading taken, in this
order:

1. log alpha = -5 * sigmoid(gate) = -5 / (1 + e^-gate) per key channel; the
   recurrence then clamps to [-5, 0] as for a given log alpha.
2. q and k are scaled to unit L2 norm over their dk channels for each
   (token, head): x / max(||x||_2, 1e-12).
3. The normalised q and k are rounded to bfloat16 (nearest, ties to even):
   the values a caller would hand to the unfused entry points.

Everything here is float64 and written out step by step.
"""
from __future__ import annotations

import numpy as np

from . import decode_steps, forward

NORM_EPS = 1e-12


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact float64 values of bfloat16 bit patterns (uint16)."""
    u32 = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value (ties to even), as float64.

    A bfloat16 keeps 8 significant bits: with x = m * 2^e and 0.5 <= |m| < 1,
    the result is rint(m * 2^8) * 2^(e - 8); ``np.rint`` rounds halves to even.
    (Normal range only: the inputs here are at most 1 in magnitude and far
    above 2^-126.)
    """
    m, e = np.frexp(np.asarray(x, dtype=np.float64))
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def gate_log_alpha(gate: np.ndarray) -> np.ndarray:
    """Step 1: the bounded decay curve, log alpha = -5 / (1 + exp(-gate))."""
    g = np.asarray(gate, dtype=np.float64)
    return -5.0 / (1.0 + np.exp(-g))


def l2_normalise(x: np.ndarray) -> np.ndarray:
    """Step 2: each vector along the last axis divided by max(its L2 norm, 1e-12)."""
    x = np.asarray(x, dtype=np.float64)
    norm = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / np.maximum(norm, NORM_EPS)


def prepare(q_raw_bits, k_raw_bits, gate_bits):
    """Steps 1-3 on bfloat16 bit arrays; returns float64 (q, k, log_alpha)."""
    q = round_bf16(l2_normalise(bf16_bits_to_f64(q_raw_bits)))
    k = round_bf16(l2_normalise(bf16_bits_to_f64(k_raw_bits)))
    la = gate_log_alpha(bf16_bits_to_f64(gate_bits))
    return q, k, la


def forward_fused(q_raw_bits, k_raw_bits, v_bits, gate_bits, beta, S0=None, cu_seqlens=None,
                  *, heads=None, threads=None):
    """The fused prefill: prepare, then the fp64 recurrence of :func:`oracle.forward`."""
    q, k, la = prepare(q_raw_bits, k_raw_bits, gate_bits)
    v = bf16_bits_to_f64(v_bits)
    S0 = None if S0 is None else np.asarray(S0, dtype=np.float64)
    return forward(q, k, v, la, np.asarray(beta, dtype=np.float64), S0, cu_seqlens,
                   heads=heads, threads=threads)


def decode_steps_fused(q_raw_bits, k_raw_bits, v_bits, gate_bits, beta, S, *, threads=None):
    """The fused decode steps ([steps, N, H, d] inputs): prepare, then :func:`oracle.decode_steps`."""
    q, k, la = prepare(q_raw_bits, k_raw_bits, gate_bits)
    return decode_steps(q, k, bf16_bits_to_f64(v_bits), la, np.asarray(beta, dtype=np.float64),
                        np.asarray(S, dtype=np.float64), threads=threads)
