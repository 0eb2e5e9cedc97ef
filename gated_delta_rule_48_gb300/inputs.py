"""Seeded synthetic inputs for the KDA prefill and decode workloads.

This module only draws random numbers and lays them out; it holds none of the
layer's arithmetic, so both the CUDA path and the fp64 oracle consume exactly
the same values from it.

Recipe (shared by every workload):

* q, k, v ~ N(0, 1), drawn in float32.  q and k are L2-normalised per
  (token, head) over the key channels in float32, then q, k, v are rounded to
  bfloat16 (round to nearest even).  The stored q, k are therefore only
  approximately unit-norm.
* log_alpha = -5 * sigmoid(N(0, 1)) per (token, head, key channel), float32.
  This is the bounded gate curve: every value lies in (-5, 0).
* beta = sigmoid(N(0, 1)) per (token, head), float32.
* S0 ~ N(0, 0.02**2) (standard deviation 0.02) float32, or zero.

Draw order: q, k, v, log_alpha, beta, then the workload's specials, then S0;
each tensor is drawn in token blocks of ``_BLOCK`` tokens from one
``numpy.random.default_rng(seed)`` stream.

Packed layout (the library's): q, k, log_alpha [total_T, H, dk]; v [total_T,
H, dv]; beta [total_T, H]; S0 [N, H, dk, dv]; cu_seqlens int [N + 1].  A
uniform batch [B, T, H, d] is the same memory as [B*T, H, d].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

_BLOCK = 1 << 15  # tokens per generation block


@dataclass
class PrefillInputs:
    q: torch.Tensor          # bf16 [total_T, H, dk]
    k: torch.Tensor          # bf16 [total_T, H, dk]
    v: torch.Tensor          # bf16 [total_T, H, dv]
    log_alpha: torch.Tensor  # f32 [total_T, H, dk]
    beta: torch.Tensor       # f32 [total_T, H]
    S0: torch.Tensor | None  # f32 [N, H, dk, dv]
    cu_seqlens: np.ndarray   # int64 [N + 1]
    uniform: bool            # True when every sequence has the same length
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def total_T(self) -> int:
        return int(self.q.shape[0])

    @property
    def n_seqs(self) -> int:
        return int(self.cu_seqlens.shape[0] - 1)

    @property
    def H(self) -> int:
        return int(self.q.shape[1])

    @property
    def dk(self) -> int:
        return int(self.q.shape[2])

    @property
    def dv(self) -> int:
        return int(self.v.shape[2])


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The bfloat16 bit patterns of ``t`` as a numpy uint16 array (no copy of values)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _normal_blocks(rng, total_T, tail_shape):
    out = np.empty((total_T,) + tail_shape, dtype=np.float32)
    for t0 in range(0, total_T, _BLOCK):
        t1 = min(total_T, t0 + _BLOCK)
        out[t0:t1] = rng.standard_normal((t1 - t0,) + tail_shape, dtype=np.float32)
    return out


def _sigmoid(x):
    return (1.0 / (1.0 + np.exp(-x))).astype(np.float32)


def _to_bf16(x: np.ndarray, normalise: bool) -> torch.Tensor:
    out = torch.empty(x.shape, dtype=torch.bfloat16)
    for t0 in range(0, x.shape[0], _BLOCK):
        blk = x[t0:t0 + _BLOCK]
        if normalise:
            nrm = np.sqrt(np.sum(blk * blk, axis=-1, keepdims=True, dtype=np.float32))
            blk = blk / np.maximum(nrm, np.float32(1e-12))
        out[t0:t0 + _BLOCK] = torch.from_numpy(np.ascontiguousarray(blk, dtype=np.float32))
    return out


def make_prefill(seq_lens, H, dk, dv=None, *, seed=0, s0_std=0.0,
                 log_alpha_fixed=None, log_alpha_fixed_channels=None,
                 beta_mode="sigmoid", beta_value=None, name="") -> PrefillInputs:
    """General seeded prefill inputs.

    ``seq_lens``: list of sequence lengths (packed in order).
    ``log_alpha_fixed``: if given, log_alpha equals this constant on the
    channels ``log_alpha_fixed_channels`` (a slice; all channels if None).
    ``beta_mode``: "sigmoid" (the recipe), "mix" (one third each of 0, 1 and
    sigmoid(N(0,1)), chosen per token-head), or "const" (``beta_value``).
    """
    dv = dk if dv is None else dv
    seq_lens = [int(x) for x in seq_lens]
    total_T = sum(seq_lens)
    rng = np.random.default_rng(seed)
    qf = _normal_blocks(rng, total_T, (H, dk))
    kf = _normal_blocks(rng, total_T, (H, dk))
    vf = _normal_blocks(rng, total_T, (H, dv))
    q = _to_bf16(qf, True)
    del qf
    k = _to_bf16(kf, True)
    del kf
    v = _to_bf16(vf, False)
    del vf
    la = _normal_blocks(rng, total_T, (H, dk))
    for t0 in range(0, total_T, _BLOCK):
        la[t0:t0 + _BLOCK] = -5.0 * _sigmoid(la[t0:t0 + _BLOCK])
    b = _sigmoid(_normal_blocks(rng, total_T, (H,)))
    if log_alpha_fixed is not None:
        sl = log_alpha_fixed_channels if log_alpha_fixed_channels is not None else slice(None)
        la[:, :, sl] = np.float32(log_alpha_fixed)
    if beta_mode == "mix":
        pick = rng.integers(0, 3, size=(total_T, H))
        b = np.where(pick == 0, np.float32(0.0), np.where(pick == 1, np.float32(1.0), b))
        b = b.astype(np.float32)
    elif beta_mode == "const":
        b = np.full((total_T, H), np.float32(beta_value), dtype=np.float32)
    elif beta_mode != "sigmoid":
        raise ValueError(beta_mode)
    N = len(seq_lens)
    S0 = None
    if s0_std:
        S0 = torch.from_numpy(
            (rng.standard_normal((N, H, dk, dv), dtype=np.float32) * np.float32(s0_std)))
    cu = np.zeros(N + 1, dtype=np.int64)
    cu[1:] = np.cumsum(seq_lens)
    return PrefillInputs(q=q, k=k, v=v, log_alpha=torch.from_numpy(la),
                         beta=torch.from_numpy(np.ascontiguousarray(b)), S0=S0,
                         cu_seqlens=cu, uniform=len(set(seq_lens)) <= 1, name=name)


def million_token_lengths(seed=3, total=1 << 20, n=8, lo=4096, hi=524288):
    """Lengths of the packed million-token workload.

    n-1 lengths floor(exp(U(ln lo, ln hi))); the last takes the remainder.  If
    the remainder is below ``lo`` all n-1 are drawn again from the same stream.
    """
    rng = np.random.default_rng(seed)
    while True:
        lens = [int(math.floor(math.exp(rng.uniform(math.log(lo), math.log(hi)))))
                for _ in range(n - 1)]
        last = total - sum(lens)
        if last >= lo:
            return lens + [last]


# Named workloads.  Index = position in the project's workload list.
WORKLOADS = {
    0: "tiny prefill B1 H2 T256 d64 (oracle-check size)",
    1: "batched prefill B4 H32 T4096 d128",
    2: "stress-bound prefill B1 H16 T65536 d128 (half the channels at log_alpha=-5, beta mixed)",
    3: "million-token packed varlen prefill, 8 sequences, H8 d128",
    4: "batched decode 256 seqs H32 d128, 64 steps",
}


def workload(idx: int) -> PrefillInputs:
    """The prefill workloads 0..3 (decode is :func:`decode_workload`)."""
    if idx == 0:
        return make_prefill([256], 2, 64, seed=0, s0_std=0.0, name=WORKLOADS[0])
    if idx == 1:
        return make_prefill([4096] * 4, 32, 128, seed=1, s0_std=0.02, name=WORKLOADS[1])
    if idx == 2:
        return make_prefill([65536], 16, 128, seed=2, s0_std=0.0, log_alpha_fixed=-5.0,
                            log_alpha_fixed_channels=slice(0, 64), beta_mode="mix",
                            name=WORKLOADS[2])
    if idx == 3:
        return make_prefill(million_token_lengths(), 8, 128, seed=3, s0_std=0.02,
                            name=WORKLOADS[3])
    raise ValueError(f"no prefill workload {idx}")


@dataclass
class DecodeInputs:
    q: torch.Tensor          # bf16 [steps, N, H, dk]
    k: torch.Tensor          # bf16 [steps, N, H, dk]
    v: torch.Tensor          # bf16 [steps, N, H, dv]
    log_alpha: torch.Tensor  # f32 [steps, N, H, dk]
    beta: torch.Tensor       # f32 [steps, N, H]
    S: torch.Tensor          # f32 [N, H, dk, dv] state before the first step
    name: str = ""


def make_decode(N, H, dk, dv=None, steps=64, *, seed=4, s_std=0.02, name="") -> DecodeInputs:
    """Fresh per-step decode inputs drawn with the common recipe.

    The per-step tensors are drawn exactly like a prefill of ``steps * N``
    tokens laid out [steps, N] (step-major), then the state.
    """
    dv = dk if dv is None else dv
    p = make_prefill([steps * N], H, dk, dv, seed=seed, s0_std=0.0)
    rng = np.random.default_rng(seed + 1000)
    S = torch.from_numpy(rng.standard_normal((N, H, dk, dv), dtype=np.float32)
                         * np.float32(s_std))
    return DecodeInputs(q=p.q.view(steps, N, H, dk), k=p.k.view(steps, N, H, dk),
                        v=p.v.view(steps, N, H, dv),
                        log_alpha=p.log_alpha.view(steps, N, H, dk),
                        beta=p.beta.view(steps, N, H), S=S, name=name)


def decode_workload(steps=64) -> DecodeInputs:
    return make_decode(256, 32, 128, steps=steps, seed=4, name=WORKLOADS[4])


# ---------------------------------------------------------------- raw inputs
# For the entry points that prepare their inputs on load (kda_chunk_fwd_fused,
# kda_decode_step_fused): q and k are NOT normalised and the decay arrives as a
# gate logit.  Draws: q, k, v ~ N(0, 1) and gate ~ N(0, 1) in float32, each
# rounded to bfloat16 (nearest even); beta = sigmoid(N(0, 1)) float32; S0 as
# in make_prefill.  The gate's N(0, 1) is the input of the workloads'
# -5 * sigmoid curve; applying that curve is the layer's job here, not this
# module's.

@dataclass
class RawPrefillInputs:
    q_raw: torch.Tensor      # bf16 [total_T, H, dk], unnormalised
    k_raw: torch.Tensor      # bf16 [total_T, H, dk], unnormalised
    v: torch.Tensor          # bf16 [total_T, H, dv]
    gate: torch.Tensor       # bf16 [total_T, H, dk], logits
    beta: torch.Tensor       # f32 [total_T, H]
    S0: torch.Tensor | None  # f32 [N, H, dk, dv]
    cu_seqlens: np.ndarray   # int64 [N + 1]
    name: str = ""

    @property
    def total_T(self) -> int:
        return int(self.q_raw.shape[0])

    @property
    def n_seqs(self) -> int:
        return int(self.cu_seqlens.shape[0] - 1)

    @property
    def H(self) -> int:
        return int(self.q_raw.shape[1])

    @property
    def dk(self) -> int:
        return int(self.q_raw.shape[2])

    @property
    def dv(self) -> int:
        return int(self.v.shape[2])


def make_prefill_raw(seq_lens, H, dk, dv=None, *, seed=0, s0_std=0.0, q_scale=1.0,
                     name="") -> RawPrefillInputs:
    """Seeded raw prefill inputs (draw order q, k, v, gate, beta, S0).

    ``q_scale`` multiplies the q draw before rounding (the layer's
    normalisation must make the result independent of it)."""
    dv = dk if dv is None else dv
    seq_lens = [int(x) for x in seq_lens]
    total_T = sum(seq_lens)
    rng = np.random.default_rng(seed)
    q = _to_bf16(_normal_blocks(rng, total_T, (H, dk)) * np.float32(q_scale), False)
    k = _to_bf16(_normal_blocks(rng, total_T, (H, dk)), False)
    v = _to_bf16(_normal_blocks(rng, total_T, (H, dv)), False)
    gate = _to_bf16(_normal_blocks(rng, total_T, (H, dk)), False)
    b = _sigmoid(_normal_blocks(rng, total_T, (H,)))
    N = len(seq_lens)
    S0 = None
    if s0_std:
        S0 = torch.from_numpy(
            (rng.standard_normal((N, H, dk, dv), dtype=np.float32) * np.float32(s0_std)))
    cu = np.zeros(N + 1, dtype=np.int64)
    cu[1:] = np.cumsum(seq_lens)
    return RawPrefillInputs(q_raw=q, k_raw=k, v=v, gate=gate,
                            beta=torch.from_numpy(np.ascontiguousarray(b)), S0=S0,
                            cu_seqlens=cu, name=name)


@dataclass
class RawDecodeInputs:
    q_raw: torch.Tensor      # bf16 [steps, N, H, dk]
    k_raw: torch.Tensor      # bf16 [steps, N, H, dk]
    v: torch.Tensor          # bf16 [steps, N, H, dv]
    gate: torch.Tensor       # bf16 [steps, N, H, dk]
    beta: torch.Tensor       # f32 [steps, N, H]
    S: torch.Tensor          # f32 [N, H, dk, dv]
    name: str = ""


def make_decode_raw(N, H, dk, dv=None, steps=8, *, seed=5, s_std=0.02, name="") -> RawDecodeInputs:
    """Raw per-step decode inputs, drawn like a raw prefill of steps * N tokens [steps, N]."""
    dv = dk if dv is None else dv
    p = make_prefill_raw([steps * N], H, dk, dv, seed=seed)
    rng = np.random.default_rng(seed + 1000)
    S = torch.from_numpy(rng.standard_normal((N, H, dk, dv), dtype=np.float32)
                         * np.float32(s_std))
    return RawDecodeInputs(q_raw=p.q_raw.view(steps, N, H, dk), k_raw=p.k_raw.view(steps, N, H, dk),
                           v=p.v.view(steps, N, H, dv), gate=p.gate.view(steps, N, H, dk),
                           beta=p.beta.view(steps, N, H), S=S, name=name)


# ---------------------------------------------------------------- device draws
# The same recipe drawn directly on a CUDA device with torch's generator, for
# timing runs of the large workloads: the shapes, sequence lengths, value
# distributions and specials are those of :func:`workload`, the values are not
# (a different random stream).  Parity tests use :func:`workload`.

def _dev_normal(g, shape, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def _dev_unit_bf16(g, T, H, d, device, block=_BLOCK):
    out = torch.empty((T, H, d), dtype=torch.bfloat16, device=device)
    for t0 in range(0, T, block):
        x = _dev_normal(g, (min(block, T - t0), H, d), device)
        nrm = torch.linalg.vector_norm(x, dim=-1, keepdim=True).clamp_min(1e-12)
        out[t0:t0 + x.shape[0]] = (x / nrm).to(torch.bfloat16)
    return out


def make_prefill_device(seq_lens, H, dk, dv=None, *, seed=0, s0_std=0.0,
                        log_alpha_fixed=None, log_alpha_fixed_channels=None,
                        beta_mode="sigmoid", name="", device="cuda") -> PrefillInputs:
    """:func:`make_prefill`'s recipe drawn on ``device`` (tensors stay there)."""
    dv = dk if dv is None else dv
    seq_lens = [int(x) for x in seq_lens]
    T = sum(seq_lens)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    q = _dev_unit_bf16(g, T, H, dk, device)
    k = _dev_unit_bf16(g, T, H, dk, device)
    v = torch.empty((T, H, dv), dtype=torch.bfloat16, device=device)
    la = torch.empty((T, H, dk), dtype=torch.float32, device=device)
    for t0 in range(0, T, _BLOCK):
        n = min(_BLOCK, T - t0)
        v[t0:t0 + n] = _dev_normal(g, (n, H, dv), device).to(torch.bfloat16)
        la[t0:t0 + n] = -5.0 * torch.sigmoid(_dev_normal(g, (n, H, dk), device))
    b = torch.sigmoid(_dev_normal(g, (T, H), device))
    if log_alpha_fixed is not None:
        sl = log_alpha_fixed_channels if log_alpha_fixed_channels is not None else slice(None)
        la[:, :, sl] = float(log_alpha_fixed)
    if beta_mode == "mix":
        pick = torch.randint(0, 3, (T, H), generator=g, device=device)
        b = torch.where(pick == 0, torch.zeros_like(b), torch.where(pick == 1, torch.ones_like(b), b))
    elif beta_mode != "sigmoid":
        raise ValueError(beta_mode)
    N = len(seq_lens)
    S0 = _dev_normal(g, (N, H, dk, dv), device) * s0_std if s0_std else None
    cu = np.zeros(N + 1, dtype=np.int64)
    cu[1:] = np.cumsum(seq_lens)
    return PrefillInputs(q=q, k=k, v=v, log_alpha=la, beta=b.contiguous(), S0=S0,
                         cu_seqlens=cu, uniform=len(set(seq_lens)) <= 1, name=name)


def workload_device(idx: int, device="cuda") -> PrefillInputs:
    """Prefill workload ``idx`` (1..3) drawn on ``device``: same shapes, lengths,
    distributions and specials as :func:`workload`, different values."""
    if idx == 1:
        return make_prefill_device([4096] * 4, 32, 128, seed=1, s0_std=0.02,
                                   name=WORKLOADS[1], device=device)
    if idx == 2:
        return make_prefill_device([65536], 16, 128, seed=2, s0_std=0.0, log_alpha_fixed=-5.0,
                                   log_alpha_fixed_channels=slice(0, 64), beta_mode="mix",
                                   name=WORKLOADS[2], device=device)
    if idx == 3:
        return make_prefill_device(million_token_lengths(), 8, 128, seed=3, s0_std=0.02,
                                   name=WORKLOADS[3], device=device)
    raise ValueError(f"no device-drawn prefill workload {idx}")
