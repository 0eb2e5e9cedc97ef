"""Kimi Delta Attention oracle -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU
baseline and ``--impl reference`` legs) may import this package.  The CUDA
library never calls it, and it imports nothing from the CUDA package.

Two independent evaluators live here:

* :func:`forward` -- the fp64 token-by-token recurrence in ``kda_oracle.c``
  (plain C, compiled with ``gcc -O2``, no fast-math), threaded over
  independent (sequence, head) chains.  This is the parity reference.
* :mod:`oracle.naive_chunked` -- the chunk-parallel form (WY/UT transform,
  explicit matrix inverse) written in numpy fp64 for tiny inputs; it exists
  to pin the recurrence against a second, differently derived algorithm.

The recurrence, per head, with S of shape dk x dv and one decay per key
channel (lecture "Inside Kimi K3: Architecture of an Open Frontier Model",
sequence paragraph; meridianbulletin.com article, section "Handling One
Million Tokens with a Fixed-Size State Matrix"):

    S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
    o_t = S_t^T q_t,        alpha_t = exp(clamp(log_alpha_t, -5, 0))
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

IN_F64 = 0
IN_BF16 = 1


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/libkda_oracle.so``."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC",
                               "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.kda_oracle_forward.restype = ctypes.c_int
            lib.kda_oracle_forward.argtypes = (
                [ctypes.c_void_p] * 6
                + [ctypes.c_void_p]
                + [ctypes.c_int64] * 6
                + [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int])
            _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover - non-Linux
        return os.cpu_count() or 1


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def forward(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, *,
            heads=None, threads=None):
    """Evaluate the recurrence in fp64.

    Inputs are numpy arrays in the packed layout
    ``q, k, log_alpha: [total_T, H, dk]``, ``v: [total_T, H, dv]``,
    ``beta: [total_T, H]``, ``S0: [N, H, dk, dv]`` (None = zero state),
    ``cu_seqlens: int [N+1]`` (None = one sequence of length total_T).

    Encodings: either every array is float64, or q/k/v are bfloat16 bit
    patterns (uint16) and log_alpha/beta/S0 are float32 -- the values the GPU
    path receives, widened exactly.

    ``heads`` = (begin, end) evaluates only those heads; outputs then carry
    ``end - begin`` heads.  Returns ``(out [total_T, nh, dv], S_final
    [N, nh, dk, dv])``, both float64.
    """
    lib = _load()
    if q.dtype == np.uint16:
        kind = IN_BF16
        qkv_t, gate_t = np.uint16, np.float32
    else:
        kind = IN_F64
        qkv_t, gate_t = np.float64, np.float64
    q = np.ascontiguousarray(q, dtype=qkv_t)
    k = np.ascontiguousarray(k, dtype=qkv_t)
    v = np.ascontiguousarray(v, dtype=qkv_t)
    log_alpha = np.ascontiguousarray(log_alpha, dtype=gate_t)
    beta = np.ascontiguousarray(beta, dtype=gate_t)
    total_T, H, dk = q.shape
    dv = v.shape[2]
    if k.shape != q.shape or log_alpha.shape != q.shape:
        raise ValueError("q, k and log_alpha must share a shape")
    if v.shape[:2] != (total_T, H) or beta.shape != (total_T, H):
        raise ValueError("v / beta shape mismatch")
    if cu_seqlens is None:
        cu_seqlens = np.array([0, total_T], dtype=np.int64)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    N = cu.shape[0] - 1
    if cu[-1] != total_T:
        raise ValueError("cu_seqlens[-1] must equal total_T")
    if S0 is not None:
        S0 = np.ascontiguousarray(S0, dtype=gate_t)
        if S0.shape != (N, H, dk, dv):
            raise ValueError("S0 shape mismatch")
    h0, h1 = (0, H) if heads is None else heads
    nh = h1 - h0
    out = np.zeros((total_T, nh, dv), dtype=np.float64)
    S_final = np.zeros((N, nh, dk, dv), dtype=np.float64)
    rc = lib.kda_oracle_forward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S0),
        _ptr(cu), N, H, dk, dv, h0, h1, kind, _ptr(out), _ptr(S_final),
        int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_forward failed with code {rc}")
    return out, S_final


def decode_steps(q, k, v, log_alpha, beta, S, *, threads=None):
    """Apply single-token steps to a batch of states.

    ``q, k, log_alpha: [steps, N, H, dk]``, ``v: [steps, N, H, dv]``,
    ``beta: [steps, N, H]``, ``S: [N, H, dk, dv]``.  Every one of the N
    sequences advances by one token per step; the state after each step feeds
    the next.  Returns ``(out [steps, N, H, dv], S_after [N, H, dk, dv])`` in
    float64.  This is the same recurrence as :func:`forward`: the N sequences
    are packed so that sequence n owns tokens ``n*steps .. n*steps+steps-1``.
    """
    steps, N, H, dk = q.shape
    dv = v.shape[3]

    def pack(a):
        # [steps, N, ...] -> [N*steps, ...] with each sequence contiguous
        return np.ascontiguousarray(np.swapaxes(a, 0, 1)).reshape((N * steps,) + a.shape[2:])

    cu = np.arange(N + 1, dtype=np.int64) * steps
    out, S_after = forward(pack(q), pack(k), pack(v), pack(log_alpha), pack(beta), S, cu,
                           threads=threads)
    out = np.swapaxes(out.reshape(N, steps, H, dv), 0, 1)
    return out, S_after
