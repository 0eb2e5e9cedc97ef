"""Chunk-parallel evaluation of Kimi Delta Attention in fp64 -- TEST INFRASTRUCTURE ONLY.

A second, independently derived algorithm for the same recurrence, used only
to pin the token-by-token oracle (``oracle.forward``) on tiny inputs.  It
follows the chunked route the pages describe: the tokens of one chunk are
handled together and only the state is handed from chunk to chunk
(meridianbulletin.com article, section "Parallelizing Sequential State
Updates"); the within-chunk decay enters through differences of cumulative
log-decays (orkas.ai close read, section "A lower bound that deleted a GPU
code path").

Derivation (one head, one chunk of C tokens, S the state entering the chunk,
g_r = sum_{s<=r} clamp(log_alpha_s) the within-chunk cumulative log-decay per
key channel).  Unrolling the recurrence inside the chunk,

    S_r = Diag(e^{g_r}) S + sum_{i<=r} Diag(e^{g_r - g_i}) k_i u_i^T

and the delta-rule correction u_r = beta_r (v_r - (Diag(alpha_r) S_{r-1})^T k_r)
becomes the lower-triangular system

    u_r + sum_{i<r} A_kk[r,i] u_i = beta_r (v_r - S^T (e^{g_r} * k_r)),
    A_kk[r,i] = beta_r sum_c k_{r,c} k_{i,c} e^{g_{r,c} - g_{i,c}}   (i < r)

so U = T (V - K_G S) with T = (I + A_kk)^{-1} Diag(beta) (the UT transform)
and K_G = k * e^{g}.  The chunk outputs and the state handed on are

    O = Q_G S + A_qk U,   A_qk[r,i] = sum_c q_{r,c} k_{i,c} e^{g_{r,c} - g_{i,c}} (i <= r)
    S <- Diag(e^{g_last}) S + (k * e^{g_last - g})^T U

Everything is plain numpy fp64 with an explicit matrix inverse and no
blocking beyond the chunk itself.  All exponents here are <= 0, so nothing
overflows at any chunk size.
"""
from __future__ import annotations

import numpy as np


def chunk_step(q, k, v, log_alpha, beta, S):
    """One chunk of one head.

    q, k, log_alpha: [C, dk]; v: [C, dv]; beta: [C]; S: [dk, dv] (entering).
    Returns (O [C, dv], S_next [dk, dv], intermediates dict).
    """
    la = np.clip(np.asarray(log_alpha, np.float64), -5.0, 0.0)
    g = np.cumsum(la, axis=0)                          # [C, dk]
    C = q.shape[0]
    # pairwise decay e^{g_r - g_i}, only needed for i <= r (exponent <= 0)
    diff = g[:, None, :] - g[None, :, :]               # [C(r), C(i), dk]
    lower_incl = np.tril(np.ones((C, C), dtype=bool))
    lower_strict = np.tril(np.ones((C, C), dtype=bool), -1)
    decay = np.where(lower_incl[:, :, None], np.exp(np.minimum(diff, 0.0)), 0.0)
    A_kk = np.einsum("rc,ic,ric->ri", k, k, decay) * beta[:, None]
    A_kk = np.where(lower_strict, A_kk, 0.0)
    A_qk = np.einsum("rc,ic,ric->ri", q, k, decay)
    A_qk = np.where(lower_incl, A_qk, 0.0)
    T = np.linalg.inv(np.eye(C) + A_kk) @ np.diag(beta)
    K_G = k * np.exp(g)
    Q_G = q * np.exp(g)
    U = T @ (v - K_G @ S)
    O = Q_G @ S + A_qk @ U
    K_tail = k * np.exp(g[-1][None, :] - g)
    S_next = np.exp(g[-1])[:, None] * S + K_tail.T @ U
    return O, S_next, {"g": g, "A_kk": A_kk, "A_qk": A_qk, "T": T, "U": U}


def forward(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, chunk=64):
    """Chunked evaluation over packed sequences, same layout as ``oracle.forward``.

    All inputs float64 (tiny sizes only).  Chunks restart at every sequence
    start; the last chunk of a sequence may be short.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    log_alpha = np.asarray(log_alpha, np.float64)
    beta = np.asarray(beta, np.float64)
    total_T, H, dk = q.shape
    dv = v.shape[2]
    if cu_seqlens is None:
        cu_seqlens = np.array([0, total_T])
    N = len(cu_seqlens) - 1
    out = np.zeros((total_T, H, dv))
    S_final = np.zeros((N, H, dk, dv))
    for n in range(N):
        t0, t1 = int(cu_seqlens[n]), int(cu_seqlens[n + 1])
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else np.asarray(S0[n, h], np.float64).copy()
            for c0 in range(t0, t1, chunk):
                c1 = min(c0 + chunk, t1)
                O, S, _ = chunk_step(q[c0:c1, h], k[c0:c1, h], v[c0:c1, h],
                                     log_alpha[c0:c1, h], beta[c0:c1, h], S)
                out[c0:c1, h] = O
            S_final[n, h] = S
    return out, S_final
