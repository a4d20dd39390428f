"""Chunk-wise fp64 form of the KDA recurrence (TEST INFRASTRUCTURE ONLY).

This exists to pin the chunk algebra that a parallel implementation uses: it is
compared against the token-by-token oracle for every chunk size.  It is plain
numpy in float64 with no sub-tiling and no reference-point tricks; decay
ratios are formed directly as exp(gamma_r - gamma_i) for i <= r.

Source: "Kimi K3's Architecture: Kimi Delta Attention, Attention Residuals, and
896 Experts", section "Channel-wise decay, and the floor K3 puts under it":
chunk-wise processing is parallel inside a chunk and recurrent across chunks,
built on the cumulative decay inside the chunk.  The pages print no chunk
equations, so the per-chunk algebra below is derived from the recurrence
S_r = Diag(alpha_r) S_{r-1} + k_r u_r^T,  u_r = beta_r (v_r - (Diag(alpha_r) S_{r-1})^T k_r)
by unrolling it over the chunk (S0 = state entering the chunk):

  gamma_r  = sum_{u<=r} log alpha_u                (inclusive, per channel)
  A[r,i]   = beta_r sum_c k_r[c] k_i[c] e^{gamma_r[c]-gamma_i[c]}   (i < r)
  P[r,i]   = sum_c q_r[c] k_i[c] e^{gamma_r[c]-gamma_i[c]}          (i <= r)
  (I + A) U = diag(beta) (V - K~ S0),  K~_r = k_r * e^{gamma_r}
  O        = scale (Q~ S0 + P U),       Q~_r = q_r * e^{gamma_r}
  S_C      = Diag(e^{gamma_C}) S0 + K^^T U,  K^_i = k_i * e^{gamma_C - gamma_i}
"""
from __future__ import annotations

import numpy as np


def kda_chunked_single(q, k, v, log_alpha, beta, S0, chunk, scale):
    """One sequence, one head.  q, k, log_alpha: [T, dk]; v: [T, dv]; beta: [T];
    S0: [dk, dv].  Returns (o [T, dv], S_final [dk, dv])."""
    q, k, v, la = (np.asarray(x, np.float64) for x in (q, k, v, log_alpha))
    beta = np.asarray(beta, np.float64)
    T = q.shape[0]
    S = np.array(S0, np.float64, copy=True)
    o = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, chunk):
        sl = slice(c0, min(c0 + chunk, T))
        n = sl.stop - sl.start
        qc, kc, vc, bc = q[sl], k[sl], v[sl], beta[sl]
        gam = np.cumsum(la[sl], axis=0)
        causal = np.tril(np.ones((n, n), bool))
        diff = np.where(causal[:, :, None], gam[:, None, :] - gam[None, :, :], -np.inf)
        decay = np.exp(diff)                                  # e^{gamma_r - gamma_i}, i <= r
        kk = np.einsum("rc,ic,ric->ri", kc, kc, decay)
        A = bc[:, None] * np.tril(kk, -1)
        P = np.einsum("rc,ic,ric->ri", qc, kc, decay)
        K_tilde = kc * np.exp(gam)
        Q_tilde = qc * np.exp(gam)
        K_hat = kc * np.exp(gam[-1] - gam)
        M = np.eye(n) + A
        U = np.linalg.solve(M, bc[:, None] * (vc - K_tilde @ S))
        o[sl] = scale * (Q_tilde @ S + P @ U)
        S = np.exp(gam[-1])[:, None] * S + K_hat.T @ U
    return o, S
