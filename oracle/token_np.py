"""NumPy twin of the fp64 token recurrence -- TEST INFRASTRUCTURE ONLY (tiny inputs).

Same definition as ``kda_oracle.c`` (KDA recurrence with the FlashKDA README
"Kernel API" conventions), written independently with whole-matrix NumPy
operations so that the two can check one another:

    ghat = lower_bound * sigmoid(exp(A_log[h]) * (g + dt_bias[h]))
    S    = (I - beta k k^T) Diag(exp(ghat)) S + beta k v^T
    o    = scale * S^T q                      (q, k L2-normalised, eps 1e-6)

Arrays are fp64 NumPy: q, k, g [B,T,H,K], v [B,T,H,V], beta [B,T,H];
initial/final state [N,H,V,K] (state[n,h,v,c] = S[c,v]).
"""
from __future__ import annotations

import numpy as np

L2_EPS = 1e-6


def gate_log_decay(g, dt_bias_h, A_log_h, lower_bound):
    """Per-channel log-decay ghat (natural log) of one token and head."""
    x = np.exp(A_log_h) * (g + dt_bias_h)
    return lower_bound * (1.0 / (1.0 + np.exp(-x)))


def l2_normalise(x):
    return x / np.sqrt(np.dot(x, x) + L2_EPS)


def forward(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, initial_state=None,
            cu_seqlens=None):
    """Token recurrence in the product form S <- (I - b k k^T) D S + b k v^T."""
    B, T, H, K = q.shape
    V = v.shape[-1]
    qf, kf, vf, gf = (a.reshape(B * T, H, -1) for a in (q, k, v, g))
    bf = beta.reshape(B * T, H)
    if cu_seqlens is None:
        bounds = [(n * T, (n + 1) * T) for n in range(B)]
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        bounds = [(int(cu[n]), int(cu[n + 1])) for n in range(len(cu) - 1)]
    N = len(bounds)
    out = np.zeros((B * T, H, V))
    fin = np.zeros((N, H, V, K))
    eye = np.eye(K)
    for n, (t0, t1) in enumerate(bounds):
        for h in range(H):
            S = np.zeros((K, V)) if initial_state is None else initial_state[n, h].T.copy()
            for t in range(t0, t1):
                qh, kh = l2_normalise(qf[t, h]), l2_normalise(kf[t, h])
                b = 1.0 / (1.0 + np.exp(-bf[t, h]))
                D = np.diag(np.exp(gate_log_decay(gf[t, h], dt_bias[h], A_log[h], lower_bound)))
                S = (eye - b * np.outer(kh, kh)) @ D @ S + b * np.outer(kh, vf[t, h])
                out[t, h] = scale * S.T @ qh
            fin[n, h] = S.T
    return out, fin
