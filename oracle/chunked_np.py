"""Chunked (WY/UT) form of the KDA forward pass in NumPy fp64 -- TEST INFRASTRUCTURE ONLY.

FlashKDA processes a sequence in 16-token chunks ("Delta Attention Algorithm
... processes 16-token chunks") and inverts the chunk's unit lower-triangular
system with a Neumann-series product ("Neumann-series expansion ... matrix
inversion").  This module writes that chunked form out plainly, one chunk at
a time, with the chunk length C as a parameter (C = 16 is FlashKDA's; any C
reaches the same result as the token recurrence up to rounding).

Per chunk, with S0 the state (K x V) on entry, rows i, j < n_valid:
    G[i]    = sum_{r<=i} ghat[r]                 (per channel, natural log)
    Akk[i,j]= beta_i * sum_c kh[i,c] kh[j,c] exp(G[i,c]-G[j,c])   (j < i)
    Aqk[i,j]=          sum_c qh[i,c] kh[j,c] exp(G[i,c]-G[j,c])   (j <= i)
    Tm      = (I + Akk)^{-1} Diag(beta)
    W       = Tm (kh * exp(G)),   U = Tm V
    Vn      = U - W S0
    O       = scale * ((qh * exp(G)) S0 + Aqk Vn)
    S_C     = Diag(exp(G[-1])) S0 + (kh * exp(G[-1] - G))^T Vn
"""
from __future__ import annotations

import numpy as np

from .token_np import gate_log_decay, l2_normalise


def unit_lower_inverse_neumann(A):
    """(I + A)^{-1} for strictly lower-triangular A (n x n) as the product
    (I - A)(I + A^2)(I + A^4)... ; exact because A^n = 0."""
    n = A.shape[0]
    eye = np.eye(n)
    X = -A
    result = eye + X
    P = X @ X
    span = 2
    while span < n:
        result = result @ (eye + P)
        P = P @ P
        span *= 2
    return result


def unit_lower_inverse_substitution(A):
    """(I + A)^{-1} for strictly lower-triangular A by forward substitution."""
    n = A.shape[0]
    X = np.zeros((n, n))
    for i in range(n):
        X[i, i] = 1.0
        for j in range(i):
            X[i, j] = -np.dot(A[i, j:i], X[j:i, j])
    return X


def forward(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, initial_state=None,
            cu_seqlens=None, chunk=16, inverse="neumann"):
    """Chunked forward; same argument conventions as ``token_np.forward``."""
    inv = unit_lower_inverse_neumann if inverse == "neumann" else unit_lower_inverse_substitution
    B, T, H, K = q.shape
    V = v.shape[-1]
    qf, kf, vf, gf = (a.reshape(B * T, H, -1) for a in (q, k, v, g))
    bf = beta.reshape(B * T, H)
    if cu_seqlens is None:
        bounds = [(n * T, (n + 1) * T) for n in range(B)]
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        bounds = [(int(cu[n]), int(cu[n + 1])) for n in range(len(cu) - 1)]
    out = np.zeros((B * T, H, V))
    fin = np.zeros((len(bounds), H, V, K))
    for n, (t0, t1) in enumerate(bounds):
        for h in range(H):
            S = np.zeros((K, V)) if initial_state is None else initial_state[n, h].T.copy()
            for c0 in range(t0, t1, chunk):
                c1 = min(t1, c0 + chunk)
                m = c1 - c0
                qh = np.stack([l2_normalise(qf[t, h]) for t in range(c0, c1)])
                kh = np.stack([l2_normalise(kf[t, h]) for t in range(c0, c1)])
                Vc = vf[c0:c1, h]
                b = 1.0 / (1.0 + np.exp(-bf[c0:c1, h]))
                gh = np.stack([gate_log_decay(gf[t, h], dt_bias[h], A_log[h], lower_bound)
                               for t in range(c0, c1)])
                G = np.cumsum(gh, axis=0)                       # [m, K]
                decay = np.exp(G[:, None, :] - G[None, :, :])   # [i, j, K]
                Akk = b[:, None] * np.einsum("ic,jc,ijc->ij", kh, kh, decay)
                Akk = np.tril(Akk, -1)
                Aqk = np.tril(np.einsum("ic,jc,ijc->ij", qh, kh, decay), 0)
                Tm = inv(Akk) @ np.diag(b)
                W = Tm @ (kh * np.exp(G))
                U = Tm @ Vc
                Vn = U - W @ S
                out[c0:c1, h] = scale * ((qh * np.exp(G)) @ S + Aqk @ Vn)
                S = np.diag(np.exp(G[-1])) @ S + (kh * np.exp(G[-1][None, :] - G)).T @ Vn
                del m
            fin[n, h] = S.T
    return out, fin
