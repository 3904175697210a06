"""Chunked (WY/UT) form of the KDA gradient in NumPy fp64 -- TEST INFRASTRUCTURE ONLY.

The gradient the token-level oracle (kda_oracle_bwd.c) computes, reached instead through the
16-token chunked form of the forward (the form oracle/chunked_np.py writes out; FlashKDA works
in chunks of 16 tokens, instagit index, delta-attention article), differentiated chunk by chunk.
Every step is a small dense product, the shape a tensor-core backward would take; this
module states and checks that math before any kernel does.  The reference call's switches
change only the per-token ends: the gate (safe sigmoid, softplus or pre-activated), the beta
sigmoid and the L2 norms.

Per chunk of m tokens with S0 (K x V) on entry, G the inclusive cumsum of ghat (natural log),
Gam = exp(G), Gc = Gam[m-1]:
    Kp = kh Gam,  Km = kh / Gam,  Qp = qh Gam,  Kd = kh Gc / Gam          (rows, per channel)
    A  = Diag(beta) strict_lower(Kp Km^T),  M = (I + A)^{-1},  Tm = M Diag(beta)
    W  = Tm Kp,  U = Tm V,  Vn = U - W S0,  P = lower(Qp Km^T)
    O  = scale (Qp S0 + P Vn),  S1 = Diag(Gc) S0 + Kd^T Vn
Reverse, from dO and dS1:
    dVn = scale P^T dO + Kd dS1;  dP = lower(scale dO Vn^T)
    dQp = scale dO S0^T + dP Km;  dKm = dP^T Qp;  dKd = Vn dS1^T
    dS0 = scale Qp^T dO + Diag(Gc) dS1 - W^T dVn
    dT = dVn V^T - dVn S0^T Kp^T;  dV = Tm^T dVn;  dKp = -Tm^T dVn S0^T
    dM = dT Diag(beta);  dbeta_s += sum_r dT[r,s] M[r,s];  dA = -M^T dM M^T (strictly lower)
    dR = Diag(beta) dA;  dbeta_r += sum_s dA[r,s] R[r,s];  dKp += dR Km;  dKm += dR^T Kp
    dkh = dKp Gam + dKm / Gam + dKd Gc / Gam;  dqh = dQp Gam
    dG  = dKp Kp - dKm Km + dQp Qp - dKd Kd;  dG[m-1] += sum_r dKd_r Kd_r + Gc sum_j dS1 S0
    dghat = reverse cumsum of dG over the chunk
then the norms, the sigmoid and the gate as in the token oracle.
"""
from __future__ import annotations

import numpy as np


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def backward(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, dout, initial_state=None, dfinal=None,
             cu_seqlens=None, chunk=16, use_gate_in_kernel=True, use_beta_sigmoid_in_kernel=True,
             use_qk_l2norm_in_kernel=True, safe_gate=True):
    """fp64 arrays in the token oracle's conventions; returns the same dict of gradients."""
    B, T, H, K = q.shape
    V = v.shape[-1]
    qf, kf, vf, gf, dof = (a.reshape(B * T, H, -1) for a in (q, k, v, g, dout))
    bf = beta.reshape(B * T, H)
    if cu_seqlens is None:
        bounds = [(n * T, (n + 1) * T) for n in range(B)]
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        bounds = [(int(cu[n]), int(cu[n + 1])) for n in range(len(cu) - 1)]
    N = len(bounds)
    r = dict(dq=np.zeros((B * T, H, K)), dk=np.zeros((B * T, H, K)), dv=np.zeros((B * T, H, V)),
             dg=np.zeros((B * T, H, K)), dbeta=np.zeros((B * T, H)), dh0=np.zeros((N, H, V, K)),
             dA_log=np.zeros(H), ddt_bias=np.zeros((H, K)))
    for n, (t0, t1) in enumerate(bounds):
        for h in range(H):
            rate = np.exp(A_log[h]) if use_gate_in_kernel else 0.0

            def prep(c0, c1):
                qq, kk = qf[c0:c1, h], kf[c0:c1, h]
                ones = np.ones(c1 - c0)
                rq = 1.0 / np.sqrt(np.sum(qq * qq, axis=1) + 1e-6) if use_qk_l2norm_in_kernel else ones
                rk = 1.0 / np.sqrt(np.sum(kk * kk, axis=1) + 1e-6) if use_qk_l2norm_in_kernel else ones
                if not use_gate_in_kernel:
                    x = s = None
                    gh = gf[c0:c1, h]
                elif not safe_gate:
                    x = gf[c0:c1, h] + dt_bias[h][None, :]
                    s = _sigmoid(x)
                    gh = -rate * np.where(x > 0, x + np.log1p(np.exp(-np.abs(x))), np.log1p(np.exp(np.minimum(x, 0))))
                else:
                    x = gf[c0:c1, h] + dt_bias[h][None, :]
                    s = _sigmoid(rate * x)
                    gh = lower_bound * s
                b = bf[c0:c1, h] if not use_beta_sigmoid_in_kernel else _sigmoid(bf[c0:c1, h])
                return dict(qh=qq * rq[:, None], kh=kk * rk[:, None], rq=rq, rk=rk, x=x, s=s, gh=gh,
                            b=b, G=np.cumsum(gh, axis=0), V=vf[c0:c1, h])

            def chunk_terms(c, S0):
                Gam = np.exp(c["G"])
                Gc = Gam[-1]
                Kp, Km, Qp = c["kh"] * Gam, c["kh"] / Gam, c["qh"] * Gam
                Kd = c["kh"] * (Gc[None, :] / Gam)
                m = Kp.shape[0]
                R = Kp @ Km.T
                A = c["b"][:, None] * np.tril(R, -1)
                M = np.linalg.inv(np.eye(m) + A)
                Tm = M @ np.diag(c["b"])
                W, U = Tm @ Kp, Tm @ c["V"]
                Vn = U - W @ S0
                P = np.tril(Qp @ Km.T)
                return dict(Gam=Gam, Gc=Gc, Kp=Kp, Km=Km, Qp=Qp, Kd=Kd, R=R, M=M, Tm=Tm, W=W, Vn=Vn, P=P)

            # forward over the chunks, keeping each chunk's entering state
            S = np.zeros((K, V)) if initial_state is None else initial_state[n, h].T.copy()
            starts = list(range(t0, t1, chunk))
            S0s = []
            for c0 in starts:
                c1 = min(t1, c0 + chunk)
                S0s.append(S)
                f = chunk_terms(prep(c0, c1), S)
                S = np.diag(f["Gc"]) @ S + f["Kd"].T @ f["Vn"]
            # reverse over the chunks
            dS = np.zeros((K, V)) if dfinal is None else dfinal[n, h].T.copy()
            for c0, S0 in zip(reversed(starts), reversed(S0s)):
                c1 = min(t1, c0 + chunk)
                c = prep(c0, c1)
                f = chunk_terms(c, S0)
                dO = dof[c0:c1, h]
                dS1 = dS
                dVn = scale * f["P"].T @ dO + f["Kd"] @ dS1
                dP = np.tril(scale * dO @ f["Vn"].T)
                dQp = scale * dO @ S0.T + dP @ f["Km"]
                dKm = dP.T @ f["Qp"]
                dKd = f["Vn"] @ dS1.T
                dS = scale * f["Qp"].T @ dO + f["Gc"][:, None] * dS1 - f["W"].T @ dVn
                dW = -dVn @ S0.T
                dT = dVn @ c["V"].T + dW @ f["Kp"].T
                dV = f["Tm"].T @ dVn
                dKp = f["Tm"].T @ dW
                dM = dT * c["b"][None, :]
                dbeta = np.sum(dT * f["M"], axis=0)
                dA = np.tril(-f["M"].T @ dM @ f["M"].T, -1)
                dR = c["b"][:, None] * dA
                dbeta += np.sum(dA * f["R"], axis=1)
                dKp += dR @ f["Km"]
                dKm += dR.T @ f["Kp"]
                Gam, Gc = f["Gam"], f["Gc"]
                dkh = dKp * Gam + dKm / Gam + dKd * (Gc[None, :] / Gam)
                dqh = dQp * Gam
                dG = dKp * f["Kp"] - dKm * f["Km"] + dQp * f["Qp"] - dKd * f["Kd"]
                dG[-1] += np.sum(dKd * f["Kd"], axis=0) + Gc * np.sum(dS1 * S0, axis=1)
                dgh = np.cumsum(dG[::-1], axis=0)[::-1]
                # the norms, the beta sigmoid and the gate
                qh, kh = c["qh"], c["kh"]
                if use_qk_l2norm_in_kernel:
                    dqh = c["rq"][:, None] * (dqh - qh * np.sum(qh * dqh, axis=1)[:, None])
                    dkh = c["rk"][:, None] * (dkh - kh * np.sum(kh * dkh, axis=1)[:, None])
                r["dq"][c0:c1, h] = dqh
                r["dk"][c0:c1, h] = dkh
                r["dv"][c0:c1, h] = dV
                r["dbeta"][c0:c1, h] = dbeta * c["b"] * (1.0 - c["b"]) if use_beta_sigmoid_in_kernel else dbeta
                if not use_gate_in_kernel:
                    r["dg"][c0:c1, h] = dgh
                    continue
                if safe_gate:     # ghat = lb sigmoid(rate x): d/dx = rate lb s (1 - s), d/dA_log = x d/dx
                    dx = dgh * lower_bound * c["s"] * (1.0 - c["s"]) * rate
                    r["dA_log"][h] += np.sum(dx * c["x"])
                else:             # ghat = -rate softplus(x): d/dx = -rate sigmoid(x), d/dA_log = ghat
                    dx = dgh * (-rate) * c["s"]
                    r["dA_log"][h] += np.sum(dgh * c["gh"])
                r["dg"][c0:c1, h] = dx
                r["ddt_bias"][h] += np.sum(dx, axis=0)
            r["dh0"][n, h] = dS.T
    for key in ("dq", "dk", "dg"):
        r[key] = r[key].reshape(B, T, H, K)
    r["dv"] = r["dv"].reshape(B, T, H, V)
    r["dbeta"] = r["dbeta"].reshape(B, T, H)
    return r
