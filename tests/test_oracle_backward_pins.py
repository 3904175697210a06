"""Pins of the oracle's gradient (oracle/kda_oracle_bwd.c) against things other than itself.

* Central finite differences: for L = sum(dout * out) + sum(dfinal * final_state), the
  derivative of L along a random direction of each input (computed from two fp64 forward
  runs) equals the gradient's inner product with that direction.  Every input (q, k, v, g,
  the beta logits, the initial state, A_log, dt_bias) and every switch of the reference
  call (the three gates, beta and the L2 norms off) are covered, with varlen sequences, a
  zero-length one, and with and without the final-state term.
* A closed form: one token from a zero state gives o = scale beta (qh . kh) v, so dv and
  the beta-logit gradient are known exactly.
* Reverse-mode autograd through a plain torch fp64 restatement of the recurrence gives the
  same gradient to rounding (1e-10 relative), for four switch combinations with varlen.
* The fp64 forward the finite differences use is itself pinned to the bf16 forward oracle
  (kda_oracle.c, pinned by its own tests) on bf16-exact inputs.
* Four plausible mistakes planted in copies of the gradient code fail the pins.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle

FLAG_SETS = {
    "default": dict(),
    "softplus_gate": dict(safe_gate=False),
    "preactivated_gate": dict(use_gate_in_kernel=False),
    "beta_given": dict(use_beta_sigmoid_in_kernel=False),
    "no_l2norm": dict(use_qk_l2norm_in_kernel=False),
    "softplus_beta_given_no_norm": dict(safe_gate=False, use_beta_sigmoid_in_kernel=False,
                                        use_qk_l2norm_in_kernel=False),
}


def _case(seed, B=1, T=7, H=2, K=5, V=3, lens=None, init=True, kw=None):
    rng = np.random.default_rng(seed)
    kw = kw or {}
    x = dict(q=rng.standard_normal((B, T, H, K)), k=rng.standard_normal((B, T, H, K)),
             v=rng.standard_normal((B, T, H, V)), g=rng.standard_normal((B, T, H, K)),
             beta=rng.standard_normal((B, T, H)), A_log=rng.uniform(-1, 1, H),
             dt_bias=0.3 * rng.standard_normal((H, K)))
    if kw.get("use_gate_in_kernel") is False:
        x["g"] = -np.abs(x["g"]) * 0.5          # a natural-log decay, at most 0
    if kw.get("use_beta_sigmoid_in_kernel") is False:
        x["beta"] = rng.uniform(0.05, 0.95, (B, T, H))
    N = B if lens is None else len(lens)
    x["initial_state"] = 0.3 * rng.standard_normal((N, H, V, K)) if init else None
    x["cu_seqlens"] = None if lens is None else np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    x["scale"] = 0.7
    x["lower_bound"] = -2.5
    dout = rng.standard_normal((B, T, H, V))
    dfinal = rng.standard_normal((N, H, V, K))
    return x, dout, dfinal


def _loss(x, dout, dfinal, kw):
    out, fin = oracle.kda_forward64(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["A_log"],
                                    x["dt_bias"], x["lower_bound"], x["initial_state"], x["cu_seqlens"], **kw)
    L = float(np.sum(dout * out))
    if dfinal is not None:
        L += float(np.sum(dfinal * fin))
    return L


def _grads(x, dout, dfinal, kw):
    return oracle.kda_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["A_log"], x["dt_bias"],
                               x["lower_bound"], dout, x["initial_state"], dfinal, x["cu_seqlens"], **kw)


GRAD_OF = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", initial_state="dh0", A_log="dA_log",
               dt_bias="ddt_bias")


def _check_directional(x, dout, dfinal, kw, seed, eps=1e-6, rtol=2e-6):
    gr = _grads(x, dout, dfinal, kw)
    rng = np.random.default_rng(seed)
    names = [n for n in GRAD_OF if x.get(n) is not None]
    if kw.get("use_gate_in_kernel") is False:
        names = [n for n in names if n not in ("A_log", "dt_bias")]
    for name in names:
        for _ in range(2):
            d = rng.standard_normal(np.shape(x[name]))
            xp, xm = dict(x), dict(x)
            xp[name] = x[name] + eps * d
            xm[name] = x[name] - eps * d
            fd = (_loss(xp, dout, dfinal, kw) - _loss(xm, dout, dfinal, kw)) / (2 * eps)
            an = float(np.sum(gr[GRAD_OF[name]] * d))
            assert abs(fd - an) <= rtol * max(1.0, abs(an)), f"{name}: finite difference {fd} vs gradient {an}"
    return gr


@pytest.mark.parametrize("name", list(FLAG_SETS))
def test_gradient_matches_finite_differences(name):
    kw = FLAG_SETS[name]
    x, dout, dfinal = _case(11, kw=kw)
    _check_directional(x, dout, dfinal, kw, seed=12)


def test_gradient_varlen_zero_length_and_no_final_term():
    x, dout, dfinal = _case(21, T=11, H=2, lens=[4, 0, 6, 1])
    _check_directional(x, dout, None, {}, seed=22)
    gr = _check_directional(x, dout, dfinal, {}, seed=23)
    # the zero-length sequence: its initial state reaches only its final state
    assert np.array_equal(gr["dh0"][1], dfinal[1])


def test_gradient_without_initial_state_matches_a_zero_initial_state():
    x, dout, dfinal = _case(31, init=False)
    g0 = _grads(x, dout, dfinal, {})
    x2 = dict(x)
    x2["initial_state"] = np.zeros((1, 2, 3, 5))
    g1 = _check_directional(x2, dout, dfinal, {}, seed=32)
    for n in ("dq", "dk", "dv", "dg", "dbeta", "dh0", "dA_log", "ddt_bias"):
        assert np.array_equal(g0[n], g1[n])


def test_gradient_wider_heads_fixed_batch():
    x, dout, dfinal = _case(41, B=2, T=9, H=1, K=16, V=8)
    _check_directional(x, dout, dfinal, {}, seed=42)


def test_one_token_closed_form():
    # S_0 = 0: u = v, S_1 = beta kh v^T, o = scale beta (qh . kh) v
    x, dout, _ = _case(51, T=1, H=1, init=False)
    gr = _grads(x, dout, None, {})
    q, k = x["q"][0, 0, 0], x["k"][0, 0, 0]
    qh = q / np.sqrt(q @ q + 1e-6)
    kh = k / np.sqrt(k @ k + 1e-6)
    b = 1.0 / (1.0 + np.exp(-x["beta"][0, 0, 0]))
    v, do = x["v"][0, 0, 0], dout[0, 0, 0]
    s = x["scale"] * (qh @ kh)
    np.testing.assert_allclose(gr["dv"][0, 0, 0], s * b * do, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(gr["dbeta"][0, 0, 0], s * (v @ do) * b * (1 - b), rtol=1e-12)
    # the decay multiplies a zero state: the gate and its parameters get no gradient
    assert np.all(gr["dg"] == 0) and np.all(gr["dA_log"] == 0) and np.all(gr["ddt_bias"] == 0)


@pytest.mark.parametrize("name", ["default", "softplus_gate", "preactivated_gate", "no_l2norm"])
def test_fp64_forward_matches_the_bf16_oracle(name):
    kw = FLAG_SETS[name]
    rng = np.random.default_rng(61)
    B, T, H, K, V = 1, 40, 2, 128, 128

    def bf(a):
        return torch.tensor(a, dtype=torch.float32).to(torch.bfloat16)

    t = dict(q=bf(rng.standard_normal((B, T, H, K))), k=bf(rng.standard_normal((B, T, H, K))),
             v=bf(rng.standard_normal((B, T, H, V))), g=bf(rng.standard_normal((B, T, H, K))),
             beta=bf(rng.standard_normal((B, T, H))))
    if kw.get("use_gate_in_kernel") is False:
        t["g"] = bf(-np.abs(rng.standard_normal((B, T, H, K))))
    A = torch.tensor(rng.uniform(-1, 1, H), dtype=torch.float32)
    D = torch.tensor(0.1 * rng.standard_normal((H, K)), dtype=torch.float32)
    s0 = torch.tensor(0.02 * rng.standard_normal((B, H, V, K)), dtype=torch.float32)
    cu = np.array([0, 15, 40], dtype=np.int64)
    scale, lb = float(np.float32(K ** -0.5)), -3.0
    o_ref, f_ref = oracle.kda_forward(t["q"], t["k"], t["v"], t["g"], t["beta"], scale, A, D, lb,
                                      torch.cat([s0, s0]), cu, **kw)
    f64 = {n: t[n].double().numpy() for n in t}
    o, f = oracle.kda_forward64(f64["q"], f64["k"], f64["v"], f64["g"], f64["beta"], scale, A.double().numpy(),
                                D.double().numpy(), lb, torch.cat([s0, s0]).double().numpy(), cu, **kw)
    # the two differ only in the order of fp64 roundings
    np.testing.assert_allclose(o.reshape(o_ref.shape), o_ref, rtol=0, atol=1e-12 * max(1.0, np.abs(o_ref).max()))
    np.testing.assert_allclose(f, f_ref, rtol=0, atol=1e-12 * max(1.0, np.abs(f_ref).max()))


MUTATIONS = {
    "sign of the P du term": ("W->dkh[c] = b * s1 - s2;", "W->dkh[c] = b * s1 + s2;"),
    "dalpha against S_t": ("s += dP[c * V + j] * Sprev[c * V + j];", "s += dP[c * V + j] * St[c * V + j];"),
    "dropped output term": ("dS[c * V + j] += J->scale * qh[c] * dO[j];", "(void)0;"),
    "decay not carried": ("for (int64_t j = 0; j < V; ++j) dS[c * V + j] = al[c] * dP[c * V + j];",
                          "for (int64_t j = 0; j < V; ++j) dS[c * V + j] = dP[c * V + j];"),
}


@pytest.mark.parametrize("what", list(MUTATIONS))
def test_finite_differences_catch_a_planted_mistake(tmp_path, monkeypatch, what):
    """A plausible mistake planted in a copy of the backward oracle fails the pins."""
    import ctypes
    import os
    import subprocess

    src = open(os.path.join(os.path.dirname(oracle.__file__), "kda_oracle_bwd.c")).read()
    a, b = MUTATIONS[what]
    assert src.count(a) == 1
    (tmp_path / "m.c").write_text(src.replace(a, b))
    fwd = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")
    lib_path = str(tmp_path / "libm.so")
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", fwd,
                           str(tmp_path / "m.c"), "-o", lib_path, "-lm"])
    good = oracle._load()
    bad = ctypes.CDLL(lib_path)
    for fn in ("kda_oracle_fwd", "kda_oracle_fwd64", "kda_oracle_bwd"):
        getattr(bad, fn).argtypes = getattr(good, fn).argtypes
        getattr(bad, fn).restype = ctypes.c_int
    monkeypatch.setattr(oracle, "_lib", bad)
    x, dout, dfinal = _case(71)
    with pytest.raises(AssertionError):
        _check_directional(x, dout, dfinal, {}, seed=72)


def _torch_forward(t, kw):
    """The recurrence restated with torch fp64 operations (for autograd), token by token."""
    B, T, H, K = t["q"].shape
    V = t["v"].shape[-1]
    cu = t["cu_seqlens"]
    N = B if cu is None else len(cu) - 1
    outs = torch.zeros(B * T, H, V, dtype=torch.float64)
    fins = []
    q, k, v, g = (t[n].reshape(B * T, H, -1) for n in ("q", "k", "v", "g"))
    b = t["beta"].reshape(B * T, H)
    for n in range(N):
        t0, t1 = (n * T, (n + 1) * T) if cu is None else (int(cu[n]), int(cu[n + 1]))
        for h in range(H):
            S = t["initial_state"][n, h].T if t["initial_state"] is not None else torch.zeros(K, V, dtype=torch.float64)
            for i in range(t0, t1):
                qi, ki, gi = q[i, h], k[i, h], g[i, h]
                if kw.get("use_qk_l2norm_in_kernel", True):
                    qi = qi / torch.sqrt(qi @ qi + 1e-6)
                    ki = ki / torch.sqrt(ki @ ki + 1e-6)
                if kw.get("use_gate_in_kernel", True) is False:
                    gh = gi
                elif kw.get("safe_gate", True) is False:
                    gh = -torch.exp(t["A_log"][h]) * torch.nn.functional.softplus(gi + t["dt_bias"][h])
                else:
                    gh = t["lower_bound"] * torch.sigmoid(torch.exp(t["A_log"][h]) * (gi + t["dt_bias"][h]))
                bi = b[i, h] if kw.get("use_beta_sigmoid_in_kernel", True) is False else torch.sigmoid(b[i, h])
                P = torch.exp(gh)[:, None] * S
                u = v[i, h] - P.T @ ki
                S = P + bi * torch.outer(ki, u)
                outs[i, h] = t["scale"] * (S.T @ qi)
            fins.append(S.T)
    return outs.reshape(B, T, H, V), torch.stack(fins).reshape(N, H, V, K)


@pytest.mark.parametrize("name", ["default", "softplus_gate", "preactivated_gate", "softplus_beta_given_no_norm"])
def test_gradient_equals_autograd_of_a_torch_restatement(name):
    """Reverse-mode autograd through plain torch fp64 operations gives the same gradient to
    rounding (an exact check, where finite differences hold to about 1e-6)."""
    kw = FLAG_SETS[name]
    x, dout, dfinal = _case(81, T=6, H=2, K=4, V=3, lens=[2, 0, 4], kw=kw)
    gr = _grads(x, dout, dfinal, kw)
    t = {n: (torch.tensor(x[n], dtype=torch.float64, requires_grad=True) if n in GRAD_OF and x[n] is not None
             else x[n]) for n in x}
    out, fin = _torch_forward(t, kw)
    L = (out * torch.tensor(dout)).sum() + (fin * torch.tensor(dfinal)).sum()
    L.backward()
    for n, gn in GRAD_OF.items():
        if kw.get("use_gate_in_kernel") is False and n in ("A_log", "dt_bias"):
            continue
        np.testing.assert_allclose(t[n].grad.numpy(), gr[gn], rtol=1e-10, atol=1e-12, err_msg=n)


@pytest.mark.parametrize("chunk,name", [(16, "default"), (5, "default"), (1, "default"), (16, "softplus_gate"),
                                        (7, "preactivated_gate"), (16, "softplus_beta_given_no_norm"),
                                        (4, "beta_given"), (16, "no_l2norm")])
def test_chunked_form_gradient_equals_the_token_gradient(chunk, name):
    """The chunked (WY/UT) gradient of oracle/chunked_bwd_np.py, a separate derivation through
    dense per-chunk products, equals the token oracle's gradient to fp64 rounding, for every
    switch of the reference call."""
    from oracle import chunked_bwd_np

    kw = FLAG_SETS[name]
    x, dout, dfinal = _case(91, T=45, H=2, K=6, V=4, lens=[17, 0, 3, 25], kw=kw)
    ref = _grads(x, dout, dfinal, kw)
    got = chunked_bwd_np.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["A_log"],
                                  x["dt_bias"], x["lower_bound"], dout, x["initial_state"], dfinal,
                                  x["cu_seqlens"], chunk=chunk, **kw)
    for n in GRAD_OF.values():
        np.testing.assert_allclose(got[n], ref[n], rtol=1e-9, atol=1e-11 * max(1.0, np.abs(ref[n]).max()),
                                   err_msg=n)
