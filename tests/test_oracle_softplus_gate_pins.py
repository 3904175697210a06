"""Pins for the oracle's second gate, the one the reference call selects with its safe_gate
switch off (FlashKDA README, the chunk_kda call): ghat = -exp(A_log) softplus(g + dt_bias),
with no lower bound.  Each pin recomputes the result in numpy from the definition (softplus
as numpy's logaddexp(0, x)), or uses a value the definition fixes exactly."""
from __future__ import annotations

import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from tests.oracle_helpers import as_f64, l2n

K = V = 128


def _inputs(T, seed, beta_pre=False, g_shift=0.0):
    gen = torch.Generator().manual_seed(seed)
    beta = torch.rand(1, T, 1, generator=gen) if beta_pre else torch.randn(1, T, 1, generator=gen)
    return dict(q=torch.randn(1, T, 1, K, generator=gen).to(torch.bfloat16),
                k=torch.randn(1, T, 1, K, generator=gen).to(torch.bfloat16),
                v=torch.randn(1, T, 1, V, generator=gen).to(torch.bfloat16),
                g=(torch.randn(1, T, 1, K, generator=gen) + g_shift).to(torch.bfloat16),
                beta=beta.to(torch.bfloat16), A_log=torch.rand(1, generator=gen) * 2 - 1,
                dt_bias=torch.randn(1, K, generator=gen) * 0.1, scale=1.0 / math.sqrt(K), lower_bound=-3.0,
                initial_state=torch.randn(1, 1, V, K, generator=gen, dtype=torch.float64) * 0.02)


def _run(x, beta_pre=False, no_norm=False, safe_gate=False):
    return oracle.kda_forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["A_log"], x["dt_bias"],
                              x["lower_bound"], x["initial_state"], use_beta_sigmoid_in_kernel=not beta_pre,
                              use_qk_l2norm_in_kernel=not no_norm, safe_gate=safe_gate)


def _alpha(x, t):
    pre = as_f64(x["g"][0, t, 0]) + x["dt_bias"][0].double().numpy()
    return np.exp(-math.exp(float(x["A_log"][0])) * np.logaddexp(0.0, pre))


@pytest.mark.parametrize("beta_pre,no_norm", list(itertools.product([False, True], repeat=2)))
def test_t1_step(beta_pre, no_norm):
    x = _inputs(1, 61 + 2 * beta_pre + no_norm, beta_pre)
    if no_norm:
        x["q"] = (x["q"].float() / math.sqrt(K)).to(torch.bfloat16)
        x["k"] = (x["k"].float() / math.sqrt(K)).to(torch.bfloat16)
    out, fin = _run(x, beta_pre, no_norm)
    alpha = _alpha(x, 0)
    braw = float(x["beta"][0, 0, 0].float())
    b = braw if beta_pre else 1.0 / (1.0 + math.exp(-braw))
    kk, qq = as_f64(x["k"][0, 0, 0]), as_f64(x["q"][0, 0, 0])
    kh, qh = (kk, qq) if no_norm else (l2n(kk), l2n(qq))
    vv = as_f64(x["v"][0, 0, 0])
    S = alpha[:, None] * as_f64(x["initial_state"][0, 0]).T
    S = S + b * np.outer(kh, vv - S.T @ kh)
    np.testing.assert_allclose(fin[0, 0], S.T, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(out[0, 0], float(np.float32(x["scale"])) * S.T @ qh, rtol=1e-11, atol=1e-14)


def test_half_decay_at_zero_preactivation():
    # A_log = 0 and g + dt_bias = 0: ghat = -softplus(0) = -ln 2, so alpha = 1/2 on every channel
    x = _inputs(1, 62, beta_pre=True)
    x["A_log"] = torch.zeros(1)
    x["dt_bias"] = torch.zeros(1, K)
    x["g"] = torch.zeros(1, 1, 1, K, dtype=torch.bfloat16)
    x["beta"] = torch.zeros(1, 1, 1, dtype=torch.bfloat16)     # no update: the state is only decayed
    out, fin = _run(x, beta_pre=True)
    np.testing.assert_allclose(fin[0, 0], 0.5 * as_f64(x["initial_state"][0, 0]), rtol=1e-15, atol=0)


def test_decay_only_run_with_large_preactivations():
    # beta = 0 given directly: the state after T tokens is Diag(exp(sum ghat)) S0; g around +6 gives
    # a decay of about exp(-6 exp(A_log)) per token, well past the safe gate's lower bound of -5
    T = 6
    x = _inputs(T, 63, beta_pre=True, g_shift=6.0)
    x["beta"] = torch.zeros(1, T, 1, dtype=torch.bfloat16)
    out, fin = _run(x, beta_pre=True)
    decay = np.prod([_alpha(x, t) for t in range(T)], axis=0)
    S0 = as_f64(x["initial_state"][0, 0]).T
    assert decay.max() < math.exp(-5.0 * T * 0.3)
    np.testing.assert_allclose(fin[0, 0], (decay[:, None] * S0).T, rtol=1e-12, atol=1e-300)
    qh = l2n(as_f64(x["q"][0, T - 1, 0]))
    np.testing.assert_allclose(out[T - 1, 0], float(np.float32(x["scale"])) * (decay[:, None] * S0).T @ qh,
                               rtol=1e-11, atol=1e-300)


def test_lower_bound_is_not_used():
    x = _inputs(3, 64)
    ref_out, ref_fin = _run(x)
    x["lower_bound"] = float("nan")
    out, fin = _run(x)
    np.testing.assert_array_equal(out, ref_out)
    np.testing.assert_array_equal(fin, ref_fin)


def test_differs_from_the_safe_gate():
    x = _inputs(3, 65)
    a_out, a_fin = _run(x, safe_gate=False)
    b_out, b_fin = _run(x, safe_gate=True)
    assert np.abs(a_fin - b_fin).max() > 1e-6


def test_needs_the_in_kernel_gate():
    x = _inputs(1, 66)
    with pytest.raises(ValueError):
        oracle.kda_forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["A_log"], x["dt_bias"],
                           x["lower_bound"], x["initial_state"], use_gate_in_kernel=False, safe_gate=False)
