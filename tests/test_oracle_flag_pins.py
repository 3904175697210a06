"""Pins for the oracle's three switches, named after the flags of the chunk_kda
call in FlashKDA's README (chunk_kda: use_gate_in_kernel, use_beta_sigmoid_in_kernel,
use_qk_l2norm_in_kernel).  When a flag is off, that step was done by the caller:
g holds the natural-log decay itself, beta holds beta itself, q and k are used as
given.  Each pin recomputes the T = 1 step (or a decay-only run) in numpy from
the definitions, for every combination of the flags."""
from __future__ import annotations

import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from tests.oracle_helpers import as_f64, l2n

K = V = 128


def _inputs(T, seed, gate_pre, beta_pre, no_norm):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(1, T, 1, K, generator=gen)
    k = torch.randn(1, T, 1, K, generator=gen)
    if no_norm:   # unnormalised keys of moderate norm keep the update contractive
        q, k = q / math.sqrt(K), k / math.sqrt(K)
    g = (-5.0 * torch.rand(1, T, 1, K, generator=gen)) if gate_pre else torch.randn(1, T, 1, K, generator=gen)
    beta = torch.rand(1, T, 1, generator=gen) if beta_pre else torch.randn(1, T, 1, generator=gen)
    return dict(q=q.to(torch.bfloat16), k=k.to(torch.bfloat16),
                v=torch.randn(1, T, 1, V, generator=gen).to(torch.bfloat16), g=g.to(torch.bfloat16),
                beta=beta.to(torch.bfloat16), A_log=torch.rand(1, generator=gen) * 2 - 1,
                dt_bias=torch.randn(1, K, generator=gen) * 0.1, scale=1.0 / math.sqrt(K), lower_bound=-3.0,
                initial_state=torch.randn(1, 1, V, K, generator=gen, dtype=torch.float64) * 0.02)


def _run(x, gate_pre, beta_pre, no_norm, **kw):
    return oracle.kda_forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["A_log"], x["dt_bias"],
                              x["lower_bound"], x["initial_state"], use_gate_in_kernel=not gate_pre,
                              use_beta_sigmoid_in_kernel=not beta_pre, use_qk_l2norm_in_kernel=not no_norm, **kw)


@pytest.mark.parametrize("gate_pre,beta_pre,no_norm", list(itertools.product([False, True], repeat=3)))
def test_t1_step_for_every_flag_combination(gate_pre, beta_pre, no_norm):
    x = _inputs(1, 31 + 4 * gate_pre + 2 * beta_pre + no_norm, gate_pre, beta_pre, no_norm)
    out, fin = _run(x, gate_pre, beta_pre, no_norm)
    g = as_f64(x["g"][0, 0, 0])
    if gate_pre:
        alpha = np.exp(g)
    else:
        rate = math.exp(float(x["A_log"][0]))
        pre = rate * (g + x["dt_bias"][0].double().numpy())
        alpha = np.exp(float(np.float32(x["lower_bound"])) / (1.0 + np.exp(-pre)))
    braw = float(x["beta"][0, 0, 0].float())
    b = braw if beta_pre else 1.0 / (1.0 + math.exp(-braw))
    kk, qq = as_f64(x["k"][0, 0, 0]), as_f64(x["q"][0, 0, 0])
    kh, qh = (kk, qq) if no_norm else (l2n(kk), l2n(qq))
    vv = as_f64(x["v"][0, 0, 0])
    S = alpha[:, None] * as_f64(x["initial_state"][0, 0]).T          # decay, K x V
    S = S + b * np.outer(kh, vv - S.T @ kh)                          # delta update
    np.testing.assert_allclose(fin[0, 0], S.T, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(out[0, 0], float(np.float32(x["scale"])) * S.T @ qh, rtol=1e-11, atol=1e-14)


def test_preactivated_gate_ignores_the_gate_parameters():
    x = _inputs(3, 41, True, False, False)
    ref_out, ref_fin = _run(x, True, False, False)
    x["A_log"] = torch.full((1,), float("nan"))
    x["dt_bias"] = torch.full((1, K), float("nan"))
    x["lower_bound"] = 123.0
    out, fin = _run(x, True, False, False)
    np.testing.assert_array_equal(out, ref_out)
    np.testing.assert_array_equal(fin, ref_fin)


def test_preactivated_gate_decay_only_run():
    # beta = 0 given directly: no update, so the state after T tokens is Diag(exp(sum g)) S0
    T = 5
    x = _inputs(T, 42, True, True, False)
    x["beta"] = torch.zeros(1, T, 1, dtype=torch.bfloat16)
    out, fin = _run(x, True, True, False)
    gsum = as_f64(x["g"][0, :, 0]).sum(axis=0)
    S0 = as_f64(x["initial_state"][0, 0]).T
    np.testing.assert_allclose(fin[0, 0], (np.exp(gsum)[:, None] * S0).T, rtol=1e-12, atol=1e-16)
    # the output of the last token reads the decayed state
    qh = l2n(as_f64(x["q"][0, T - 1, 0]))
    np.testing.assert_allclose(out[T - 1, 0], float(np.float32(x["scale"])) * (np.exp(gsum)[:, None] * S0).T @ qh,
                               rtol=1e-11, atol=1e-16)
