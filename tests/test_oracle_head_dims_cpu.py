"""The oracle at K = 64, V = 64 and V = 256 against itself at K = V = 128.

The GPU tests compare the K = 64 and V = 64 paths with the oracle at those sizes; this pins
that the oracle's own K = 64 / V = 64 results are the K = V = 128 recurrence with the
extra key channels (q = k = g = dt_bias = 0, initial state 0 there) or value columns
(v = 0, initial state 0 there) padded in: the padded state columns stay zero and add
nothing, so the results agree to fp64 rounding.  The forward oracle (bf16 inputs) and the
gradient oracle (fp64 inputs) are both checked.  V = 256 is two independent V = 128
problems that share q, k, g and beta (the value columns of the state never mix).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle


def _inputs(seed, K, V, lens):
    g = torch.Generator().manual_seed(seed)
    T, H = sum(lens), 2
    bf = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)
    x = dict(q=bf(1, T, H, K), k=bf(1, T, H, K), v=bf(1, T, H, V), g=bf(1, T, H, K), beta=bf(1, T, H),
             A_log=torch.rand(H, generator=g) * 2 - 1, dt_bias=0.1 * torch.randn(H, K, generator=g),
             s0=0.02 * torch.randn(len(lens), H, V, K, generator=g))
    x["cu"] = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    return x


def _pad(x, K2, V2):
    K, V = x["q"].shape[-1], x["v"].shape[-1]
    y = dict(x)
    for n in ("q", "k", "g"):
        y[n] = torch.nn.functional.pad(x[n], (0, K2 - K))
    y["v"] = torch.nn.functional.pad(x["v"], (0, V2 - V))
    y["dt_bias"] = torch.nn.functional.pad(x["dt_bias"], (0, K2 - K))
    y["s0"] = torch.nn.functional.pad(x["s0"], (0, K2 - K, 0, V2 - V))
    return y


@pytest.mark.parametrize("K,V", [(64, 128), (128, 64), (64, 64)])
def test_forward_oracle_at_small_head_dims_equals_the_padded_full_size(K, V):
    x = _inputs(11 + K + V, K, V, [5, 0, 37])
    y = _pad(x, 128, 128)
    scale = K ** -0.5
    o1, f1 = oracle.kda_forward(x["q"], x["k"], x["v"], x["g"], x["beta"], scale, x["A_log"], x["dt_bias"], -3.0,
                                x["s0"], x["cu"])
    o2, f2 = oracle.kda_forward(y["q"], y["k"], y["v"], y["g"], y["beta"], scale, y["A_log"], y["dt_bias"], -3.0,
                                y["s0"], y["cu"])
    np.testing.assert_allclose(o1, o2[..., :V], rtol=0, atol=1e-13)
    np.testing.assert_allclose(f1, f2[:, :, :V, :K], rtol=0, atol=1e-13)
    assert np.all(f2[:, :, V:, :] == 0) and np.all(f2[:, :, :, K:] == 0)


@pytest.mark.parametrize("K,V", [(64, 128), (128, 64)])
def test_gradient_oracle_at_small_head_dims_equals_the_padded_full_size(K, V):
    x = _inputs(21 + K + V, K, V, [9, 14])
    y = _pad(x, 128, 128)
    g = torch.Generator().manual_seed(5)
    dout = torch.randn(1, 23, 2, V, generator=g).double().numpy()
    dfin = torch.randn(2, 2, V, K, generator=g).double().numpy()
    d = lambda t: t.double().numpy() if isinstance(t, torch.Tensor) else t
    r1 = oracle.kda_backward(*(d(x[n]) for n in ("q", "k", "v", "g", "beta")), K ** -0.5, d(x["A_log"]),
                             d(x["dt_bias"]), -3.0, dout, d(x["s0"]), dfin, x["cu"])
    dout2 = np.pad(dout, ((0, 0), (0, 0), (0, 0), (0, 128 - V)))
    dfin2 = np.pad(dfin, ((0, 0), (0, 0), (0, 128 - V), (0, 128 - K)))
    r2 = oracle.kda_backward(*(d(y[n]) for n in ("q", "k", "v", "g", "beta")), K ** -0.5, d(y["A_log"]),
                             d(y["dt_bias"]), -3.0, dout2, d(y["s0"]), dfin2, y["cu"])
    tol = lambda a: 1e-12 * max(1.0, np.abs(a).max())
    for n, sl in (("dq", (..., slice(0, K))), ("dk", (..., slice(0, K))), ("dg", (..., slice(0, K))),
                  ("dv", (..., slice(0, V))), ("dbeta", (...,)), ("dh0", (..., slice(0, V), slice(0, K))),
                  ("dA_log", (...,)), ("ddt_bias", (..., slice(0, K)))):
        np.testing.assert_allclose(r1[n], r2[n][sl], rtol=0, atol=tol(r1[n]), err_msg=n)


def test_forward_oracle_at_v256_equals_two_independent_v128_halves():
    """Value columns evolve independently: V = 256 is two V = 128 problems sharing q, k, g, beta."""
    x = _inputs(31, 128, 256, [12, 29])
    scale = 128 ** -0.5
    o, f = oracle.kda_forward(x["q"], x["k"], x["v"], x["g"], x["beta"], scale, x["A_log"], x["dt_bias"], -2.0,
                              x["s0"], x["cu"])
    for half in (slice(0, 128), slice(128, 256)):
        oh, fh = oracle.kda_forward(x["q"], x["k"], x["v"][..., half].contiguous(), x["g"], x["beta"], scale,
                                    x["A_log"], x["dt_bias"], -2.0, x["s0"][:, :, half].contiguous(), x["cu"])
        np.testing.assert_allclose(o[..., half], oh, rtol=0, atol=1e-13)
        np.testing.assert_allclose(f[:, :, half], fh, rtol=0, atol=1e-13)
