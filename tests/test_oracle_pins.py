"""Pins for the CPU oracle: checks against what FlashKDA's README and the mathematics fix.

FlashKDA's README and articles print no worked numbers, so every pin is a closed form, an
invariant, a special case with an exactly known answer, or an independent
derivation (the 16-token chunked form) that must agree with the token
recurrence.  Each pin is chosen so that a plausible slip in the oracle -- a
wrong sign, a dropped term, a transposed state, the wrong exponent base, the
update and the decay swapped -- breaks at least one of them.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import chunked_np, token_np
from gated_delta_rule_51_gb300 import inputs as I
from tests.oracle_helpers import as_f64, bf16, l2n, rel_fro

K = V = 128


def run(x, **kw):
    return oracle.kda_forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["A_log"],
                              x["dt_bias"], x["lower_bound"], x.get("initial_state"),
                              x.get("cu_seqlens"), **kw)


def rand_inputs(B, T, H, seed, lb=-5.0, init=True, k_dim=K, v_dim=V, cu=None, scale=None):
    gen = torch.Generator().manual_seed(seed)
    N = B if cu is None else len(cu) - 1
    x = dict(
        q=torch.randn(B, T, H, k_dim, generator=gen).to(torch.bfloat16),
        k=torch.randn(B, T, H, k_dim, generator=gen).to(torch.bfloat16),
        v=torch.randn(B, T, H, v_dim, generator=gen).to(torch.bfloat16),
        g=torch.randn(B, T, H, k_dim, generator=gen).to(torch.bfloat16),
        beta=torch.randn(B, T, H, generator=gen).to(torch.bfloat16),
        A_log=torch.rand(H, generator=gen) * 2 - 1,
        dt_bias=torch.randn(H, k_dim, generator=gen) * 0.1,
        scale=(1.0 / math.sqrt(k_dim)) if scale is None else scale,
        lower_bound=lb,
        initial_state=(torch.randn(N, H, v_dim, k_dim, generator=gen, dtype=torch.float64) * 0.02
                       if init else None),
        cu_seqlens=None if cu is None else torch.tensor(cu, dtype=torch.int64),
    )
    return x


# ---------------------------------------------------------------------------
# T = 1 closed form (README Kernel API: beta is a logit with the sigmoid applied
# internally; state layout [B,H,V,K]; out = scale * S^T q with q, k L2-normalised)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("beta_logit", [0.0, 1.5, -2.25])
def test_t1_closed_form_from_zero_state(beta_logit):
    x = rand_inputs(1, 1, 2, seed=11, init=False)
    x["beta"] = torch.full((1, 1, 2), beta_logit).to(torch.bfloat16)
    out, fin = run(x)
    b = 1.0 / (1.0 + math.exp(-float(torch.tensor(beta_logit).to(torch.bfloat16))))
    for h in range(2):
        qh = l2n(as_f64(x["q"][0, 0, h]))
        kh = l2n(as_f64(x["k"][0, 0, h]))
        vv = as_f64(x["v"][0, 0, h])
        scale = float(np.float32(x["scale"]))
        # S_1 = b kh v^T (K x V); stored transposed: fin[v, c] = b * v[v] * kh[c]
        np.testing.assert_allclose(fin[0, h], b * np.outer(vv, kh), rtol=1e-13, atol=1e-15)
        # o = scale * S_1^T qh = scale * b * (kh . qh) * v
        np.testing.assert_allclose(out[0, h], scale * b * np.dot(kh, qh) * vv, rtol=1e-12,
                                   atol=1e-15)
    if beta_logit == 0.0:
        assert b == 0.5


def test_t1_with_initial_state_and_unit_decay():
    """lower_bound = 0 makes every decay exactly 1 (README: range -5.0 .. 0)."""
    x = rand_inputs(1, 1, 1, seed=12, lb=0.0)
    out, fin = run(x)
    S0 = as_f64(x["initial_state"][0, 0]).T          # K x V
    kh = l2n(as_f64(x["k"][0, 0, 0]))
    qh = l2n(as_f64(x["q"][0, 0, 0]))
    vv = as_f64(x["v"][0, 0, 0])
    b = 1.0 / (1.0 + math.exp(-float(x["beta"][0, 0, 0])))
    # rank-one correction of the prediction error (v - S0^T kh)
    S1 = S0 + b * np.outer(kh, vv - S0.T @ kh)
    np.testing.assert_allclose(fin[0, 0], S1.T, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(out[0, 0], float(np.float32(x["scale"])) * S1.T @ qh, rtol=1e-11,
                               atol=1e-14)


# ---------------------------------------------------------------------------
# Gate: special inputs with exactly known decays.  With beta-logit = -64 the
# delta update is suppressed (sigmoid(-64) ~ 1.6e-28) and the final state is
# Diag(prod alpha) S0, so the decay can be read off channel by channel.
# ---------------------------------------------------------------------------
def _decay_only_inputs(T, A_log, dt_bias, g, lb):
    x = rand_inputs(1, T, 1, seed=13, lb=lb)
    x["beta"] = torch.full((1, T, 1), -64.0).to(torch.bfloat16)
    x["A_log"] = torch.tensor([A_log], dtype=torch.float32)
    x["dt_bias"] = torch.as_tensor(np.asarray(dt_bias, np.float32)).reshape(1, K)
    x["g"] = torch.as_tensor(np.asarray(g, np.float32)).reshape(1, T, 1, K).to(torch.bfloat16)
    return x


@pytest.mark.parametrize("lb", [-5.0, -2.0, -1.0, -0.5])
def test_gate_zero_preactivation_gives_half_lower_bound(lb):
    # g + dt_bias = 0 exactly => sigmoid(0) = 1/2 => ghat = lb/2, for any A_log
    rng = np.random.default_rng(0)
    dt = as_f64(bf16(rng.normal(0, 0.5, K)))         # bf16-representable biases
    T = 3
    x = _decay_only_inputs(T, 0.37, dt, np.tile(-dt, (T, 1)), lb)
    _, fin = run(x)
    S0 = as_f64(x["initial_state"][0, 0])
    expected = S0 * math.exp(T * lb / 2.0)         # natural exponent, not base 2
    np.testing.assert_allclose(fin[0, 0], expected, rtol=1e-12, atol=1e-30)


def test_gate_uses_exp_of_A_log_and_adds_dt_bias():
    # A_log = 0 (rate 1): preactivation g + dt_bias = ln 3 => sigmoid = 3/4
    # A_log = ln 2 (rate 2): preactivation (ln 3)/2 gives the same decay
    lb = -2.0
    ln3 = math.log(3.0)
    half = np.full(K, 0.5, np.float32)               # exact in bf16
    for A_log, pre in ((0.0, ln3), (math.log(2.0), ln3 / 2)):
        g_val = np.float32(pre) - half               # g = pre - dt_bias (bf16 rounding below)
        g_b = as_f64(bf16(np.tile(g_val, (1, 1))))[0]
        x = _decay_only_inputs(1, A_log, half, g_b, lb)
        _, fin = run(x)
        rate = math.exp(float(np.float32(A_log)))
        sig = 1.0 / (1.0 + np.exp(-rate * (g_b + 0.5)))
        S0 = as_f64(x["initial_state"][0, 0])
        np.testing.assert_allclose(fin[0, 0], S0 * np.exp(lb * sig)[None, :], rtol=1e-12)
        # and the decay is close to exp(3 lb / 4) (bf16 rounding of g only)
        np.testing.assert_allclose(sig, 0.75, atol=3e-3)


def test_gate_channel_and_sign_conventions():
    # channel c gets its own bias: dt_bias[c] = +-1 with g = 0 => decays differ by sign
    lb = -3.0
    dt = np.where(np.arange(K) % 2 == 0, 1.0, -1.0)
    x = _decay_only_inputs(2, 0.0, dt, np.zeros((2, K)), lb)
    _, fin = run(x)
    S0 = as_f64(x["initial_state"][0, 0])
    s = 1.0 / (1.0 + np.exp(-dt))                    # sigmoid(+1) / sigmoid(-1)
    np.testing.assert_allclose(fin[0, 0], S0 * np.exp(2 * lb * s)[None, :], rtol=1e-12)
    assert s[0] > 0.5 > s[1]                         # larger bias => stronger decay


# ---------------------------------------------------------------------------
# Delta-rule invariant: with beta = 1 and a unit key the update makes the
# state reproduce the value exactly: kh_t^T S_t = v_t^T (decay applied first).
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("lb", [0.0, -5.0])
def test_delta_rule_invariant(lb):
    T = 6
    x = rand_inputs(1, T, 2, seed=14, lb=lb)
    x["beta"] = torch.full((1, T, 2), 64.0).to(torch.bfloat16)   # sigmoid(64) = 1 - 1.6e-28
    for t in range(1, T + 1):
        xt = dict(x)
        for name in ("q", "k", "v", "g", "beta"):
            xt[name] = x[name][:, :t].contiguous()
        _, fin = run(xt)
        for h in range(2):
            kk = as_f64(x["k"][0, t - 1, h])
            kh = l2n(kk)
            vv = as_f64(x["v"][0, t - 1, h])
            pred = fin[0, h] @ kh                     # (S_t^T kh)[v] = sum_c fin[v,c] kh[c]
            # |kh|^2 = 1 - 1e-6/|k|^2, so the invariant holds to ~1e-8 relative
            tol = 2e-6 / float(kk @ kk) * np.abs(vv).max() + 1e-12
            np.testing.assert_allclose(pred, vv, atol=tol + 1e-9 * np.abs(vv).max())


def test_update_then_decay_would_break_invariant():
    """Sanity of the invariant pin itself: the reversed order does not satisfy it."""
    x = rand_inputs(1, 2, 1, seed=15, lb=-5.0)
    _, fin = run(x)
    kh = l2n(as_f64(x["k"][0, 1, 0]))
    g = as_f64(x["g"][0, 1, 0])
    alpha = np.exp(token_np.gate_log_decay(g, as_f64(x["dt_bias"][0]), float(x["A_log"][0]), -5.0))
    S = fin[0, 0].T
    # decaying after the update moves kh^T S away from v
    assert np.abs((np.diag(alpha) @ S).T @ kh - S.T @ kh).max() > 1e-3


# ---------------------------------------------------------------------------
# State carry, varlen batching, batch rows (README: initial/final state, cu_seqlens)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("t0", [1, 16, 37])
def test_split_and_carry_equals_one_call(t0):
    T = 70
    x = rand_inputs(1, T, 2, seed=16)
    out, fin = run(x)
    a = dict(x)
    b = dict(x)
    for name in ("q", "k", "v", "g", "beta"):
        a[name] = x[name][:, :t0].contiguous()
        b[name] = x[name][:, t0:].contiguous()
    out_a, fin_a = run(a)
    b["initial_state"] = torch.from_numpy(fin_a)
    out_b, fin_b = run(b)
    np.testing.assert_allclose(np.concatenate([out_a, out_b]), out, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(fin_b, fin, rtol=1e-12, atol=1e-15)


def test_varlen_equals_separate_calls():
    lens = [5, 16, 1, 40, 17]
    cu = np.concatenate([[0], np.cumsum(lens)])
    x = rand_inputs(1, int(cu[-1]), 2, seed=17, cu=cu)
    out, fin = run(x)
    for n, L in enumerate(lens):
        s = dict(x)
        for name in ("q", "k", "v", "g", "beta"):
            s[name] = x[name][:, cu[n]:cu[n + 1]].contiguous()
        s["initial_state"] = x["initial_state"][n:n + 1]
        s["cu_seqlens"] = None
        o_n, f_n = run(s)
        np.testing.assert_allclose(out[cu[n]:cu[n + 1]], o_n, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(fin[n], f_n[0], rtol=1e-13, atol=1e-15)


def test_batch_rows_equal_varlen_with_equal_lengths():
    B, T = 3, 21
    x = rand_inputs(B, T, 2, seed=18)
    out, fin = run(x)
    y = dict(x)
    for name in ("q", "k", "v", "g", "beta"):
        y[name] = x[name].reshape(1, B * T, *x[name].shape[2:]).contiguous()
    y["cu_seqlens"] = torch.arange(0, B * T + 1, T, dtype=torch.int64)
    out2, fin2 = run(y)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(fin, fin2)


def test_zero_length_sequence_keeps_state():
    cu = [0, 7, 7, 12]
    x = rand_inputs(1, 12, 1, seed=19, cu=cu)
    out, fin = run(x)
    np.testing.assert_array_equal(fin[1], as_f64(x["initial_state"][1]))
    assert np.abs(fin[0] - as_f64(x["initial_state"][0])).max() > 1e-3


# ---------------------------------------------------------------------------
# The chunked (WY/UT) form -- FlashKDA's 16-token chunks with a Neumann inverse
# -- must reach the token recurrence's result (exact method).
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("chunk", [1, 4, 16, 64])
@pytest.mark.parametrize("inverse", ["neumann", "substitution"])
def test_chunked_form_equals_token_recurrence(chunk, inverse):
    lens = [40, 16, 3, 33]
    cu = np.concatenate([[0], np.cumsum(lens)])
    x = rand_inputs(1, int(cu[-1]), 2, seed=20, cu=cu, k_dim=32, v_dim=24)
    out, fin = run(x)
    f64 = as_f64
    o2, f2 = chunked_np.forward(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["g"]),
                                f64(x["beta"]), float(np.float32(x["scale"])), f64(x["A_log"]),
                                f64(x["dt_bias"]), float(np.float32(x["lower_bound"])),
                                f64(x["initial_state"]), cu_seqlens=cu, chunk=chunk,
                                inverse=inverse)
    assert rel_fro(o2.reshape(out.shape), out) < 1e-12
    assert rel_fro(f2, fin) < 1e-12


def test_chunked_form_full_head_dim_lower_bound_extremes():
    for lb in (-5.0, 0.0):
        x = rand_inputs(1, 50, 1, seed=21, lb=lb)
        out, fin = run(x)
        f64 = as_f64
        o2, f2 = chunked_np.forward(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["g"]),
                                    f64(x["beta"]), float(np.float32(x["scale"])),
                                    f64(x["A_log"]), f64(x["dt_bias"]), lb,
                                    f64(x["initial_state"]))
        assert rel_fro(o2, out) < 1e-12 and rel_fro(f2, fin) < 1e-12


def test_neumann_product_is_the_inverse():
    rng = np.random.default_rng(3)
    for n in (2, 5, 16):
        A = np.tril(rng.normal(0, 0.7, (n, n)), -1)
        X1 = chunked_np.unit_lower_inverse_neumann(A)
        X2 = chunked_np.unit_lower_inverse_substitution(A)
        ref = np.linalg.inv(np.eye(n) + A)
        np.testing.assert_allclose(X1, ref, rtol=1e-10, atol=1e-10)
        np.testing.assert_allclose(X2, ref, rtol=1e-10, atol=1e-10)


# ---------------------------------------------------------------------------
# Structure: linearity in (v, S0), V-column independence, NumPy twin agreement
# ---------------------------------------------------------------------------
def test_joint_linearity_in_values_and_state():
    x = rand_inputs(1, 33, 1, seed=22)
    out, fin = run(x)
    y = dict(x)
    y["v"] = (x["v"].to(torch.float32) * 2).to(torch.bfloat16)     # exact doubling
    y["initial_state"] = x["initial_state"] * 2
    out2, fin2 = run(y)
    np.testing.assert_array_equal(out2, 2 * out)
    np.testing.assert_array_equal(fin2, 2 * fin)
    # additivity with values that add exactly in bf16 (multiples of 1/8 in [-4, 4])
    rng = np.random.default_rng(5)
    v1 = rng.integers(-16, 17, x["v"].shape) / 8.0
    v2 = rng.integers(-16, 17, x["v"].shape) / 8.0
    parts = []
    for vv, s0 in ((v1, x["initial_state"]), (v2, x["initial_state"] * 0.5),
                   (v1 + v2, x["initial_state"] * 1.5)):
        z = dict(x)
        z["v"] = bf16(vv)
        z["initial_state"] = s0
        parts.append(run(z))
    np.testing.assert_allclose(parts[0][0] + parts[1][0], parts[2][0], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(parts[0][1] + parts[1][1], parts[2][1], rtol=1e-11, atol=1e-13)


def test_value_columns_are_independent():
    x = rand_inputs(1, 30, 1, seed=23)
    out, fin = run(x)
    perm = np.random.default_rng(6).permutation(V)
    y = dict(x)
    y["v"] = x["v"][..., perm].contiguous()
    y["initial_state"] = x["initial_state"][:, :, perm, :].contiguous()
    out2, fin2 = run(y)
    np.testing.assert_allclose(out2, out[..., perm], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(fin2, fin[:, :, perm, :], rtol=1e-13, atol=1e-15)


def test_numpy_twin_agrees_small_dims():
    cu = [0, 3, 9, 10]
    x = rand_inputs(1, 10, 2, seed=24, cu=cu, k_dim=3, v_dim=4)
    out, fin = run(x)
    f64 = as_f64
    o2, f2 = token_np.forward(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["g"]),
                              f64(x["beta"]), float(np.float32(x["scale"])), f64(x["A_log"]),
                              f64(x["dt_bias"]), -5.0, f64(x["initial_state"]), cu_seqlens=cu)
    np.testing.assert_allclose(out, o2, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(fin, f2, rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------------------
# L2 normalisation reading (epsilon 1e-6 inside the square root) and zero vectors
# ---------------------------------------------------------------------------
def test_l2_norm_epsilon_and_zero_query():
    x = rand_inputs(1, 2, 1, seed=25, init=False)
    q = np.zeros((1, 2, 1, K), np.float32)
    q[0, 1, 0, 3] = 2.0 ** -10                         # |q|^2 = 2^-20 ~ 9.5e-7, comparable to eps
    x["q"] = bf16(q)
    out, fin = run(x)
    assert np.all(out[0] == 0.0)                       # zero query => zero output
    S = fin[0, 0].T
    qh = np.zeros(K)
    qh[3] = 2.0 ** -10 / math.sqrt(2.0 ** -20 + 1e-6)
    np.testing.assert_allclose(out[1, 0], float(np.float32(x["scale"])) * S.T @ qh, rtol=1e-12)


def test_out_rows_sampling_matches_full_run():
    x = rand_inputs(2, 19, 2, seed=26)
    out, fin = run(x)
    rows = [0, 5, 18, 19, 37]
    o2, f2 = run(x, out_rows=rows)
    np.testing.assert_array_equal(o2, out[rows])
    np.testing.assert_array_equal(f2, fin)


def test_named_workloads_follow_their_recipes():
    ws = I.named_workloads()
    w2 = ws["varlen_T32768_N8_H32"]
    assert len(w2.seq_lens) == 8 and sum(w2.seq_lens) == 32768
    assert all(1 <= L <= 8192 for L in w2.seq_lens)
    for total in I.SWEEP_TOTALS:
        for H in I.SWEEP_HEADS:
            w = ws[f"sweep_T{total}_H{H}"]
            assert sum(w.seq_lens) == total
            assert all(64 <= L <= 16384 for L in w.seq_lens)
    x = I.make_inputs(ws["tiny_B1_T64_H1"])
    assert x["q"].shape == (1, 64, 1, 128) and x["q"].dtype == torch.bfloat16
    assert x["beta"].shape == (1, 64, 1) and x["A_log"].dtype == torch.float32
    assert float(x["A_log"].min()) >= -1.0 and float(x["A_log"].max()) <= 1.0
