"""GPU parity of the chunked tensor-core backward (kda_bwd's default for the gate with a lower
bound) with the fp64 oracle's gradient (oracle/kda_oracle_bwd.c, pinned by finite
differences in test_oracle_backward_pins.py), through the C ABI.

Bounds (stated, with their derivation, before the kernels were written): the chunked form
rounds the state copies that feed its state-sized GEMMs, the operands W, scale Q_p and K_d of
those GEMMs, and the stored S0 and dS1 to bf16 (unit roundoff 2^-9); Tm, P, Vn and dVn are
split into bf16 hi + lo.  Two to four such roundings lie on each path to a gradient entry, so
the relative Frobenius error of a gradient tensor is expected near 1.6e-3..2.3e-3, a small
multiple of that where the gate hardly decays; a CPU emulation of exactly these rounding
points measured at most 1.8e-3 at lower_bound <= -1 and 3.8e-3 at lower_bound 0.
- dq, dk, dv, dg, dbeta, dh0, ddt_bias: relative Frobenius error <= 1e-2;
- dA_log, a sum over every token and channel of terms of both signs that can nearly cancel:
  |error| <= 1e-3 * sum_{t,c} |dg_{t,c} (g_{t,c} + dt_bias_c)|, the terms' absolute sum
  (the emulation: 8.5e-6 of it at lower_bound -5).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from tests.gpu_helpers import _report, random_case, rel_fro
from tests.test_bwd_gpu import NAMES, _grads_in, _gpu, _oracle

pytestmark = pytest.mark.gpu

BOUND = 1e-2
DA_BOUND = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_51_gb300 import kda

    kda.load_library()


def _da_scale(x, ref, heads=None):
    """Per head, the absolute sum of dA_log's terms dg (g + dt_bias) from the oracle's dg."""
    hs = slice(None) if heads is None else list(heads)
    g = x["g"].detach().cpu().double().numpy()[:, :, hs]
    dtb = x["dt_bias"].detach().cpu().double().numpy()[hs]
    return np.abs(ref["dg"] * (g + dtb[None, None])).sum(axis=(0, 1, 3))


def _compare(gpu, ref, x, label, heads=None):
    for n in NAMES:
        g = gpu[n].detach().cpu().double().numpy()
        if heads is not None:
            g = g[:, :, list(heads)] if n in ("dq", "dk", "dv", "dg", "dbeta") else (
                g[:, list(heads)] if n == "dh0" else g[list(heads)])
        assert np.all(np.isfinite(g)), f"{label}: non-finite {n}"
        if n == "dA_log":
            scale = _da_scale(x, ref, heads)
            e = float(np.max(np.abs(g - ref[n]) / np.maximum(scale, 1e-30)))
            _report(label, "bwd_chunked_dA_log_err_over_terms", e)
            assert e <= DA_BOUND, f"{label}: dA_log error {e:.3e} of its terms' absolute sum > {DA_BOUND}"
            continue
        e = rel_fro(g, ref[n])
        _report(label, f"bwd_chunked_{n}_rel_fro", e)
        assert e <= BOUND, f"{label}: {n} rel-Fro {e:.3e} > {BOUND}"


@pytest.mark.parametrize("lens,init_dtype,dfin", [
    ([100, 7, 0, 193], torch.float32, True),   # partial chunks, a one-chunk and an empty sequence
    ([300], torch.bfloat16, False),
    ([5, 16, 31, 8], None, True),
    ([16, 32, 48], torch.float32, True),        # whole chunks only
])
def test_chunked_backward_varlen_matches_oracle(lens, init_dtype, dfin):
    x = random_case(1, sum(lens), 2, seed=1961 + len(lens), lens=lens, init_dtype=init_dtype)
    dout, dfinal = _grads_in(x, 1962, dfin)
    _compare(_gpu(x, dout, dfinal, recurrent=False), _oracle(x, dout, dfinal), x, f"bwd chunked varlen {lens}")


@pytest.mark.parametrize("lb", [-5.0, -2.0, -0.3, 0.0])
def test_chunked_backward_lower_bounds(lb):
    # lower_bound 0 is the weakest decay the gate admits (no decay at all): the rounding of the
    # state copies is then never forgotten between chunks
    x = random_case(2, 700, 2, seed=1963, lb=lb)
    dout, dfinal = _grads_in(x, 1964)
    _compare(_gpu(x, dout, dfinal, recurrent=False), _oracle(x, dout, dfinal), x, f"bwd chunked lb={lb}")


@pytest.mark.parametrize("switch", ["beta_given", "no_l2norm"])
def test_chunked_backward_switches_match_oracle(switch):
    x = random_case(1, 150, 2, seed=1965, lens=[60, 90])
    kw = {"beta_given": dict(use_beta_sigmoid_in_kernel=False),
          "no_l2norm": dict(use_qk_l2norm_in_kernel=False)}[switch]
    if switch == "beta_given":
        x["beta"] = torch.sigmoid(x["beta"].float()).to(torch.bfloat16)
    if switch == "no_l2norm":
        # raw q and k of norm about 1, as a caller that normalised them would pass
        x["q"] = (x["q"].float() / 11.3).to(torch.bfloat16)
        x["k"] = (x["k"].float() / 11.3).to(torch.bfloat16)
    dout, dfinal = _grads_in(x, 1966)
    r = _gpu(x, dout, dfinal, recurrent=False, **kw)
    _compare(r, _oracle(x, dout, dfinal, **kw), x, f"bwd chunked {switch}")


def test_chunked_backward_fixed_workload_sampled_heads():
    """The fixed workload's full size (B=2, T=4096, H=16, fp32 states); heads are independent,
    so the oracle runs three of them and every gradient of those heads is compared."""
    from gated_delta_rule_51_gb300 import inputs as I

    w = I.fixed_batch_workload()
    x = I.make_inputs(w, device="cuda")
    dout, dfinal = _grads_in(x, 1969)
    r = _gpu(x, dout, dfinal, recurrent=False)
    heads = (0, 7, 15)
    _compare(r, _oracle(x, dout, dfinal, heads=heads), x, "bwd chunked fixed workload heads 0,7,15", heads=heads)


def test_chunked_backward_two_parts_at_the_limit():
    """kda_bwd cuts each sequence of two or more chunks in two while the four runs per (sequence,
    head) fit one wave of two CTAs per SM; this case sits at that limit (SMs / 2 chains)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n_seq = sms // 4   # chains = 2 n_seq <= SMs / 2
    assert 4 * 2 * n_seq <= 2 * sms
    gen = np.random.default_rng(1980)
    lens = [int(x) for x in gen.integers(20, 120, size=n_seq)]
    x = random_case(1, sum(lens), 2, seed=1981, lens=lens)
    dout, dfinal = _grads_in(x, 1982)
    _compare(_gpu(x, dout, dfinal, recurrent=False), _oracle(x, dout, dfinal), x, f"bwd chunked {2 * n_seq} chains")


def test_chunked_backward_many_chains_unsplit():
    """With many (sequence, head) chains kda_bwd keeps every sequence whole."""
    gen = np.random.default_rng(1977)
    lens = [int(x) for x in gen.integers(1, 70, size=40)]
    x = random_case(1, sum(lens), 2, seed=1978, lens=lens)   # 80 chains: more than SMs / 2
    dout, dfinal = _grads_in(x, 1979)
    _compare(_gpu(x, dout, dfinal, recurrent=False), _oracle(x, dout, dfinal), x, "bwd chunked 80 chains")


def test_chunked_backward_without_dh0_or_parameter_gradients():
    from gated_delta_rule_51_gb300 import kda

    x = random_case(1, 90, 2, seed=1971, lens=[40, 50])
    dout, dfinal = _grads_in(x, 1972)
    full = _gpu(x, dout, dfinal, recurrent=False)
    r = {n: torch.full_like(full[n], 7.0) for n in ("dq", "dk", "dv", "dg", "dbeta")}
    kda.bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["A_log"], x["dt_bias"], x["lower_bound"],
            dout, initial_state=x["initial_state"], dfinal=dfinal, cu_seqlens=x["cu_seqlens"], out=r)
    torch.cuda.synchronize()
    for n in r:
        assert torch.equal(r[n], full[n]), n


def test_chunked_backward_is_deterministic():
    x = random_case(1, 400, 3, seed=1970, lens=[150, 250])
    dout, dfinal = _grads_in(x, 1973)
    a, b = _gpu(x, dout, dfinal, recurrent=False), _gpu(x, dout, dfinal, recurrent=False)
    for n in NAMES:
        assert torch.equal(a[n], b[n]), n


def test_chunked_backward_captured_in_a_cuda_graph_replays_identically():
    """A few chains: each sequence is cut in two and the correction launch starts beside the
    runs (a programmatic dependency, a graph edge once captured); each replay of the captured
    call gives the direct call's gradients bit for bit."""
    from gated_delta_rule_51_gb300 import kda

    x = random_case(1, 400, 2, seed=1983, lens=[150, 250])
    dout, dfinal = _grads_in(x, 1984)
    ref = _gpu(x, dout, dfinal, recurrent=False)
    ws = torch.empty(kda.bwd_workspace_size(kda.make_shape(1, 400, 2, 2)), dtype=torch.uint8, device="cuda")
    r = {n: torch.full_like(ref[n], float("nan")) for n in NAMES}
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            kda.bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["A_log"], x["dt_bias"],
                    x["lower_bound"], dout, initial_state=x["initial_state"], dfinal=dfinal,
                    cu_seqlens=x["cu_seqlens"], workspace=ws, out=r)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        for n in NAMES:
            r[n].fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for n in NAMES:
            assert torch.equal(r[n], ref[n]), n


def test_chunked_backward_malformed_cu_seqlens_is_flagged():
    from gated_delta_rule_51_gb300 import kda

    x = random_case(1, 64, 1, seed=1974, lens=[32, 32])
    x["cu_seqlens"] = torch.tensor([0, 40, 32], dtype=torch.int64, device="cuda")   # decreasing
    dout, dfinal = _grads_in(x, 1975)
    ws = torch.empty(kda.bwd_workspace_size(kda.make_shape(1, 64, 1, 2)), dtype=torch.uint8, device="cuda")
    _gpu(x, dout, dfinal, workspace=ws, recurrent=False)
    assert kda.check_device_error(ws) & 2
    x["cu_seqlens"] = torch.tensor([0, 32, 64], dtype=torch.int64, device="cuda")
    _gpu(x, dout, dfinal, workspace=ws, recurrent=False)
    assert kda.check_device_error(ws) == 0


def test_chunked_autograd_matches_the_oracle_gradient():
    """kda.kda_attention with its default (chunked) backward: gradients in the inputs' dtypes;
    the bf16 ones add their own rounding (2^-9 relative half-ulp) to the chunked bound."""
    from gated_delta_rule_51_gb300 import kda

    x = random_case(1, 200, 2, seed=1975, lens=[80, 120])
    leaves = {n: x[n].detach().clone().requires_grad_(True)
              for n in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state")}
    out, fin = kda.kda_attention(leaves["q"], leaves["k"], leaves["v"], leaves["g"], leaves["beta"], x["scale"],
                                 leaves["A_log"], leaves["dt_bias"], x["lower_bound"],
                                 initial_state=leaves["initial_state"], cu_seqlens=x["cu_seqlens"])
    gen = torch.Generator().manual_seed(1976)
    wo = torch.randn(out.shape, generator=gen).to(torch.bfloat16).cuda()
    wf = (0.1 * torch.randn(fin.shape, generator=gen)).cuda()
    ((out.float() * wo.float()).sum() + (fin * wf).sum()).backward()
    torch.cuda.synchronize()
    ref = _oracle(x, wo, wf)
    for n, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"),
                     ("dt_bias", "ddt_bias"), ("initial_state", "dh0")):
        gr = leaves[n].grad
        assert gr is not None and gr.dtype == x[n].dtype, n
        e = rel_fro(gr.detach().cpu().double().numpy(), ref[gname])
        _report("bwd chunked autograd", f"{gname}_rel_fro", e)
        assert e <= BOUND, f"{n}: rel-Fro {e:.3e} > {BOUND}"
    scale = _da_scale(x, ref)
    e = float(np.max(np.abs(leaves["A_log"].grad.detach().cpu().double().numpy() - ref["dA_log"]) / scale))
    assert e <= DA_BOUND, f"A_log: error {e:.3e} of its terms' absolute sum"
