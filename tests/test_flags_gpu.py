"""Parity of the GPU path with the oracle when the caller has done some steps.

The switches mirror the reference call's use_gate_in_kernel,
use_beta_sigmoid_in_kernel and use_qk_l2norm_in_kernel flags.  When off, g holds
the natural-log decay (drawn in [-5, 0], the range the in-kernel gate keeps to),
beta holds beta (drawn in (0, 1)), and q, k are used as given (drawn with norm
about 1).  Same bounds as the other parity tests.
"""
from __future__ import annotations

import itertools
import math

import pytest
import torch

from tests.gpu_helpers import check_out, check_state, random_case, run_oracle

pytestmark = pytest.mark.gpu


def _case(B, T, H, seed, gate_pre, beta_pre, no_norm, lens=None, init_dtype=torch.float32):
    x = random_case(B, T, H, seed=seed, lens=lens, lb=-5.0, init_dtype=init_dtype)
    gen = torch.Generator(device="cuda").manual_seed(seed + 1000)
    if gate_pre:
        x["g"] = (-5.0 * torch.rand(x["g"].shape, generator=gen, device="cuda")).to(torch.bfloat16)
    if beta_pre:
        x["beta"] = torch.rand(x["beta"].shape, generator=gen, device="cuda").to(torch.bfloat16)
    if no_norm:
        x["q"] = (x["q"].float() / math.sqrt(128)).to(torch.bfloat16)
        x["k"] = (x["k"].float() / math.sqrt(128)).to(torch.bfloat16)
    return x


def _kw(gate_pre, beta_pre, no_norm):
    return dict(use_gate_in_kernel=not gate_pre, use_beta_sigmoid_in_kernel=not beta_pre,
                use_qk_l2norm_in_kernel=not no_norm)


def _oracle(x, kw):
    import oracle
    from tests.gpu_helpers import to_cpu

    xc = to_cpu(x)
    return oracle.kda_forward(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["scale"], xc["A_log"],
                              xc["dt_bias"], xc["lower_bound"], xc.get("initial_state"), xc.get("cu_seqlens"), **kw)


@pytest.mark.parametrize("gate_pre,beta_pre,no_norm", list(itertools.product([False, True], repeat=3)))
def test_forward_flags_match_oracle(gate_pre, beta_pre, no_norm):
    from gated_delta_rule_51_gb300 import kda

    seed = 801 + 4 * gate_pre + 2 * beta_pre + no_norm
    x = _case(1, 700, 3, seed, gate_pre, beta_pre, no_norm, lens=[300, 17, 383])
    kw = _kw(gate_pre, beta_pre, no_norm)
    ref_out, ref_fin = _oracle(x, kw)
    out = torch.full_like(x["v"], float("nan"))
    fin = torch.full_like(x["initial_state"], float("nan"))
    a_log, dt = (None, None) if gate_pre else (x["A_log"], x["dt_bias"])
    kda.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], out, a_log, dt, x["lower_bound"],
            initial_state=x["initial_state"], final_state=fin, cu_seqlens=x["cu_seqlens"], **kw)
    torch.cuda.synchronize()
    label = f"flags g{int(gate_pre)} b{int(beta_pre)} n{int(no_norm)}"
    check_out(out, ref_out, label=label)
    check_state(fin, ref_fin, label=label)


def test_forward_flags_through_the_segment_scan(monkeypatch):
    # segments of 256 tokens: local, transition and carried runs all see the flags
    from gated_delta_rule_51_gb300 import kda

    monkeypatch.setenv("KDA_SEG_TOKENS", "256")
    x = _case(2, 1100, 2, 811, True, True, True)
    kw = _kw(True, True, True)
    ref_out, ref_fin = _oracle(x, kw)
    out = torch.empty_like(x["v"])
    fin = torch.empty_like(x["initial_state"])
    kda.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], out, None, None, 0.0,
            initial_state=x["initial_state"], final_state=fin, **kw)
    torch.cuda.synchronize()
    check_out(out, ref_out, label="flags segment scan")
    check_state(fin, ref_fin, label="flags segment scan")


@pytest.mark.parametrize("gate_pre,beta_pre,no_norm", [(True, False, False), (False, True, True), (True, True, True)])
def test_decode_flags_match_oracle(gate_pre, beta_pre, no_norm):
    from gated_delta_rule_51_gb300 import kda

    x = _case(3, 4, 2, 821 + 4 * gate_pre + 2 * beta_pre + no_norm, gate_pre, beta_pre, no_norm,
              init_dtype=torch.bfloat16)
    kw = _kw(gate_pre, beta_pre, no_norm)
    ref_out, ref_fin = _oracle(x, kw)
    state = x["initial_state"].clone()
    out = torch.full_like(x["v"], float("nan"))
    a_log, dt = (None, None) if gate_pre else (x["A_log"], x["dt_bias"])
    kda.decode(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], out, a_log, dt, x["lower_bound"], state, **kw)
    torch.cuda.synchronize()
    label = f"decode flags g{int(gate_pre)} b{int(beta_pre)} n{int(no_norm)}"
    check_out(out, ref_out, label=label)
    check_state(state, ref_fin, label=label)
