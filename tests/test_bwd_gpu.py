"""GPU parity of the recurrent backward (kda_bwd with KDA_BWD_RECURRENT, through the C ABI) with
the fp64 oracle's gradient; the chunked form is tested in test_bwd_chunked_gpu.py.

The oracle (oracle/kda_oracle_bwd.c, pinned by finite differences in
test_oracle_backward_pins.py) receives exactly the GPU's inputs: the bf16 tensors, fp32
parameters and states converted to fp64, scale and lower_bound rounded to fp32.

Bound: every gradient tensor within relative Frobenius error 1e-5 of the oracle's.  The
kernels run the recurrence and its reverse in fp32 (plain loads, FMAs and warp sums, no
tensor cores); each operation rounds at about 6e-8 relative, and the decay (alpha < 1) and
the projection (I - beta kh kh^T) keep the state gradient from growing, so the errors stay
at the level of a few roundings: 1.2e-7 to 4.9e-7 measured over these cases on a GB300
(dA_log, a sum over every token, the largest).  1e-5 keeps a 20x margin and still fails
any wrong term (a dropped or mis-signed term moves a gradient by O(1) relative).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from tests.gpu_helpers import _report, random_case, rel_fro

pytestmark = pytest.mark.gpu

BOUND = 1e-5
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dh0", "dA_log", "ddt_bias")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_51_gb300 import kda

    kda.load_library()


def _grads_in(x, seed, with_dfinal=True):
    gen = torch.Generator().manual_seed(seed)
    B, T, H, _ = x["q"].shape
    N = x["cu_seqlens"].numel() - 1 if x.get("cu_seqlens") is not None else B
    dout = torch.randn((B, T, H, 128), generator=gen).to(torch.bfloat16).cuda()
    dfinal = (0.1 * torch.randn((N, H, 128, 128), generator=gen)).cuda() if with_dfinal else None
    return dout, dfinal


def _oracle(x, dout, dfinal, heads=None, **kw):
    import oracle

    def c(t, sl=None):
        if t is None:
            return None
        t = t.detach().cpu()
        if sl is not None:
            t = t[sl]
        return t.double().numpy()

    hs = slice(None) if heads is None else list(heads)
    tok = (slice(None), slice(None), hs)
    st = (slice(None), hs)
    cu = x.get("cu_seqlens")
    return oracle.kda_backward(
        c(x["q"], tok), c(x["k"], tok), c(x["v"], tok), c(x["g"], tok), c(x["beta"], tok),
        float(np.float32(x["scale"])), c(x["A_log"], (hs,)), c(x["dt_bias"], (hs,)),
        float(np.float32(x["lower_bound"])), c(dout, tok), c(x.get("initial_state"), st), c(dfinal, st),
        None if cu is None else cu.cpu().numpy(), **kw)


def _gpu(x, dout, dfinal, workspace=None, recurrent=True, **kw):
    from gated_delta_rule_51_gb300 import kda

    r = kda.bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["A_log"], x["dt_bias"],
                x["lower_bound"], dout, initial_state=x.get("initial_state"), dfinal=dfinal,
                cu_seqlens=x.get("cu_seqlens"), workspace=workspace, recurrent=recurrent, **kw)
    torch.cuda.synchronize()
    return r


def _compare(gpu, ref, label, heads=None, skip=()):
    for n in NAMES:
        if n in skip:
            continue
        g = gpu[n].detach().cpu().double().numpy()
        if heads is not None:
            g = g[:, :, list(heads)] if n in ("dq", "dk", "dv", "dg", "dbeta") else (
                g[:, list(heads)] if n == "dh0" else g[list(heads)])
        assert np.all(np.isfinite(g)), f"{label}: non-finite {n}"
        e = rel_fro(g, ref[n])
        _report(label, f"bwd_{n}_rel_fro", e)
        assert e <= BOUND, f"{label}: {n} rel-Fro {e:.3e} > {BOUND}"


@pytest.mark.parametrize("lens,init_dtype,dfin", [
    ([100, 7, 0, 193], torch.float32, True),
    ([300], torch.bfloat16, False),
    ([5, 16, 31, 8], None, True),
])
def test_backward_varlen_matches_oracle(lens, init_dtype, dfin):
    x = random_case(1, sum(lens), 2, seed=961 + len(lens), lens=lens, init_dtype=init_dtype)
    dout, dfinal = _grads_in(x, 962, dfin)
    r = _gpu(x, dout, dfinal)
    ref = _oracle(x, dout, dfinal)
    _compare(r, ref, f"bwd varlen {lens}")


def test_backward_fixed_batch_matches_oracle():
    x = random_case(2, 64, 3, seed=963, lb=-2.0)
    dout, dfinal = _grads_in(x, 964)
    _compare(_gpu(x, dout, dfinal), _oracle(x, dout, dfinal), "bwd fixed")


@pytest.mark.parametrize("gate", ["softplus", "preactivated", "beta_given", "no_l2norm"])
def test_backward_switches_match_oracle(gate):
    x = random_case(1, 150, 2, seed=965, lens=[60, 90])
    kw = {"softplus": dict(safe_gate=False), "preactivated": dict(use_gate_in_kernel=False),
          "beta_given": dict(use_beta_sigmoid_in_kernel=False),
          "no_l2norm": dict(use_qk_l2norm_in_kernel=False)}[gate]
    if gate == "preactivated":
        x["g"] = (-torch.nn.functional.softplus(x["g"].float())).to(torch.bfloat16)
    if gate == "beta_given":
        x["beta"] = torch.sigmoid(x["beta"].float()).to(torch.bfloat16)
    if gate == "no_l2norm":
        # raw q and k of norm about 1, as a caller that normalised them would pass
        x["q"] = (x["q"].float() / 11.3).to(torch.bfloat16)
        x["k"] = (x["k"].float() / 11.3).to(torch.bfloat16)
    dout, dfinal = _grads_in(x, 966)
    r = _gpu(x, dout, dfinal, **kw)
    ref = _oracle(x, dout, dfinal, **kw)
    _compare(r, ref, f"bwd {gate}")
    if gate == "preactivated":
        assert torch.count_nonzero(r["dA_log"]) == 0 and torch.count_nonzero(r["ddt_bias"]) == 0


def test_backward_long_sequence_weak_decay():
    x = random_case(1, 1000, 2, seed=967, lb=-1.0)
    dout, dfinal = _grads_in(x, 968)
    _compare(_gpu(x, dout, dfinal), _oracle(x, dout, dfinal), "bwd T=1000 lb=-1")


def test_backward_fixed_workload_sampled_heads():
    """The fixed workload's full size (B=2, T=4096, H=16, fp32 states); heads are independent,
    so the oracle runs three of them and every gradient of those heads is compared."""
    from gated_delta_rule_51_gb300 import inputs as I

    w = I.fixed_batch_workload()
    x = I.make_inputs(w, device="cuda")
    dout, dfinal = _grads_in(x, 969)
    r = _gpu(x, dout, dfinal)
    heads = (0, 7, 15)
    _compare(r, _oracle(x, dout, dfinal, heads=heads), "bwd fixed workload heads 0,7,15", heads=heads)


def test_backward_is_deterministic():
    x = random_case(1, 400, 3, seed=970, lens=[150, 250])
    dout, dfinal = _grads_in(x, 971)
    a, b = _gpu(x, dout, dfinal), _gpu(x, dout, dfinal)
    for n in NAMES:
        assert torch.equal(a[n], b[n]), n


def test_backward_malformed_cu_seqlens_is_flagged():
    from gated_delta_rule_51_gb300 import kda

    x = random_case(1, 64, 1, seed=972, lens=[32, 32])
    x["cu_seqlens"] = torch.tensor([0, 40, 32], dtype=torch.int64, device="cuda")   # decreasing
    dout, dfinal = _grads_in(x, 973)
    ws = torch.empty(kda.bwd_workspace_size(kda.make_shape(1, 64, 1, 2)), dtype=torch.uint8, device="cuda")
    _gpu(x, dout, dfinal, workspace=ws)
    assert kda.check_device_error(ws) & 2
    x["cu_seqlens"] = torch.tensor([0, 32, 64], dtype=torch.int64, device="cuda")
    _gpu(x, dout, dfinal, workspace=ws)
    assert kda.check_device_error(ws) == 0


def test_autograd_function_matches_the_oracle_gradient():
    """kda.kda_attention: the forward and backward kernels behind torch autograd.  Gradients
    come back in the inputs' dtypes: the bf16 ones carry their own rounding (relative error
    at most 2^-8 = 3.9e-3 an element; 1.7e-3 to 2.6e-3 relative Frobenius measured on a
    GB300), so they get the 5e-3 bound of bf16 results; the fp32 ones (A_log, dt_bias, the
    initial state) keep the 1e-5 bound (measured 0.9e-7 to 3.2e-7)."""
    from gated_delta_rule_51_gb300 import kda

    x = random_case(1, 200, 2, seed=975, lens=[80, 120])
    leaves = {n: x[n].detach().clone().requires_grad_(True)
              for n in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state")}
    out, fin = kda.kda_attention(leaves["q"], leaves["k"], leaves["v"], leaves["g"], leaves["beta"], x["scale"],
                                 leaves["A_log"], leaves["dt_bias"], x["lower_bound"],
                                 initial_state=leaves["initial_state"], cu_seqlens=x["cu_seqlens"],
                                 recurrent_backward=True)
    gen = torch.Generator().manual_seed(976)
    wo = torch.randn(out.shape, generator=gen).to(torch.bfloat16).cuda()
    wf = (0.1 * torch.randn(fin.shape, generator=gen)).cuda()
    ((out.float() * wo.float()).sum() + (fin * wf).sum()).backward()
    torch.cuda.synchronize()
    ref = _oracle(x, wo, wf)
    for n, gname, bound in (("q", "dq", 5e-3), ("k", "dk", 5e-3), ("v", "dv", 5e-3), ("g", "dg", 5e-3),
                            ("beta", "dbeta", 5e-3), ("A_log", "dA_log", BOUND), ("dt_bias", "ddt_bias", BOUND),
                            ("initial_state", "dh0", BOUND)):
        gr = leaves[n].grad
        assert gr is not None and gr.dtype == x[n].dtype, n
        e = rel_fro(gr.detach().cpu().double().numpy(), ref[gname])
        _report("bwd autograd", f"{gname}_rel_fro", e)
        assert e <= bound, f"{n}: rel-Fro {e:.3e} > {bound}"
