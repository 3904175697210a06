"""kda.kda_attention's autograd glue on CPU: the two CUDA entry points are replaced by
oracle-backed stand-ins (test only), so what is checked is the Function itself: which
tensors reach the backward, how dout and dfinal are passed, the dtypes the gradients come
back in, and the inputs that get none."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_51_gb300 import kda


def _fake_fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state=None, final_state=None,
              cu_seqlens=None, **sw):
    o, f = oracle.kda_forward(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, initial_state,
                              cu_seqlens, **sw)
    out.copy_(torch.from_numpy(o).reshape(out.shape).to(out.dtype))
    final_state.copy_(torch.from_numpy(f).to(final_state.dtype))
    return out, final_state


CALLS = []


def _fake_bwd(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, dout, initial_state=None, dfinal=None,
              cu_seqlens=None, workspace=None, recurrent=False, **sw):
    CALLS.append(dict(dout_dtype=dout.dtype, dfinal_dtype=None if dfinal is None else dfinal.dtype,
                      workspace=workspace is not None, recurrent=recurrent))
    d = lambda t: None if t is None else t.detach().double().numpy()
    r = oracle.kda_backward(d(q), d(k), d(v), d(g), d(beta), float(np.float32(scale)), d(A_log), d(dt_bias),
                            float(np.float32(lower_bound)), d(dout), d(initial_state), d(dfinal),
                            None if cu_seqlens is None else cu_seqlens.numpy(), **sw)
    return {n: torch.from_numpy(a).float() for n, a in r.items()}


@pytest.fixture(autouse=True)
def _fakes(monkeypatch):
    monkeypatch.setattr(kda, "fwd", _fake_fwd)
    monkeypatch.setattr(kda, "bwd", _fake_bwd)
    CALLS.clear()


def _leaf(t):
    return t.detach().clone().requires_grad_(True)


@pytest.mark.parametrize("init_dtype,lens", [(torch.float32, [7, 0, 9]), (torch.bfloat16, None), (None, [16])])
def test_gradients_reach_every_input_in_its_dtype(init_dtype, lens):
    gen = torch.Generator().manual_seed(3)
    B, T, H = (1, sum(lens), 2) if lens else (2, 8, 2)
    N = len(lens) if lens else B
    bf = lambda *s: torch.randn(*s, generator=gen).to(torch.bfloat16)
    x = dict(q=bf(B, T, H, 128), k=bf(B, T, H, 128), v=bf(B, T, H, 128), g=bf(B, T, H, 128), beta=bf(B, T, H),
             A_log=torch.rand(H, generator=gen) - 0.5, dt_bias=0.1 * torch.randn(H, 128, generator=gen))
    init = None if init_dtype is None else (0.02 * torch.randn(N, H, 128, 128, generator=gen)).to(init_dtype)
    cu = None if lens is None else torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int64)
    leaves = {n: _leaf(t) for n, t in x.items()}
    h0 = None if init is None else _leaf(init)
    out, fin = kda.kda_attention(leaves["q"], leaves["k"], leaves["v"], leaves["g"], leaves["beta"], 0.088,
                                 leaves["A_log"], leaves["dt_bias"], -3.0, initial_state=h0, cu_seqlens=cu)
    assert out.dtype == torch.bfloat16 and fin.dtype == (init_dtype or torch.float32)
    wo = torch.randn(out.shape, generator=gen).to(torch.bfloat16)
    wf = torch.randn(fin.shape, generator=gen)
    ((out.float() * wo.float()).sum() + (fin.float() * wf).sum()).backward()
    assert CALLS == [dict(dout_dtype=torch.bfloat16, dfinal_dtype=torch.float32, workspace=False, recurrent=False)]
    ref = _fake_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], 0.088, x["A_log"], x["dt_bias"], -3.0, wo,
                    init, wf.to(fin.dtype).float(), cu)
    for n, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"), ("A_log", "dA_log"),
                     ("dt_bias", "ddt_bias")):
        assert leaves[n].grad.dtype == x[n].dtype, n
        assert torch.equal(leaves[n].grad, ref[gname].to(x[n].dtype)), n
    if h0 is not None:
        assert h0.grad.dtype == init.dtype and torch.equal(h0.grad, ref["dh0"].to(init.dtype))


def test_a_preactivated_gate_gives_its_parameters_no_gradient():
    gen = torch.Generator().manual_seed(4)
    bf = lambda *s: torch.randn(*s, generator=gen).to(torch.bfloat16)
    q, k, v = (_leaf(bf(1, 5, 1, 128)) for _ in range(3))
    beta = _leaf(bf(1, 5, 1))
    g = _leaf((-torch.rand(1, 5, 1, 128, generator=gen)).to(torch.bfloat16))
    A, D = _leaf(torch.zeros(1)), _leaf(torch.zeros(1, 128))
    out, fin = kda.kda_attention(q, k, v, g, beta, 0.1, A, D, 0.0, use_gate_in_kernel=False)
    out.float().sum().backward()
    assert A.grad is None and D.grad is None
    assert g.grad is not None and g.grad.dtype == torch.bfloat16
    assert CALLS[0]["dfinal_dtype"] is None      # the final state was not used


def _small(K=128, V=128, seed=5):
    gen = torch.Generator().manual_seed(seed)
    bf = lambda *s: torch.randn(*s, generator=gen).to(torch.bfloat16)
    return dict(q=_leaf(bf(1, 6, 1, K)), k=_leaf(bf(1, 6, 1, K)), v=_leaf(bf(1, 6, 1, V)), g=_leaf(bf(1, 6, 1, K)),
                beta=_leaf(bf(1, 6, 1)), A_log=_leaf(torch.zeros(1)), dt_bias=_leaf(torch.zeros(1, K)))


@pytest.mark.parametrize("K,V", [(64, 128), (128, 256), (128, 64)])
def test_other_head_dims_with_grad_are_refused_before_the_forward(monkeypatch, K, V):
    ran = []
    monkeypatch.setattr(kda, "fwd", lambda *a, **kw: ran.append(1))
    x = _small(K, V)
    with pytest.raises(ValueError, match="K = V = 128"):
        kda.kda_attention(x["q"], x["k"], x["v"], x["g"], x["beta"], 0.1, x["A_log"], x["dt_bias"], -1.0)
    assert ran == []
    # without gradients the same shapes run
    d = {n: t.detach() for n, t in x.items()}
    monkeypatch.setattr(kda, "fwd", lambda *a, **kw: ran.append(1))
    kda.kda_attention(d["q"], d["k"], d["v"], d["g"], d["beta"], 0.1, d["A_log"], d["dt_bias"], -1.0)
    assert ran == [1]


def test_check_errors_raises_on_the_device_error_word(monkeypatch):
    seen = []

    def fake_check(workspace=None, device=None):
        seen.append(workspace is not None)
        return 2   # malformed cu_seqlens

    monkeypatch.setattr(kda, "check_device_error", fake_check)
    x = _small()
    with pytest.raises(kda.KDAError, match="BAD_SEQLENS"):
        kda.kda_attention(x["q"], x["k"], x["v"], x["g"], x["beta"], 0.1, x["A_log"], x["dt_bias"], -1.0,
                          check_errors=True)
    assert seen == [False]   # the forward's own (cached) workspace
    # unchecked calls never read the word
    seen.clear()
    out, fin = kda.kda_attention(x["q"], x["k"], x["v"], x["g"], x["beta"], 0.1, x["A_log"], x["dt_bias"], -1.0)
    assert seen == []
    # the backward reads the error word of a workspace it allocated itself
    monkeypatch.setattr(kda, "check_device_error", lambda workspace=None, device=None: seen.append(workspace) or 0)
    out, fin = kda.kda_attention(x["q"], x["k"], x["v"], x["g"], x["beta"], 0.1, x["A_log"], x["dt_bias"], -1.0,
                                 check_errors=True)
    out.float().sum().backward()
    assert seen[0] is None and seen[1] is not None and CALLS[-1]["workspace"]


def test_raise_on_device_error_maps_each_bit():
    kda.raise_on_device_error(0, "x")
    for bit, name in ((1, "TIMEOUT"), (2, "BAD_SEQLENS"), (4, "GATE_RANGE")):
        with pytest.raises(kda.KDAError, match=name):
            kda.raise_on_device_error(bit, "x")
