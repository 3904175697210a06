"""Key head dimension K = 64: parity of the chunked forward and the decode step with the
fp64 oracle, which is written for any K and V.

Both paths run a K = 64 head with its key channels 64-127 held at zero: q = k = 0 there and
the gate 0 (decay 1), so those state columns start at zero, stay zero and add nothing to
any output; they are neither read from nor written to the caller's [.., V, 64] states.
Checked against the plain recurrence (scale 1/8) with partial chunks, varlen sequences,
the segment scan, bf16 states, the three gates and V = 64 / 256, and bit for bit against
a K = 128 call whose channels 64-127 are zero.
"""
from __future__ import annotations

import pytest
import torch

from tests.gpu_helpers import check_out, check_state, random_case, run_gpu, run_oracle, to_cpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_51_gb300 import kda

    kda.load_library()


@pytest.mark.parametrize("B,T,H,lens,dtype,V,seed", [
    (1, 700, 3, [300, 17, 383], torch.float32, 128, 931),
    (2, 200, 2, None, torch.bfloat16, 128, 932),
    (1, 333, 2, [1, 16, 316], torch.float32, 64, 933),
    (1, 260, 2, [130, 130], torch.float32, 256, 934),
])
def test_forward_k64_matches_oracle(B, T, H, lens, dtype, V, seed):
    x = random_case(B, T, H, seed=seed, lens=lens, init_dtype=dtype, V=V, K=64)
    assert x["q"].shape[-1] == 64 and x["scale"] == 0.125
    ref_out, ref_fin = run_oracle(x)
    out, fin = run_gpu(x)
    check_out(out, ref_out, label=f"k64 B{B} T{T} H{H} V{V}")
    check_state(fin, ref_fin, label=f"k64 B{B} T{T} H{H} V{V}")


def test_forward_k64_through_the_segment_scan(monkeypatch):
    monkeypatch.setenv("KDA_SEG_TOKENS", "256")
    for dtype, seed in ((torch.float32, 935), (torch.bfloat16, 936)):
        x = random_case(1, 1100, 2, seed=seed, lb=-1.0, init_dtype=dtype, K=64)
        ref_out, ref_fin = run_oracle(x)
        out, fin = run_gpu(x)
        check_out(out, ref_out, label=f"k64 segments {dtype}")
        check_state(fin, ref_fin, label=f"k64 segments {dtype}")


def test_forward_k64_without_states_and_with_empty_sequences():
    x = random_case(1, 90, 2, seed=937, lens=[0, 45, 0, 45], init_dtype=None, K=64)
    ref_out, _ = run_oracle(x)
    out, fin = run_gpu(x, final_dtype=None)
    assert fin is None
    check_out(out, ref_out, label="k64 no states")


@pytest.mark.parametrize("gate", ["softplus", "preactivated"])
def test_forward_k64_other_gates(gate):
    import oracle
    from gated_delta_rule_51_gb300 import kda

    x = random_case(1, 400, 2, seed=938, lens=[150, 250], K=64)
    kw = dict(safe_gate=False) if gate == "softplus" else dict(use_gate_in_kernel=False)
    if gate == "preactivated":
        # a natural-log decay at most 0, as the caller's own gate would give
        x["g"] = (-torch.nn.functional.softplus(x["g"].float())).to(torch.bfloat16)
    xc = to_cpu(x)
    ref_out, ref_fin = oracle.kda_forward(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["scale"], xc["A_log"],
                                          xc["dt_bias"], xc["lower_bound"], xc["initial_state"], xc["cu_seqlens"],
                                          **kw)
    ws = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
    out = torch.full_like(x["v"], float("nan"))
    fin = torch.full_like(x["initial_state"], float("nan"))
    kda.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], out, x["A_log"], x["dt_bias"],
            x["lower_bound"], initial_state=x["initial_state"], final_state=fin, cu_seqlens=x["cu_seqlens"],
            workspace=ws, **kw)
    torch.cuda.synchronize()
    assert kda.check_device_error(ws) == 0
    check_out(out, ref_out, label=f"k64 {gate}")
    check_state(fin, ref_fin, label=f"k64 {gate}")


def _pad_k(x):
    """The same problem at K = 128: channels 64-127 of q, k, g, dt_bias and the state zero."""
    y = dict(x)
    for n in ("q", "k", "g"):
        y[n] = torch.cat([x[n], torch.zeros_like(x[n])], dim=-1).contiguous()
    y["dt_bias"] = torch.cat([x["dt_bias"], torch.zeros_like(x["dt_bias"])], dim=-1).contiguous()
    if x.get("initial_state") is not None:
        y["initial_state"] = torch.cat([x["initial_state"], torch.zeros_like(x["initial_state"])],
                                       dim=-1).contiguous()
    return y


def test_k64_equals_a_k128_call_with_zero_upper_channels():
    x = random_case(1, 300, 2, seed=939, lens=[100, 200], K=64)
    out, fin = run_gpu(x)
    oy, fy = run_gpu(_pad_k(x))
    assert torch.equal(out, oy)
    assert torch.equal(fin, fy[..., :64])
    assert torch.count_nonzero(fy[..., 64:]) == 0


def _decode(x, state, **kw):
    from gated_delta_rule_51_gb300 import kda

    out = torch.full_like(x["v"], float("nan"))
    kda.decode(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], out, x["A_log"], x["dt_bias"],
               x["lower_bound"], state, **kw)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("dtype,V", [(torch.float32, 128), (torch.bfloat16, 128), (torch.float32, 64),
                                     (torch.float32, 256)])
def test_decode_k64_matches_oracle(dtype, V):
    x = random_case(3, 4, 2, seed=940 + V, init_dtype=dtype, V=V, K=64)
    ref_out, ref_fin = run_oracle(x)
    state = x["initial_state"].clone()
    out = _decode(x, state)
    check_out(out, ref_out, label=f"decode k64 V{V}")
    check_state(state, ref_fin, label=f"decode k64 V{V}")


def test_decode_k64_equals_a_k128_step_with_zero_upper_channels():
    x = random_case(4, 1, 3, seed=941, K=64)
    s64 = x["initial_state"].clone()
    o64 = _decode(x, s64)
    y = _pad_k(x)
    s128 = y["initial_state"].clone()
    o128 = _decode(y, s128)
    assert torch.equal(o64, o128)
    assert torch.equal(s64, s128[..., :64])
    assert torch.count_nonzero(s128[..., 64:]) == 0
