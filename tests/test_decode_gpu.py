"""Parity of the recurrent decode step (kda_decode) with the fp64 oracle.

The decode step is the KDA recurrence applied to T new tokens per sequence with
the state updated in place, so the oracle is the same token recurrence run on
[B, T] rows with that initial state.  Bounds are the forward pass's: outputs
max-abs <= 1e-2 and rel-Fro <= 5e-3, fp32 state rel-Fro <= 1e-3, bf16 state
rel-Fro <= 5e-3.
"""
from __future__ import annotations

import pytest
import torch

from tests.gpu_helpers import check_out, check_state, random_case, run_oracle

pytestmark = pytest.mark.gpu


def _decode(x, state):
    from gated_delta_rule_51_gb300 import kda

    out = torch.full_like(x["v"], float("nan"))
    kda.decode(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], out, x["A_log"], x["dt_bias"],
               x["lower_bound"], state)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("B,T,H,dtype,seed", [
    (3, 1, 4, torch.float32, 701),
    (2, 3, 2, torch.float32, 702),
    (5, 8, 1, torch.bfloat16, 703),
    (1, 1, 64, torch.bfloat16, 704),
    (4, 16, 3, torch.float32, 705),
])
def test_decode_matches_oracle(B, T, H, dtype, seed):
    x = random_case(B, T, H, seed=seed, lb=-5.0, init_dtype=dtype)
    ref_out, ref_state = run_oracle(x)
    state = x["initial_state"].clone()
    out = _decode(x, state)
    check_out(out, ref_out, label=f"decode B{B} T{T} H{H} {dtype}")
    check_state(state, ref_state, label=f"decode B{B} T{T} H{H} {dtype}")


def test_token_by_token_equals_one_call_bitwise():
    # with an fp32 state, T calls of one token do exactly the arithmetic of one call of T tokens
    x = random_case(3, 6, 2, seed=711, lb=-2.0, init_dtype=torch.float32)
    s_all = x["initial_state"].clone()
    out_all = _decode(x, s_all)
    s_one = x["initial_state"].clone()
    outs = []
    for t in range(6):
        xt = {k: (v[:, t:t + 1].contiguous() if k in ("q", "k", "v", "g", "beta") else v) for k, v in x.items()}
        outs.append(_decode(xt, s_one))
    assert torch.equal(torch.cat(outs, dim=1), out_all)
    assert torch.equal(s_one, s_all)


def test_decode_agrees_with_the_chunked_forward():
    from gated_delta_rule_51_gb300 import kda

    x = random_case(2, 40, 3, seed=712, lb=-1.0, init_dtype=torch.float32)
    out_f = torch.empty_like(x["v"])
    fin_f = torch.empty_like(x["initial_state"])
    kda.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], out_f, x["A_log"], x["dt_bias"],
            x["lower_bound"], initial_state=x["initial_state"], final_state=fin_f)
    state = x["initial_state"].clone()
    out_d = _decode(x, state)
    assert float((out_d.float() - out_f.float()).abs().max()) <= 2e-2
    assert float((state - fin_f).norm() / fin_f.norm()) <= 2e-3


def test_zero_tokens_leave_the_state_untouched():
    x = random_case(2, 0, 2, seed=713, init_dtype=torch.bfloat16)
    state = x["initial_state"].clone()
    _decode(x, state)
    assert torch.equal(state, x["initial_state"])


def test_serving_batch_sampled_heads():
    # a decode step of 256 sequences x 32 heads with fp32 states (the measured batch);
    # the oracle checks 16 of the 8192 (sequence, head) pairs
    x = random_case(256, 1, 32, seed=714, lb=-5.0, init_dtype=torch.float32)
    state = x["initial_state"].clone()
    out = _decode(x, state)
    idx = torch.tensor([0, 17, 63, 100, 128, 200, 254, 255])
    heads = [0, 31]
    for h in heads:
        xs = {k: v for k, v in x.items()}
        for name in ("q", "k", "v", "g"):
            xs[name] = x[name][idx][:, :, h:h + 1].contiguous()
        xs["beta"] = x["beta"][idx][:, :, h:h + 1].contiguous()
        xs["A_log"] = x["A_log"][h:h + 1].contiguous()
        xs["dt_bias"] = x["dt_bias"][h:h + 1].contiguous()
        xs["initial_state"] = x["initial_state"][idx][:, h:h + 1].contiguous()
        ref_out, ref_state = run_oracle(xs)
        check_out(out[idx][:, :, h:h + 1].contiguous(), ref_out, label=f"decode batch head {h}")
        check_state(state[idx][:, h:h + 1].contiguous(), ref_state, label=f"decode batch head {h}")
