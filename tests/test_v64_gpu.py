"""Value head dimension V = 64 (K stays 128): parity of the chunked forward and the
decode step with the fp64 oracle, which is written for any K and V.

The chunked forward runs a V = 64 head as one chain of 128 state rows whose last 64 rows
stay zero (the v tensor's second 64 columns read as zero; those rows are neither loaded
from nor written to the caller's states and outputs); the decode step runs one 64-row
CTA per head.  Checked against the plain recurrence with partial chunks, varlen
sequences, the segment scan and bf16 states, and against the first half of a V = 128
call whose second value half is zero.
"""
from __future__ import annotations

import pytest
import torch

from tests.gpu_helpers import check_out, check_state, random_case, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,T,H,lens,dtype,seed", [
    (1, 700, 3, [300, 17, 383], torch.float32, 911),
    (2, 200, 2, None, torch.bfloat16, 912),
])
def test_forward_v64_matches_oracle(B, T, H, lens, dtype, seed):
    x = random_case(B, T, H, seed=seed, lens=lens, init_dtype=dtype, V=64)
    ref_out, ref_fin = run_oracle(x)
    out, fin = run_gpu(x)
    check_out(out, ref_out, label=f"v64 B{B} T{T} H{H}")
    check_state(fin, ref_fin, label=f"v64 B{B} T{T} H{H}")


def test_forward_v64_through_the_segment_scan(monkeypatch):
    monkeypatch.setenv("KDA_SEG_TOKENS", "256")
    x = random_case(1, 1100, 2, seed=913, lb=-1.0, V=64)
    ref_out, ref_fin = run_oracle(x)
    out, fin = run_gpu(x)
    check_out(out, ref_out, label="v64 segments")
    check_state(fin, ref_fin, label="v64 segments")


def test_v64_equals_the_first_half_of_a_v128_call_with_zero_second_half():
    x = random_case(1, 300, 2, seed=914, lens=[100, 200], V=64)
    out, fin = run_gpu(x)
    y = dict(x)
    y["v"] = torch.cat([x["v"], torch.zeros_like(x["v"])], dim=-1).contiguous()
    y["initial_state"] = torch.cat([x["initial_state"], torch.zeros_like(x["initial_state"])], dim=2).contiguous()
    oy, fy = run_gpu(y)
    assert torch.equal(out, oy[..., :64])
    assert torch.equal(fin, fy[:, :, :64])
    assert torch.count_nonzero(fy[:, :, 64:]) == 0


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_v64_matches_oracle(dtype):
    from gated_delta_rule_51_gb300 import kda

    x = random_case(3, 4, 2, seed=915, init_dtype=dtype, V=64)
    ref_out, ref_fin = run_oracle(x)
    state = x["initial_state"].clone()
    out = torch.full_like(x["v"], float("nan"))
    kda.decode(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], out, x["A_log"], x["dt_bias"],
               x["lower_bound"], state)
    torch.cuda.synchronize()
    check_out(out, ref_out, label="decode v64")
    check_state(state, ref_fin, label="decode v64")
