"""Value head dimension V = 256 (K stays 128): parity of the chunked forward and the
decode step with the fp64 oracle, which is written for any K and V.

The value columns of the state are independent (rows v of S^T never mix), so the
GPU runs a V = 256 head as two chains of 128 state rows that share the head's q,
k, g and beta; these tests check the result against the plain recurrence, with
partial chunks, varlen sequences, the segment scan and bf16 states.
"""
from __future__ import annotations

import pytest
import torch

from tests.gpu_helpers import check_out, check_state, random_case, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,T,H,lens,dtype,seed", [
    (1, 700, 3, [300, 17, 383], torch.float32, 901),
    (2, 200, 2, None, torch.bfloat16, 902),
])
def test_forward_v256_matches_oracle(B, T, H, lens, dtype, seed):
    x = random_case(B, T, H, seed=seed, lens=lens, init_dtype=dtype, V=256)
    ref_out, ref_fin = run_oracle(x)
    out, fin = run_gpu(x)
    check_out(out, ref_out, label=f"v256 B{B} T{T} H{H}")
    check_state(fin, ref_fin, label=f"v256 B{B} T{T} H{H}")


def test_forward_v256_through_the_segment_scan(monkeypatch):
    monkeypatch.setenv("KDA_SEG_TOKENS", "256")
    x = random_case(1, 1100, 2, seed=903, lb=-1.0, V=256)
    ref_out, ref_fin = run_oracle(x)
    out, fin = run_gpu(x)
    check_out(out, ref_out, label="v256 segments")
    check_state(fin, ref_fin, label="v256 segments")


def test_v256_value_halves_equal_two_v128_calls():
    # the two 128-column halves of v and of the state are two independent problems
    x = random_case(1, 300, 2, seed=904, V=256)
    out, fin = run_gpu(x)
    for half in range(2):
        xh = dict(x)
        xh["v"] = x["v"][..., 128 * half:128 * half + 128].contiguous()
        xh["initial_state"] = x["initial_state"][:, :, 128 * half:128 * half + 128].contiguous()
        oh, fh = run_gpu(xh)
        assert torch.equal(oh, out[..., 128 * half:128 * half + 128])
        assert torch.equal(fh, fin[:, :, 128 * half:128 * half + 128])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_v256_matches_oracle(dtype):
    from gated_delta_rule_51_gb300 import kda

    x = random_case(3, 4, 2, seed=905, init_dtype=dtype, V=256)
    ref_out, ref_fin = run_oracle(x)
    state = x["initial_state"].clone()
    out = torch.full_like(x["v"], float("nan"))
    kda.decode(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], out, x["A_log"], x["dt_bias"],
               x["lower_bound"], state)
    torch.cuda.synchronize()
    check_out(out, ref_out, label="decode v256")
    check_state(state, ref_fin, label="decode v256")
