"""The allocation-free entry point, kda_fwd_static_workspace.

Callers that cannot allocate device memory (their allocator belongs to a host
framework, or allocation is forbidden after start-up) call this variant, which
uses a workspace array built into the library instead of one they pass in.
This test calls it through the C ABI twice in a row, on two different
problems, and checks each result against kda_fwd with a caller-provided
workspace, within the bounds used by the parity tests.  The file sorts last
so that a run stopping at the first failure has run every other test first.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

from tests.gpu_helpers import OUT_MAX_ABS, OUT_REL_FRO, STATE_REL_FRO_FP32, random_case

pytestmark = pytest.mark.gpu


def _declare(lib):
    p = ctypes.c_void_p
    fn = lib.kda_fwd_static_workspace
    fn.argtypes = [ctypes.c_void_p, p, p, p, p, p, ctypes.c_float, p, p, p, ctypes.c_float, p, ctypes.c_int,
                   p, ctypes.c_int, p, p]
    fn.restype = ctypes.c_int
    return fn


def _no_alloc_call(fn, x, out, fin):
    from gated_delta_rule_51_gb300 import kda

    B, T, H, _ = x["q"].shape
    cu = x.get("cu_seqlens")
    N = cu.numel() - 1 if cu is not None else B
    shape = kda.make_shape(B, T, H, N)
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    init = x.get("initial_state")
    st = fn(ctypes.byref(shape), ptr(x["q"]), ptr(x["k"]), ptr(x["v"]), ptr(x["g"]), ptr(x["beta"]),
            ctypes.c_float(x["scale"]), ptr(out), ptr(x["A_log"]), ptr(x["dt_bias"]),
            ctypes.c_float(x["lower_bound"]), ptr(init), kda._state_code(init), ptr(fin), kda._state_code(fin),
            ptr(cu), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def _compare(a: torch.Tensor, b: torch.Tensor, rel_bound: float, abs_bound=None):
    a64, b64 = a.double(), b.double()
    assert torch.isfinite(a64).all()
    if abs_bound is not None:
        assert float((a64 - b64).abs().max()) <= abs_bound
    den = float(b64.norm())
    assert float((a64 - b64).norm()) <= rel_bound * (den if den > 0 else 1.0)


def test_static_workspace_matches_kda_fwd_twice_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_51_gb300 import kda

    fn = _declare(kda.load_library())
    cases = [
        # long single sequences: split into segments, so the workspace slots are used
        random_case(2, 4096, 16, seed=501, lb=-2.0),
        # a varlen batch with a partial chunk and an empty sequence, bf16 states
        random_case(1, 700, 4, seed=502, lens=[300, 0, 17, 383], init_dtype=torch.bfloat16),
    ]
    for x in cases:
        B, T, H, _ = x["q"].shape
        N = x["initial_state"].shape[0]
        out_ref = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device="cuda")
        fin_ref = torch.empty_like(x["initial_state"])
        kda.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], out_ref, x["A_log"], x["dt_bias"],
                x["lower_bound"], initial_state=x["initial_state"], final_state=fin_ref,
                cu_seqlens=x["cu_seqlens"])
        out = torch.full_like(out_ref, float("nan"))
        fin = torch.full_like(fin_ref, float("nan"))
        assert _no_alloc_call(fn, x, out, fin) == kda.KDA_OK
        torch.cuda.synchronize()
        assert fin.shape[0] == N
        _compare(out.float(), out_ref.float(), OUT_REL_FRO, OUT_MAX_ABS)
        bound = STATE_REL_FRO_FP32 if fin.dtype == torch.float32 else OUT_REL_FRO
        _compare(fin.float(), fin_ref.float(), bound)


def test_static_workspace_rejects_problems_beyond_its_size():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_51_gb300 import kda

    fn = _declare(kda.load_library())
    # a million one-token sequences over 64 heads: a work list far beyond 64 MiB
    shape = kda.make_shape(1 << 20, 1, 64, 1 << 20)
    assert kda.workspace_size(shape) > (64 << 20)
    dummy = torch.zeros(16, dtype=torch.float32, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    st = fn(ctypes.byref(shape), p, p, p, p, p, ctypes.c_float(0.1), p, p, p, ctypes.c_float(-1.0), None, 0,
            None, 0, None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 3   # KDA_ERR_WORKSPACE_TOO_SMALL, nothing launched


def test_static_workspace_at_its_size_limit():
    """The largest problem of a family whose workspace still fits the built-in array runs and
    matches kda_fwd; the next larger one is refused."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_51_gb300 import kda

    fn = _declare(kda.load_library())
    limit, H = 64 << 20, 8
    ws = lambda n: kda.workspace_size(kda.make_shape(1, n, H, n))   # n one-token sequences
    lo, hi = 1, 1
    while ws(hi) <= limit:
        lo, hi = hi, 2 * hi
    while hi - lo > 1:   # ws(lo) <= limit < ws(hi)
        mid = (lo + hi) // 2
        lo, hi = (mid, hi) if ws(mid) <= limit else (lo, mid)
    assert ws(lo) <= limit < ws(hi) and ws(lo) > limit // 2
    # (no states: one per sequence would dwarf the rest of the problem)
    x = random_case(1, lo, H, seed=503, lens=[1] * lo, init_dtype=None)
    out_ref = torch.empty((1, lo, H, 128), dtype=torch.bfloat16, device="cuda")
    kda.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], out_ref, x["A_log"], x["dt_bias"],
            x["lower_bound"], cu_seqlens=x["cu_seqlens"])
    out = torch.full_like(out_ref, float("nan"))
    assert _no_alloc_call(fn, x, out, None) == kda.KDA_OK
    torch.cuda.synchronize()
    _compare(out.float(), out_ref.float(), OUT_REL_FRO, OUT_MAX_ABS)
    # one size up: refused before anything runs, outputs untouched
    y = random_case(1, hi, H, seed=504, lens=[1] * hi, init_dtype=None)
    out2 = torch.full((1, hi, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert _no_alloc_call(fn, y, out2, None) == 3
    torch.cuda.synchronize()
    assert torch.isnan(out2.float()).all()
