"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Every case draws seeded synthetic inputs, runs ``kda_fwd`` on the GPU and the
token-by-token oracle on the CPU, and compares element by element with the
bounds in ``tests/gpu_helpers.py``.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

from gated_delta_rule_51_gb300 import inputs as I
from tests.gpu_helpers import (check_out, check_state, random_case, run_gpu, run_oracle, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_51_gb300 import kda

    kda.load_library()


@pytest.fixture
def seg_tokens(monkeypatch):
    """Force the segment length (exercises the segment scan on small inputs)."""
    def set_(n):
        if n is None:
            monkeypatch.delenv("KDA_SEG_TOKENS", raising=False)
        else:
            monkeypatch.setenv("KDA_SEG_TOKENS", str(n))
    return set_


def _compare(x, final_dtype=torch.float32, label="", seg=None):
    out, fin = run_gpu(x, final_dtype=final_dtype)
    ref_out, ref_fin = run_oracle(x)
    B, T, H, _ = x["q"].shape
    m, r = check_out(out, ref_out.reshape(B * T, H, 128), label=label)
    s = check_state(fin, ref_fin, label=label) if fin is not None else None
    return m, r, s


def test_tiny_workload():
    w = I.tiny_workload()
    x = I.make_inputs(w, device="cuda")
    _compare(x, torch.float32, "tiny")


@pytest.mark.parametrize("T", [1, 2, 7, 15, 16, 17, 31, 32, 33, 48, 127, 129])
def test_partial_chunks_single_sequence(T):
    x = random_case(1, T, 2, seed=100 + T)
    _compare(x, torch.float32, f"T={T}")


def test_partial_chunk_sweep_varlen():
    lens = list(range(1, 34)) + [127, 129]
    x = random_case(1, sum(lens), 2, seed=7, lens=lens)
    _compare(x, torch.float32, "sweep varlen")


def test_varlen_with_empty_sequences_bf16_state():
    lens = [0, 5, 0, 40, 16, 0]
    x = random_case(1, sum(lens), 3, seed=8, lens=lens, init_dtype=torch.bfloat16)
    _compare(x, torch.bfloat16, "empty seqs")


@pytest.mark.parametrize("lb", [0.0, -1.0, -5.0])
def test_lower_bound_range(lb):
    x = random_case(2, 100, 2, seed=9, lb=lb)
    _compare(x, torch.float32, f"lb={lb}")


def test_no_initial_state_no_final_state():
    x = random_case(1, 50, 2, seed=10, init_dtype=None)
    out, fin = run_gpu(x, final_dtype=None)
    assert fin is None
    ref_out, _ = run_oracle(x)
    check_out(out, ref_out.reshape(50, 2, 128), label="no states")


@pytest.mark.parametrize("seg", [16, 48, 64, 512])
def test_segment_scan_matches_oracle(seg_tokens, seg):
    """Short segments force the three-phase segment scan (carry + composition)."""
    seg_tokens(seg)
    lens = [300, 17, 1000, 64, 129]
    x = random_case(1, sum(lens), 2, seed=11 + seg, lens=lens)
    _compare(x, torch.float32, f"seg={seg}")
    x2 = random_case(1, sum(lens), 2, seed=12 + seg, lens=lens, init_dtype=torch.bfloat16)
    _compare(x2, torch.bfloat16, f"seg={seg} bf16")


@pytest.mark.parametrize("lb,seg", [(-0.1, 48), (-0.1, 512), (0.0, 64)])
def test_segment_scan_with_a_gate_that_keeps_its_state(seg_tokens, lb, seg):
    """A gate that barely decays (lower_bound near 0): within a segment the transition never
    becomes zero in fp32, so the transition and correction runs go through every chunk and the
    composition multiplies every transition."""
    seg_tokens(seg)
    lens = [1500, 17, 700, 64]
    x = random_case(1, sum(lens), 2, seed=21 + seg, lens=lens, lb=lb)
    out, fin = run_gpu(x)
    ref_out, ref_fin = run_oracle(x)
    check_out(out, ref_out.reshape(sum(lens), 2, 128), label=f"keep lb={lb} seg={seg}")
    check_state(fin, ref_fin, label=f"keep lb={lb} seg={seg}")


def test_segment_scan_heads_that_forget_and_heads_that_keep(seg_tokens):
    """In one call: head 0 decays slowly (A_log 0, dt_bias -4.6: sigmoid(g - 4.6) is about
    0.01, a decay near exp(-0.05) per token), so within a 64-token segment its transition never
    reaches zero and its transition and correction runs go to the end; head 1 forgets within a
    few chunks, so its runs stop early.  Both must match the oracle."""
    seg_tokens(64)
    lens = [900, 300, 33]
    x = random_case(1, sum(lens), 2, seed=31, lens=lens, lb=-5.0)
    x["A_log"][0] = 0.0
    x["dt_bias"][0].fill_(-4.6)
    _compare(x, torch.float32, "forget and keep")
    x2 = random_case(1, sum(lens), 2, seed=32, lens=lens, lb=-5.0, init_dtype=None)
    x2["A_log"][1] = 0.0
    x2["dt_bias"][1].fill_(-4.6)
    _compare(x2, torch.float32, "forget and keep, no initial state")


def test_segment_scan_without_initial_state(seg_tokens):
    seg_tokens(32)
    x = random_case(2, 200, 2, seed=13, init_dtype=None)
    _compare(x, torch.float32, "seg no init")


def test_fixed_batch_workload():
    w = I.fixed_batch_workload()
    x = I.make_inputs(w, device="cuda")
    _compare(x, torch.float32, w.name)


def test_varlen_workload():
    w = I.varlen_workload()
    x = I.make_inputs(w, device="cuda")
    _compare(x, torch.bfloat16, w.name)


@pytest.mark.parametrize("total,H", [(8192, 32), (8192, 64), (32768, 32)])
def test_sweep_workloads_small_cells(total, H):
    w = I.sweep_workload(total, H)
    x = I.make_inputs(w, device="cuda")
    _compare(x, torch.float32, w.name)


def test_segment_length_refined_to_fit_one_wave():
    """One sequence of 4096 tokens with 40 heads: on a GPU of 152 SMs (304 resident chain CTAs)
    the host's segment length cuts it into 8 segments, 320 forward runs, a few more than one
    wave, and the schedule kernel takes a longer segment (7 segments, 280 runs).  Whatever the
    SM count, the result must match the oracle."""
    x = random_case(1, 4096, 40, seed=1990, lens=[4096])
    _compare(x, torch.float32, "one sequence, 40 heads")


def test_determinism_bitwise():
    x = random_case(1, 3000, 4, seed=14, lens=[1000, 2000])
    o1, f1 = run_gpu(x)
    o2, f2 = run_gpu(x)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(f1, f2)


def test_in_place_state_update(seg_tokens):
    for seg in (None, 64):
        seg_tokens(seg)
        x = random_case(1, 400, 2, seed=15, lens=[150, 250])
        ref_out, ref_fin = run_oracle(x)
        state = x["initial_state"].clone()
        y = dict(x)
        y["initial_state"] = state
        out, fin = run_gpu(y, final_state=state)
        assert fin.data_ptr() == state.data_ptr()
        check_out(out, ref_out, label="in place")
        check_state(state, ref_fin, label="in place")


def test_split_and_carry_on_gpu():
    x = random_case(1, 300, 2, seed=16)
    out, fin = run_gpu(x)
    a = dict(x)
    b = dict(x)
    for n in ("q", "k", "v", "g", "beta"):
        a[n] = x[n][:, :137].contiguous()
        b[n] = x[n][:, 137:].contiguous()
    oa, fa = run_gpu(a)
    b["initial_state"] = fa
    ob, fb = run_gpu(b)
    ref_out, ref_fin = run_oracle(x)
    check_out(torch.cat([oa, ob], 1), ref_out, label="carry")
    check_state(fb, ref_fin, label="carry")


def test_batch_rows_equal_varlen_equal_lengths():
    x = random_case(3, 80, 2, seed=17)
    o1, f1 = run_gpu(x)
    y = dict(x)
    for n in ("q", "k", "v", "g", "beta"):
        y[n] = x[n].reshape(1, 240, *x[n].shape[2:]).contiguous()
    y["cu_seqlens"] = torch.tensor([0, 80, 160, 240], dtype=torch.int64, device="cuda")
    o2, f2 = run_gpu(y)
    assert torch.equal(o1.reshape(-1).view(torch.int16), o2.reshape(-1).view(torch.int16))
    assert torch.equal(f1, f2)


def test_malformed_cu_seqlens_is_flagged_not_trapped():
    from gated_delta_rule_51_gb300 import kda

    x = random_case(1, 64, 1, seed=18, lens=[32, 32])
    x["cu_seqlens"] = torch.tensor([0, 40, 32], dtype=torch.int64, device="cuda")   # decreasing
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    run_gpu(x, workspace=ws)
    flags = kda.check_device_error(ws)
    assert flags & 2
    # a well-formed call on the same workspace clears the word
    x["cu_seqlens"] = torch.tensor([0, 32, 64], dtype=torch.int64, device="cuda")
    run_gpu(x, workspace=ws)
    assert kda.check_device_error(ws) == 0


def test_long_workload_sampled():
    """T = 1,048,576, H = 8: final state in full, outputs on sampled rows."""
    w = I.long_workload()
    x = I.make_inputs(w, device="cuda")
    out, fin = run_gpu(x)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(0, 64), rng.integers(0, w.T, 2048),
                                     np.arange(w.T - 64, w.T)]))
    ref_out, ref_fin = run_oracle(x, out_rows=rows)
    check_out(out, ref_out, rows=rows, label=w.name)
    check_state(fin, ref_fin, label=w.name)


def test_forward_captured_in_a_cuda_graph_replays_identically():
    # kda_fwd allocates nothing and never waits on the host, so a call can be captured
    # once and replayed; each replay gives the direct call's result bit for bit
    from gated_delta_rule_51_gb300 import kda

    x = random_case(1, 700, 3, seed=951, lens=[300, 17, 383])
    out_ref, fin_ref = run_gpu(x)
    ws = torch.empty(kda.workspace_size(kda.make_shape(1, 700, 3, 3)), dtype=torch.uint8, device="cuda")
    out = torch.full_like(out_ref, float("nan"))
    fin = torch.full_like(fin_ref, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            kda.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], out, x["A_log"], x["dt_bias"],
                    x["lower_bound"], initial_state=x["initial_state"], final_state=fin,
                    cu_seqlens=x["cu_seqlens"], workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        out.fill_(float("nan"))
        fin.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, out_ref)
        assert torch.equal(fin, fin_ref)


def test_segment_scan_captured_in_a_cuda_graph_replays_identically(monkeypatch):
    # with segments forced, a call runs the transition launch, the forward launch overlapping
    # it, the composition and the correction launch starting beside the composition; captured
    # in a graph (programmatic dependencies become graph edges), each replay still gives the
    # direct call's result bit for bit, and that result matches the oracle
    from gated_delta_rule_51_gb300 import kda

    monkeypatch.setenv("KDA_SEG_TOKENS", "96")
    x = random_case(1, 700, 3, seed=952, lens=[300, 17, 383])
    out_ref, fin_ref = run_gpu(x)
    o_or, f_or = run_oracle(x)
    check_out(out_ref, o_or.reshape(700, 3, 128), label="graph, segments of 96")
    check_state(fin_ref, f_or, label="graph, segments of 96")
    ws = torch.empty(kda.workspace_size(kda.make_shape(1, 700, 3, 3)), dtype=torch.uint8, device="cuda")
    out = torch.full_like(out_ref, float("nan"))
    fin = torch.full_like(fin_ref, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            kda.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], out, x["A_log"], x["dt_bias"],
                    x["lower_bound"], initial_state=x["initial_state"], final_state=fin,
                    cu_seqlens=x["cu_seqlens"], workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        out.fill_(float("nan"))
        fin.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, out_ref)
        assert torch.equal(fin, fin_ref)


@pytest.mark.parametrize("total,H", [(32768, 64), (131072, 32), (131072, 64), (262144, 32), (262144, 64)])
def test_sweep_workloads_large_cells_sampled(total, H):
    """The sweep cells past the three small ones (up to 16.8M token-heads at H = 64): every
    final state in full, outputs on sampled rows (the first and last rows of every sequence
    and random ones). With the small cells above, every cell of the sweep is compared."""
    w = I.sweep_workload(total, H)
    x = I.make_inputs(w, device="cuda")
    out, fin = run_gpu(x)
    cu = x["cu_seqlens"].cpu().numpy()
    rng = np.random.default_rng(total + H)
    rows = np.unique(np.concatenate([cu[:-1], np.maximum(cu[1:] - 1, 0), rng.integers(0, total, 2048)]))
    rows = rows[rows < total]
    ref_out, ref_fin = run_oracle(x, out_rows=rows)
    check_out(out, ref_out, rows=rows, label=w.name)
    check_state(fin, ref_fin, label=w.name)


@pytest.mark.parametrize("lb,T", [(-0.1, 2000), (0.0, 2000), (0.0, 8192), (-0.3, 2000)])
def test_weak_and_no_decay_long_runs(lb, T):
    """Near lower_bound = 0 nothing fades from the state.  A single bf16 copy of it (the A
    operand of the S-side GEMM) would feed back 2^-9 of rounding every chunk and, with no
    decay to forget it, build up to about 1.9e-3 rel-Fro; the library therefore reads the state
    as a bf16 pair there (lower_bound > -0.25, KDA_PRECISE_STATE), and the fp32 state meets
    the 1e-3 bound at any lower_bound.  -0.3 checks the single copy just past that switch."""
    x = random_case(1, T, 4, seed=77, lb=lb)
    ref_out, ref_fin = run_oracle(x)
    out, fin = run_gpu(x)
    check_out(out, ref_out, label=f"lb={lb} T={T}")
    check_state(fin, ref_fin, label=f"lb={lb} T={T}")


def test_precise_state_flag_on_a_decaying_gate():
    """KDA_PRECISE_STATE asked for where the library would not pick it (lower_bound -5,
    varlen with partial chunks and bf16 states): same bounds."""
    from gated_delta_rule_51_gb300 import kda

    lens = [700, 33, 1290]
    x = random_case(1, sum(lens), 3, seed=78, lens=lens, init_dtype=torch.bfloat16)
    out = torch.full((1, sum(lens), 3, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    fin = torch.full_like(x["initial_state"], float("nan"))
    kda.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], out, x["A_log"], x["dt_bias"],
            x["lower_bound"], initial_state=x["initial_state"], final_state=fin, cu_seqlens=x["cu_seqlens"],
            precise_state=True)
    torch.cuda.synchronize()
    ref_out, ref_fin = run_oracle(x)
    check_out(out, ref_out.reshape(sum(lens), 3, 128), label="precise flag")
    check_state(fin, ref_fin, label="precise flag")


def test_thousands_of_short_sequences():
    """3000 sequences of 0-40 tokens (several of the schedule kernel's 1024-sequence tiles),
    with empty ones and lengths on both sides of the 16-token chunk."""
    rng = np.random.default_rng(3000)
    lens = [int(x) for x in rng.integers(0, 41, 3000)]
    lens[0], lens[1], lens[-1] = 0, 16, 1
    x = random_case(1, sum(lens), 2, seed=3001, lens=lens)
    _compare(x, torch.float32, "3000 short sequences")
