"""Helpers for the GPU parity tests: run the CUDA path and the CPU oracle on the same inputs."""
from __future__ import annotations

import os
from typing import Optional

import numpy as np
import torch

# Acceptance bounds, written out here: bf16 output max-abs 1e-2 and relative
# Frobenius 5e-3 against the fp64 oracle; fp32 final state relative Frobenius
# 1e-3; a bf16 final state carries its own rounding (about 1.1e-3 relative
# Frobenius for RNE to 8 mantissa bits), so it gets the output's 5e-3 bound.
OUT_MAX_ABS = 1e-2
OUT_REL_FRO = 5e-3
STATE_REL_FRO_FP32 = 1e-3
STATE_REL_FRO_BF16 = 5e-3


def to_device(x: dict, device="cuda") -> dict:
    y = {}
    for k, v in x.items():
        y[k] = v.to(device) if isinstance(v, torch.Tensor) else v
    return y


def to_cpu(x: dict) -> dict:
    return to_device(x, "cpu")


def run_gpu(x: dict, final_dtype: Optional[torch.dtype] = torch.float32, out=None, final_state=None,
            workspace=None):
    """Call the CUDA path through the Python binding of the C ABI."""
    from gated_delta_rule_51_gb300 import kda

    q = x["q"]
    B, T, H, K = q.shape
    cu = x.get("cu_seqlens")
    N = cu.numel() - 1 if cu is not None else B
    V = x["v"].shape[-1]
    if out is None:
        out = torch.full((B, T, H, V), float("nan"), dtype=torch.bfloat16, device=q.device)
    init = x.get("initial_state")
    if final_state is None and final_dtype is not None:
        fd = init.dtype if init is not None else final_dtype
        final_state = torch.full((N, H, V, K), float("nan"), dtype=fd, device=q.device)
    kda.fwd(q, x["k"], x["v"], x["g"], x["beta"], x["scale"], out, x["A_log"], x["dt_bias"],
            x["lower_bound"], initial_state=init, final_state=final_state, cu_seqlens=cu,
            workspace=workspace)
    torch.cuda.synchronize()
    return out, final_state


def run_oracle(x: dict, out_rows=None, want_out=True):
    import oracle

    xc = to_cpu(x)
    return oracle.kda_forward(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["scale"], xc["A_log"],
                              xc["dt_bias"], xc["lower_bound"], xc.get("initial_state"),
                              xc.get("cu_seqlens"), out_rows=out_rows, want_out=want_out,
                              nthreads=os.cpu_count())


def _report(label: str, what: str, value: float) -> None:
    """With KDA_TEST_REPORT naming a file, append the measured error to it (tab-separated)."""
    path = os.environ.get("KDA_TEST_REPORT")
    if not path:
        return
    d = os.path.dirname(os.path.abspath(path))
    os.makedirs(d, exist_ok=True)
    with open(path, "a") as f:
        f.write(f"{label}\t{what}\t{value:.3e}\n")


def rel_fro(a: np.ndarray, b: np.ndarray) -> float:
    d = np.linalg.norm((np.asarray(a, np.float64) - np.asarray(b, np.float64)).ravel())
    n = np.linalg.norm(np.asarray(b, np.float64).ravel())
    return float(d / n) if n > 0 else float(d)


def check_out(gpu_out: torch.Tensor, ref: np.ndarray, rows=None, label=""):
    g = gpu_out.float().cpu().reshape(-1, gpu_out.shape[-2], gpu_out.shape[-1]).double().numpy()
    if rows is not None:
        g = g[np.asarray(rows)]
    assert np.all(np.isfinite(g)), f"{label}: non-finite output"
    max_abs = float(np.abs(g - ref).max()) if ref.size else 0.0
    rf = rel_fro(g, ref) if ref.size else 0.0
    _report(label, "out_max_abs", max_abs)
    _report(label, "out_rel_fro", rf)
    assert max_abs <= OUT_MAX_ABS, f"{label}: out max-abs {max_abs:.3e} > {OUT_MAX_ABS}"
    assert rf <= OUT_REL_FRO, f"{label}: out rel-Fro {rf:.3e} > {OUT_REL_FRO}"
    return max_abs, rf


def check_state(gpu_state: torch.Tensor, ref: np.ndarray, label=""):
    g = gpu_state.float().cpu().double().numpy()
    assert np.all(np.isfinite(g)), f"{label}: non-finite state"
    rf = rel_fro(g, ref)
    bound = STATE_REL_FRO_BF16 if gpu_state.dtype == torch.bfloat16 else STATE_REL_FRO_FP32
    _report(label, f"state_rel_fro_{str(gpu_state.dtype).replace('torch.', '')}", rf)
    assert rf <= bound, f"{label}: state rel-Fro {rf:.3e} > {bound}"
    return rf


def random_case(B, T, H, seed, lens=None, lb=-5.0, init_dtype=torch.float32, device="cuda", V=128, K=128):
    """Inputs in the workloads' distributions (N(0,1) bf16, gate params as the recipes)."""
    from gated_delta_rule_51_gb300 import inputs as I

    w = I.custom_workload("case", B, T, H, lens, init_dtype, init_dtype is not None, True, lb, seed, V=V, K=K)
    return I.make_inputs(w, device=device)
