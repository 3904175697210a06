"""CPU oracle for the KDA forward pass and its gradient -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never imports, links or calls anything here.

Contents:
  * ``kda_oracle.c``  -- plain fp64 token-by-token recurrence (the definition),
    threaded over (sequence, head) pairs; built with gcc by ``build()``.
  * ``kda_oracle_bwd.c`` -- the same recurrence on fp64 inputs and its gradient (the
    chain rule applied to each token step in reverse), built into the same library.
  * ``token_np.py``   -- a NumPy twin of the same definition for tiny inputs.
  * ``chunked_np.py`` -- the 16-token chunked (WY/UT) form of the method in
    NumPy fp64, used to pin the token form and to study rounding.
  * ``chunked_bwd_np.py`` -- the gradient through that chunked form (dense per-chunk
    products, the shape a tensor-core backward takes), pinned to the token gradient.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_SRC_BWD = os.path.join(_HERE, "kda_oracle_bwd.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (portable flags, no -march) and return its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_SRC_BWD))
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-ffp-contract=off", _SRC, _SRC_BWD, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            fn = lib.kda_oracle_fwd
            i64, p = ctypes.c_int64, ctypes.c_void_p
            fn.argtypes = [i64, i64, i64, i64, i64, i64, ctypes.c_int, p, p, p, p, p, ctypes.c_double, p, p,
                           ctypes.c_double, p, p, p, p, p, ctypes.c_int]
            fn.restype = ctypes.c_int
            fn = lib.kda_oracle_fwd64
            fn.argtypes = [i64, i64, i64, i64, i64, i64, ctypes.c_int, p, p, p, p, p, ctypes.c_double, p, p,
                           ctypes.c_double, p, p, p, p, ctypes.c_int]
            fn.restype = ctypes.c_int
            fn = lib.kda_oracle_bwd
            fn.argtypes = [i64, i64, i64, i64, i64, i64, ctypes.c_int, p, p, p, p, p, ctypes.c_double, p, p,
                           ctypes.c_double, p, p, p, p, p, p, p, p, p, p, p, p, ctypes.c_int]
            fn.restype = ctypes.c_int
            _lib = lib
    return _lib


def _bits(x) -> np.ndarray:
    """bf16 tensor/array -> contiguous uint16 bit patterns."""
    import torch  # local: the oracle itself needs only numpy

    if isinstance(x, torch.Tensor):
        assert x.dtype == torch.bfloat16
        return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy()
                                    .view(np.uint16))
    x = np.asarray(x)
    assert x.dtype == np.uint16
    return np.ascontiguousarray(x)


def _f64(x) -> Optional[np.ndarray]:
    import torch

    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return np.ascontiguousarray(x.detach().cpu().to(torch.float64).numpy())
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _f32(x) -> np.ndarray:
    import torch

    if isinstance(x, torch.Tensor):
        return np.ascontiguousarray(x.detach().cpu().to(torch.float32).numpy())
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def kda_forward(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, initial_state=None,
                cu_seqlens=None, out_rows=None, want_out=True, want_final_state=True,
                nthreads: Optional[int] = None, use_gate_in_kernel: bool = True,
                use_beta_sigmoid_in_kernel: bool = True, use_qk_l2norm_in_kernel: bool = True,
                safe_gate: bool = True):
    """Run the fp64 token recurrence.

    q, k, g: [B,T,H,K] bf16; v: [B,T,H,V] bf16; beta: [B,T,H] bf16 (torch
    tensors or uint16 bit arrays); A_log [H] and dt_bias [H,K] fp32; scale and
    lower_bound are rounded to fp32 first, as they cross the C ABI as floats.
    initial_state: [N,H,V,K] of any float dtype (converted exactly) or None.
    out_rows: optional sorted token-row indices (over B*T) whose outputs are
    wanted; default all rows.  Returns (out [rows,H,V] fp64 or None,
    final_state [N,H,V,K] fp64 or None).
    The three use_* switches mirror the reference call's flags: when False, g
    already holds the natural-log decay (A_log, dt_bias and lower_bound are then
    unused), beta already holds beta, or q and k are used without L2 norms.
    safe_gate=False selects the gate without a lower bound,
    ghat = -exp(A_log) * softplus(g + dt_bias) (lower_bound unused); it needs
    use_gate_in_kernel=True.
    """
    if not safe_gate and not use_gate_in_kernel:
        raise ValueError("safe_gate=False applies to the in-kernel gate only")
    qb, kb, vb, gb, bb = (_bits(x) for x in (q, k, v, g, beta))
    B, T, H, K = qb.shape
    V = vb.shape[-1]
    cu = None
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
            dtype=np.int64))
        N = cu.shape[0] - 1
    else:
        N = B
    A = _f32(A_log)
    D = _f32(dt_bias)
    s0 = _f64(initial_state)
    out = row_map = None
    if want_out:
        if out_rows is None:
            out = np.zeros((B * T, H, V), dtype=np.float64)
        else:
            rows = np.asarray(out_rows, dtype=np.int64)
            row_map = np.full(B * T, -1, dtype=np.int64)
            row_map[rows] = np.arange(rows.shape[0], dtype=np.int64)
            out = np.zeros((rows.shape[0], H, V), dtype=np.float64)
    fin = np.zeros((N, H, V, K), dtype=np.float64) if want_final_state else None
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    flags = ((0 if use_gate_in_kernel else 1) | (0 if use_beta_sigmoid_in_kernel else 2)
             | (0 if use_qk_l2norm_in_kernel else 4) | (0 if safe_gate else 8))
    rc = _load().kda_oracle_fwd(B, T, H, K, V, N, flags, _ptr(qb), _ptr(kb), _ptr(vb), _ptr(gb),
                                _ptr(bb), float(np.float32(scale)), _ptr(A), _ptr(D),
                                float(np.float32(lower_bound)), _ptr(s0), _ptr(out),
                                _ptr(row_map), _ptr(fin), _ptr(cu), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_fwd failed with code {rc}")
    return out, fin


def _flags(use_gate_in_kernel, use_beta_sigmoid_in_kernel, use_qk_l2norm_in_kernel, safe_gate) -> int:
    if not safe_gate and not use_gate_in_kernel:
        raise ValueError("safe_gate=False applies to the in-kernel gate only")
    return ((0 if use_gate_in_kernel else 1) | (0 if use_beta_sigmoid_in_kernel else 2)
            | (0 if use_qk_l2norm_in_kernel else 4) | (0 if safe_gate else 8))


def _cu(cu_seqlens):
    if cu_seqlens is None:
        return None
    return np.ascontiguousarray(np.asarray(
        cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64))


def kda_forward64(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, initial_state=None,
                  cu_seqlens=None, nthreads: Optional[int] = None, use_gate_in_kernel: bool = True,
                  use_beta_sigmoid_in_kernel: bool = True, use_qk_l2norm_in_kernel: bool = True,
                  safe_gate: bool = True):
    """The forward recurrence on fp64 inputs (any float arrays, converted to fp64; scale and
    lower_bound used as given).  Returns (out [B,T,H,V], final_state [N,H,V,K]), fp64."""
    flags = _flags(use_gate_in_kernel, use_beta_sigmoid_in_kernel, use_qk_l2norm_in_kernel, safe_gate)
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    B, T, H, K = q.shape
    V = v.shape[-1]
    cu = _cu(cu_seqlens)
    N = cu.shape[0] - 1 if cu is not None else B
    A = _f64(A_log) if A_log is not None else np.zeros(H)
    D = _f64(dt_bias) if dt_bias is not None else np.zeros((H, K))
    out = np.zeros((B, T, H, V), dtype=np.float64)
    fin = np.zeros((N, H, V, K), dtype=np.float64)
    rc = _load().kda_oracle_fwd64(B, T, H, K, V, N, flags, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                  float(scale), _ptr(A), _ptr(D), float(lower_bound), _ptr(_f64(initial_state)),
                                  _ptr(cu), _ptr(out), _ptr(fin), int(nthreads or os.cpu_count() or 1))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_fwd64 failed with code {rc}")
    return out, fin


def kda_backward(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, dout, initial_state=None,
                 dfinal=None, cu_seqlens=None, nthreads: Optional[int] = None, use_gate_in_kernel: bool = True,
                 use_beta_sigmoid_in_kernel: bool = True, use_qk_l2norm_in_kernel: bool = True,
                 safe_gate: bool = True):
    """Gradient of L = sum(dout * out) + sum(dfinal * final_state) with respect to the
    forward's inputs, in fp64.  Inputs as kda_forward64 plus dout [B,T,H,V] and dfinal
    [N,H,V,K] (None: the final state is not part of L).  Returns a dict with dq, dk, dg
    [B,T,H,K], dv [B,T,H,V], dbeta [B,T,H] (with respect to the logits unless beta is
    pre-activated), dh0 [N,H,V,K], dA_log [H] and ddt_bias [H,K]."""
    flags = _flags(use_gate_in_kernel, use_beta_sigmoid_in_kernel, use_qk_l2norm_in_kernel, safe_gate)
    q, k, v, g, beta, dout = (_f64(x) for x in (q, k, v, g, beta, dout))
    B, T, H, K = q.shape
    V = v.shape[-1]
    cu = _cu(cu_seqlens)
    N = cu.shape[0] - 1 if cu is not None else B
    A = _f64(A_log) if A_log is not None else np.zeros(H)
    D = _f64(dt_bias) if dt_bias is not None else np.zeros((H, K))
    r = dict(dq=np.zeros((B, T, H, K)), dk=np.zeros((B, T, H, K)), dv=np.zeros((B, T, H, V)),
             dg=np.zeros((B, T, H, K)), dbeta=np.zeros((B, T, H)), dh0=np.zeros((N, H, V, K)),
             dA_log=np.zeros(H), ddt_bias=np.zeros((H, K)))
    rc = _load().kda_oracle_bwd(B, T, H, K, V, N, flags, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                float(scale), _ptr(A), _ptr(D), float(lower_bound), _ptr(_f64(initial_state)),
                                _ptr(cu), _ptr(dout), _ptr(_f64(dfinal)), _ptr(r["dq"]), _ptr(r["dk"]),
                                _ptr(r["dv"]), _ptr(r["dg"]), _ptr(r["dbeta"]), _ptr(r["dh0"]),
                                _ptr(r["dA_log"]), _ptr(r["ddt_bias"]), int(nthreads or os.cpu_count() or 1))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_bwd failed with code {rc}")
    return r
