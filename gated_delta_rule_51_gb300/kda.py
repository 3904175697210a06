"""Python binding of the KDA forward library (``include/kda.h``).

Argument marshalling only: every step of the forward pass runs in the CUDA
kernels of ``libkda.so``; PyTorch provides device memory and the stream.  There
is no CPU or framework fallback -- if the library cannot be loaded, or the GPU
is not an sm_103 part, the calls raise.

``fwd`` mirrors FlashKDA's ``flash_kda.fwd(q, k, v, g, beta, scale, out,
A_log, dt_bias, lower_bound, initial_state=None, final_state=None,
cu_seqlens=None)`` (README "Kernel API").
"""
from __future__ import annotations

import ctypes
import threading
from typing import Dict, Optional, Tuple

import torch

from . import _build

KDA_OK = 0
KDA_STATE_NONE, KDA_STATE_BF16, KDA_STATE_FP32 = 0, 1, 2
STATUS_NAMES = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARGUMENT", 2: "KDA_ERR_UNSUPPORTED_SHAPE",
                3: "KDA_ERR_WORKSPACE_TOO_SMALL", 4: "KDA_ERR_UNSUPPORTED_DEVICE", 5: "KDA_ERR_CUDA",
                6: "KDA_ERR_TIMEOUT", 7: "KDA_ERR_BAD_SEQLENS", 8: "KDA_ERR_GATE_RANGE"}
EXPORTED_SYMBOLS = ("kda_status_string", "kda_workspace_size", "kda_fwd", "kda_check_device_error",
                    "kda_set_profile_events", "kda_last_launch_count", "kda_fwd_static_workspace",
                    "kda_decode", "kda_fwd_ex", "kda_bwd_workspace_size", "kda_bwd")
KDA_GATE_PREACTIVATED, KDA_BETA_PREACTIVATED, KDA_NO_QK_L2NORM, KDA_GATE_SOFTPLUS = 1, 2, 4, 8
KDA_PRECISE_STATE = 16
KDA_BWD_RECURRENT = 32


class kda_shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("B", "T", "H", "K", "V", "N")]


class KDAError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")
        self.status = status


_lib = None
_lib_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load (building first if needed) the in-tree libkda.so and declare its C ABI."""
    global _lib
    with _lib_lock:
        if _lib is not None:
            return _lib
        path = _build.build() if build_if_missing else _build.LIB
        lib = ctypes.CDLL(path)
        p, i64 = ctypes.c_void_p, ctypes.c_int64
        lib.kda_status_string.argtypes = [ctypes.c_int]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_workspace_size.argtypes = [ctypes.POINTER(kda_shape), ctypes.POINTER(ctypes.c_size_t)]
        lib.kda_workspace_size.restype = ctypes.c_int
        lib.kda_fwd.argtypes = [ctypes.POINTER(kda_shape), p, p, p, p, p, ctypes.c_float, p, p, p,
                                ctypes.c_float, p, ctypes.c_int, p, ctypes.c_int, p, p, ctypes.c_size_t, p]
        lib.kda_fwd.restype = ctypes.c_int
        lib.kda_check_device_error.argtypes = [p, p, ctypes.POINTER(ctypes.c_int)]
        lib.kda_check_device_error.restype = ctypes.c_int
        lib.kda_set_profile_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]
        lib.kda_set_profile_events.restype = ctypes.c_int
        lib.kda_last_launch_count.argtypes = []
        lib.kda_last_launch_count.restype = ctypes.c_int
        lib.kda_decode.argtypes = [ctypes.POINTER(kda_shape), p, p, p, p, p, ctypes.c_float, p, p, p,
                                   ctypes.c_float, p, ctypes.c_int, ctypes.c_uint, p]
        lib.kda_fwd_ex.argtypes = [ctypes.POINTER(kda_shape), p, p, p, p, p, ctypes.c_float, p, p, p,
                                   ctypes.c_float, p, ctypes.c_int, p, ctypes.c_int, p, ctypes.c_uint, p,
                                   ctypes.c_size_t, p]
        lib.kda_fwd_ex.restype = ctypes.c_int
        lib.kda_decode.restype = ctypes.c_int
        lib.kda_bwd_workspace_size.argtypes = [ctypes.POINTER(kda_shape), ctypes.POINTER(ctypes.c_size_t)]
        lib.kda_bwd_workspace_size.restype = ctypes.c_int
        lib.kda_bwd.argtypes = [ctypes.POINTER(kda_shape), p, p, p, p, p, ctypes.c_float, p, p, ctypes.c_float,
                                p, ctypes.c_int, p, p, p, p, p, p, p, p, p, p, p, ctypes.c_uint, p,
                                ctypes.c_size_t, p]
        lib.kda_bwd.restype = ctypes.c_int
        _lib = lib
        return lib


def make_shape(B: int, T: int, H: int, N: int, K: int = 128, V: int = 128) -> kda_shape:
    return kda_shape(B, T, H, K, V, N)


def workspace_size(shape: kda_shape) -> int:
    lib = load_library()
    n = ctypes.c_size_t(0)
    st = lib.kda_workspace_size(ctypes.byref(shape), ctypes.byref(n))
    if st != KDA_OK:
        raise KDAError(st, "kda_workspace_size")
    return int(n.value)


_workspaces: Dict[Tuple[int, int], torch.Tensor] = {}


def _workspace(device: torch.device, stream: int, nbytes: int) -> torch.Tensor:
    key = (device.index, stream)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _state_code(t: Optional[torch.Tensor]) -> int:
    if t is None:
        return KDA_STATE_NONE
    if t.dtype == torch.bfloat16:
        return KDA_STATE_BF16
    if t.dtype == torch.float32:
        return KDA_STATE_FP32
    raise TypeError(f"state dtype must be bf16 or fp32, got {t.dtype}")


def _check(t: torch.Tensor, name: str, dtype: torch.dtype, shape: Tuple[int, ...], device):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _flags(use_gate_in_kernel: bool, use_beta_sigmoid_in_kernel: bool, use_qk_l2norm_in_kernel: bool,
           safe_gate: bool = True) -> int:
    if not safe_gate and not use_gate_in_kernel:
        raise ValueError("safe_gate=False selects the in-kernel gate without a lower bound; "
                         "it needs use_gate_in_kernel=True")
    return ((0 if use_gate_in_kernel else KDA_GATE_PREACTIVATED)
            | (0 if use_beta_sigmoid_in_kernel else KDA_BETA_PREACTIVATED)
            | (0 if use_qk_l2norm_in_kernel else KDA_NO_QK_L2NORM)
            | (0 if safe_gate else KDA_GATE_SOFTPLUS))


def fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state=None,
        final_state=None, cu_seqlens=None, workspace: Optional[torch.Tensor] = None,
        stream: Optional[torch.cuda.Stream] = None, use_gate_in_kernel: bool = True,
        use_beta_sigmoid_in_kernel: bool = True, use_qk_l2norm_in_kernel: bool = True,
        safe_gate: bool = True, precise_state: bool = False):
    """KDA forward on the GPU; writes ``out`` (and ``final_state``) and returns them.

    q, k, g: [B,T,H,K] bf16 with K = 64 or 128; v, out: [B,T,H,V] bf16 with V = 64, 128
    or 256; beta: [B,T,H] bf16 logits; A_log: [H] fp32; dt_bias: [H,K] fp32 (16-byte
    aligned); states: [N,H,V,K] bf16/fp32 or None;
    cu_seqlens: int64 [N+1] on the device (then B must be 1).
    The use_* switches (default on, FlashKDA's behaviour) say which steps run in
    the kernel; off means the caller did them: g is then the natural-log decay, at
    most 0 (A_log and dt_bias may be None), beta is beta itself, q and k are used
    without L2 norms.  safe_gate=False selects the gate without a lower bound,
    ghat = -exp(A_log) softplus(g + dt_bias) (lower_bound is then not read).  Any
    decay is computed exactly: chunks past 2^-250 take a direct route in the kernel.
    precise_state=True reads the carried state as a bf16 pair (KDA_PRECISE_STATE); the
    library already does so for lower_bound > -0.25 and for the two gates without a bound.
    """
    if q.dim() != 4:
        raise ValueError("q must be [B, T, H, K]")
    B, T, H, K = q.shape
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("kda.fwd runs on CUDA tensors only")
    V = v.shape[-1]
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else B
    for name, t, dt, shp in (("q", q, torch.bfloat16, (B, T, H, K)), ("k", k, torch.bfloat16, (B, T, H, K)),
                             ("g", g, torch.bfloat16, (B, T, H, K)), ("v", v, torch.bfloat16, (B, T, H, V)),
                             ("out", out, torch.bfloat16, (B, T, H, V)),
                             ("beta", beta, torch.bfloat16, (B, T, H)),
                             ("A_log", A_log, torch.float32, (H,)), ("dt_bias", dt_bias, torch.float32, (H, K))):
        if t is None and not use_gate_in_kernel and name in ("A_log", "dt_bias"):
            continue
        _check(t, name, dt, shp, dev)
    flags = _flags(use_gate_in_kernel, use_beta_sigmoid_in_kernel, use_qk_l2norm_in_kernel, safe_gate)
    if precise_state:
        flags |= KDA_PRECISE_STATE
    for name, t in (("initial_state", initial_state), ("final_state", final_state)):
        if t is not None:
            _check(t, name, t.dtype, (N, H, V, K), dev)
    if cu_seqlens is not None:
        _check(cu_seqlens, "cu_seqlens", torch.int64, (N + 1,), dev)
    lib = load_library()
    shape = make_shape(B, T, H, N, K, V)
    need = workspace_size(shape)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    if workspace is None:
        workspace = _workspace(dev, s.cuda_stream, need)
    elif workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace needs {need} bytes")
    st = lib.kda_fwd_ex(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                        ctypes.c_float(scale), _ptr(out), _ptr(A_log), _ptr(dt_bias),
                        ctypes.c_float(lower_bound), _ptr(initial_state), _state_code(initial_state),
                        _ptr(final_state), _state_code(final_state), _ptr(cu_seqlens), ctypes.c_uint(flags),
                        _ptr(workspace), ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                        ctypes.c_void_p(s.cuda_stream))
    if st != KDA_OK:
        raise KDAError(st, "kda_fwd")
    return out, final_state


def decode(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, state,
           stream: Optional[torch.cuda.Stream] = None, use_gate_in_kernel: bool = True,
           use_beta_sigmoid_in_kernel: bool = True, use_qk_l2norm_in_kernel: bool = True,
           safe_gate: bool = True):
    """Recurrent KDA step(s) for decoding; updates ``state`` in place, writes ``out``.

    q, k, g: [B,T,H,K] bf16 with K = 64 or 128; v, out: [B,T,H,V] bf16 with V = 64, 128
    or 256 (T new tokens per sequence, usually 1); beta: [B,T,H] bf16 logits; A_log: [H]
    fp32; dt_bias: [H,K] fp32; state: [B,H,V,K] bf16 or fp32, read before the first
    token and overwritten.  The switches are those of fwd.
    """
    if q.dim() != 4:
        raise ValueError("q must be [B, T, H, K]")
    B, T, H, K = q.shape
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("kda.decode runs on CUDA tensors only")
    V = v.shape[-1]
    for name, t, dt, shp in (("q", q, torch.bfloat16, (B, T, H, K)), ("k", k, torch.bfloat16, (B, T, H, K)),
                             ("g", g, torch.bfloat16, (B, T, H, K)), ("v", v, torch.bfloat16, (B, T, H, V)),
                             ("out", out, torch.bfloat16, (B, T, H, V)),
                             ("beta", beta, torch.bfloat16, (B, T, H)),
                             ("A_log", A_log, torch.float32, (H,)), ("dt_bias", dt_bias, torch.float32, (H, K))):
        if t is None and not use_gate_in_kernel and name in ("A_log", "dt_bias"):
            continue
        _check(t, name, dt, shp, dev)
    _check(state, "state", state.dtype, (B, H, V, K), dev)
    flags = _flags(use_gate_in_kernel, use_beta_sigmoid_in_kernel, use_qk_l2norm_in_kernel, safe_gate)
    lib = load_library()
    shape = make_shape(B, T, H, B, K, V)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    st = lib.kda_decode(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                        ctypes.c_float(scale), _ptr(out), _ptr(A_log), _ptr(dt_bias), ctypes.c_float(lower_bound),
                        _ptr(state), _state_code(state), ctypes.c_uint(flags), ctypes.c_void_p(s.cuda_stream))
    if st != KDA_OK:
        raise KDAError(st, "kda_decode")
    return out, state


def check_device_error(workspace: Optional[torch.Tensor] = None, device=None) -> int:
    """Synchronise and return the device error flags left by the last fwd on this workspace."""
    lib = load_library()
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    s = torch.cuda.current_stream(dev)
    if workspace is None:
        workspace = _workspaces.get((dev.index, s.cuda_stream))
        if workspace is None:
            return 0
    flags = ctypes.c_int(0)
    lib.kda_check_device_error(_ptr(workspace), ctypes.c_void_p(s.cuda_stream), ctypes.byref(flags))
    return int(flags.value)


def raise_on_device_error(flags: int, what: str) -> None:
    """Raise KDAError for a nonzero device error word (the bits of kda_check_device_error)."""
    if flags & 1:
        raise KDAError(6, what)
    if flags & 2:
        raise KDAError(7, what)
    if flags & 4:
        raise KDAError(8, what)


def set_profile_events(events) -> None:
    """Record the given 4 torch.cuda.Events after each launch phase of fwd (None to stop)."""
    lib = load_library()
    if events is None:
        lib.kda_set_profile_events(None, 0)
        return
    arr = (ctypes.c_void_p * 4)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    st = lib.kda_set_profile_events(arr, 4)
    if st != KDA_OK:
        raise KDAError(st, "kda_set_profile_events")


def last_launch_count() -> int:
    """Kernels enqueued by this thread's most recent fwd call."""
    return int(load_library().kda_last_launch_count())


def bwd_workspace_size(shape: kda_shape) -> int:
    lib = load_library()
    n = ctypes.c_size_t(0)
    st = lib.kda_bwd_workspace_size(ctypes.byref(shape), ctypes.byref(n))
    if st != KDA_OK:
        raise KDAError(st, "kda_bwd_workspace_size")
    return int(n.value)


def bwd(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, dout, initial_state=None, dfinal=None,
        cu_seqlens=None, workspace: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
        use_gate_in_kernel: bool = True, use_beta_sigmoid_in_kernel: bool = True,
        use_qk_l2norm_in_kernel: bool = True, safe_gate: bool = True, out: Optional[dict] = None,
        recurrent: bool = False) -> dict:
    """Gradients of sum(dout * out) + sum(dfinal * final_state) for the forward fwd() computes
    with the same arguments (K = V = 128).  dout: bf16 [B,T,H,128]; dfinal: fp32 [N,H,128,128]
    or None.  Returns fp32 tensors dq, dk, dg [B,T,H,128], dv [B,T,H,128], dbeta [B,T,H],
    dh0 [N,H,128,128], dA_log [H] and ddt_bias [H,128] (allocated here unless ``out`` holds
    them).  dg is the gradient for the raw g passed in; dbeta for the beta logits.
    recurrent=True asks for the fp32 token recurrence (KDA_BWD_RECURRENT) instead of the
    chunked tensor-core form the gate with a lower bound takes by default."""
    if q.dim() != 4:
        raise ValueError("q must be [B, T, H, K]")
    B, T, H, K = q.shape
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("kda.bwd needs CUDA tensors")
    N = cu_seqlens.numel() - 1 if cu_seqlens is not None else B
    V = v.shape[-1]
    flags = _flags(use_gate_in_kernel, use_beta_sigmoid_in_kernel, use_qk_l2norm_in_kernel, safe_gate)
    if recurrent:
        flags |= KDA_BWD_RECURRENT
    for name, t, dt, shp in (("q", q, torch.bfloat16, (B, T, H, K)), ("k", k, torch.bfloat16, (B, T, H, K)),
                             ("g", g, torch.bfloat16, (B, T, H, K)), ("v", v, torch.bfloat16, (B, T, H, V)),
                             ("beta", beta, torch.bfloat16, (B, T, H)), ("dout", dout, torch.bfloat16, (B, T, H, V))):
        _check(t, name, dt, shp, dev)
    if use_gate_in_kernel:
        _check(A_log, "A_log", torch.float32, (H,), dev)
        _check(dt_bias, "dt_bias", torch.float32, (H, K), dev)
    if initial_state is not None:
        _check(initial_state, "initial_state", initial_state.dtype, (N, H, V, K), dev)
    if dfinal is not None:
        _check(dfinal, "dfinal", torch.float32, (N, H, V, K), dev)
    if cu_seqlens is not None:
        _check(cu_seqlens, "cu_seqlens", torch.int64, (N + 1,), dev)
    f32 = dict(dtype=torch.float32, device=dev)
    r = out if out is not None else dict(
        dq=torch.empty((B, T, H, K), **f32), dk=torch.empty((B, T, H, K), **f32),
        dv=torch.empty((B, T, H, V), **f32), dg=torch.empty((B, T, H, K), **f32),
        dbeta=torch.empty((B, T, H), **f32), dh0=torch.empty((N, H, V, K), **f32),
        dA_log=torch.empty((H,), **f32), ddt_bias=torch.empty((H, K), **f32))
    shape = make_shape(B, T, H, N, K, V)
    lib = load_library()
    n = ctypes.c_size_t(0)
    st = lib.kda_bwd_workspace_size(ctypes.byref(shape), ctypes.byref(n))
    if st != KDA_OK:
        raise KDAError(st, "kda_bwd_workspace_size")
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    if workspace is None:
        workspace = torch.empty(max(int(n.value), 256), dtype=torch.uint8, device=dev)
    st = lib.kda_bwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), ctypes.c_float(scale),
                     _ptr(A_log), _ptr(dt_bias), ctypes.c_float(lower_bound), _ptr(initial_state),
                     _state_code(initial_state), _ptr(cu_seqlens), _ptr(dout), _ptr(dfinal), _ptr(r["dq"]),
                     _ptr(r["dk"]), _ptr(r["dv"]), _ptr(r["dg"]), _ptr(r["dbeta"]), _ptr(r.get("dh0")),
                     _ptr(r.get("dA_log")), _ptr(r.get("ddt_bias")), ctypes.c_uint(flags), _ptr(workspace),
                     ctypes.c_size_t(workspace.numel()), ctypes.c_void_p(s.cuda_stream))
    if st != KDA_OK:
        raise KDAError(st, "kda_bwd")
    return r


class KDAFunction(torch.autograd.Function):
    """KDA as an autograd operation: forward through kda_fwd_ex, backward through kda_bwd
    (K = V = 128 for gradients).  Inputs: q, k, v, g, beta (bf16), A_log, dt_bias (fp32),
    initial_state (bf16/fp32 or None), cu_seqlens (int64 or None), then the scalars and
    switches.  Outputs: out (bf16) and final_state (the initial state's dtype, fp32 when
    there is none).  Gradients come back in each input's dtype."""

    @staticmethod
    def forward(ctx, q, k, v, g, beta, A_log, dt_bias, initial_state, cu_seqlens, scale, lower_bound,
                use_gate_in_kernel, use_beta_sigmoid_in_kernel, use_qk_l2norm_in_kernel, safe_gate,
                check_errors=False, recurrent_backward=False):
        B, T, H, K = q.shape
        N = cu_seqlens.numel() - 1 if cu_seqlens is not None else B
        V = v.shape[-1]
        # the backward (kda_bwd) takes K = V = 128 only: refuse before the forward runs rather
        # than fail inside loss.backward()
        if any(ctx.needs_input_grad) and (K != 128 or V != 128):
            raise ValueError(f"gradients need K = V = 128 (got K = {K}, V = {V}); run the forward "
                             "without requires_grad for the other head dimensions")
        out = torch.empty((B, T, H, V), dtype=torch.bfloat16, device=q.device)
        fdt = initial_state.dtype if initial_state is not None else torch.float32
        final_state = torch.empty((N, H, V, K), dtype=fdt, device=q.device)
        sw = dict(use_gate_in_kernel=use_gate_in_kernel, use_beta_sigmoid_in_kernel=use_beta_sigmoid_in_kernel,
                  use_qk_l2norm_in_kernel=use_qk_l2norm_in_kernel, safe_gate=safe_gate)
        fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state=initial_state,
            final_state=final_state, cu_seqlens=cu_seqlens, **sw)
        if check_errors:
            raise_on_device_error(check_device_error(device=q.device), "kda_fwd")
        ctx.save_for_backward(q, k, v, g, beta, A_log, dt_bias, initial_state, cu_seqlens)
        ctx.set_materialize_grads(False)   # an unused output's gradient arrives as None
        ctx.scalars = (scale, lower_bound)
        ctx.switches = sw
        ctx.check_errors = check_errors
        ctx.recurrent = recurrent_backward
        return out, final_state

    @staticmethod
    def backward(ctx, dout, dfinal):
        q, k, v, g, beta, A_log, dt_bias, initial_state, cu_seqlens = ctx.saved_tensors
        scale, lower_bound = ctx.scalars
        if dout is None:
            dout = torch.zeros(v.shape, dtype=torch.bfloat16, device=q.device)
        ws = None
        if ctx.check_errors:   # a workspace of our own, so that its error word can be read afterwards
            B, T, H, K = q.shape
            N = cu_seqlens.numel() - 1 if cu_seqlens is not None else B
            ws = torch.empty(max(bwd_workspace_size(make_shape(B, T, H, N, K, v.shape[-1])), 256),
                             dtype=torch.uint8, device=q.device)
        r = bwd(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, dout.to(torch.bfloat16).contiguous(),
                initial_state=initial_state,
                dfinal=None if dfinal is None else dfinal.to(torch.float32).contiguous(),
                cu_seqlens=cu_seqlens, workspace=ws, recurrent=ctx.recurrent, **ctx.switches)
        if ctx.check_errors:
            raise_on_device_error(check_device_error(workspace=ws, device=q.device), "kda_bwd")
        gate = ctx.switches["use_gate_in_kernel"]

        def cast(t, like):
            return None if like is None else t.to(like.dtype)

        return (cast(r["dq"], q), cast(r["dk"], k), cast(r["dv"], v), cast(r["dg"], g), cast(r["dbeta"], beta),
                cast(r["dA_log"], A_log) if gate else None, cast(r["ddt_bias"], dt_bias) if gate else None,
                cast(r["dh0"], initial_state), None, None, None, None, None, None, None, None, None)


def kda_attention(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, initial_state=None, cu_seqlens=None,
                  use_gate_in_kernel: bool = True, use_beta_sigmoid_in_kernel: bool = True,
                  use_qk_l2norm_in_kernel: bool = True, safe_gate: bool = True, check_errors: bool = False,
                  recurrent_backward: bool = False):
    """The forward with autograd: returns (out, final_state); gradients flow to q, k, v, g,
    beta, A_log, dt_bias and initial_state through the CUDA backward (K = V = 128; other
    head dimensions are refused when an input requires grad).

    The kernels report malformed cu_seqlens, a gate whose decay leaves the chunked form's
    range and timed-out waits through an error word, not an exception.  With
    check_errors=True the forward and the backward each synchronise and raise KDAError when
    that word is set; otherwise the caller validates cu_seqlens (and, for the gates without a
    lower bound, the decay range) itself.  The backward takes the chunked tensor-core form for
    the gate with a lower bound (gradients within 1e-2 relative Frobenius of the exact ones);
    recurrent_backward=True asks for the fp32 token recurrence instead."""
    return KDAFunction.apply(q, k, v, g, beta, A_log, dt_bias, initial_state, cu_seqlens, scale, lower_bound,
                             use_gate_in_kernel, use_beta_sigmoid_in_kernel, use_qk_l2norm_in_kernel, safe_gate,
                             check_errors, recurrent_backward)
