"""The C ABI without a GPU: the library builds for sm_103a, loads, exports every
symbol include/kda.h declares, and rejects bad arguments on the host before any
CUDA call (fake device addresses are never dereferenced)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from gated_delta_rule_51_gb300 import kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x10000000   # 16-byte aligned fake device address, never dereferenced


def declared_symbols():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"KDA_API\s+[\w\s\*]+?\b(kda_\w+)\s*\(", txt)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    lib = kda.load_library()
    syms = declared_symbols()
    assert set(kda.EXPORTED_SYMBOLS) <= set(syms)
    for s in syms:
        assert hasattr(lib, s), f"{s} not exported"


def test_status_strings():
    lib = kda.load_library()
    for code in range(9):
        s = lib.kda_status_string(code)
        assert s and isinstance(s, bytes)
    assert lib.kda_status_string(0) == b"ok"


def test_workspace_size_linear_in_heads_and_tiles():
    sh = kda.make_shape(1, 1 << 20, 8, 1)
    n8 = kda.workspace_size(sh)
    assert n8 > 0
    lib = kda.load_library()
    n = ctypes.c_size_t(0)
    bad = kda.make_shape(1, 64, 1, 1, K=32)
    assert lib.kda_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == 2
    assert lib.kda_workspace_size(None, ctypes.byref(n)) == 1


def _call(shape, q=FAKE, beta=FAKE, out=FAKE, A_log=FAKE, dt_bias=FAKE, lb=-1.0, scale=0.1,
          init=None, init_dt=0, fin=None, fin_dt=0, cu=None, ws=FAKE, ws_bytes=1 << 30):
    lib = kda.load_library()
    p = ctypes.c_void_p
    return lib.kda_fwd(ctypes.byref(shape), p(q), p(FAKE), p(FAKE), p(FAKE), p(beta),
                       ctypes.c_float(scale), p(out), p(A_log), p(dt_bias), ctypes.c_float(lb),
                       p(init) if init else None, init_dt, p(fin) if fin else None, fin_dt,
                       p(cu) if cu else None, p(ws), ctypes.c_size_t(ws_bytes), None)


@pytest.mark.parametrize("case,expected", [
    (dict(shape=kda.make_shape(1, 64, 1, 1, K=32)), 2),
    (dict(shape=kda.make_shape(1, 64, 1, 1, V=384)), 2),
    (dict(shape=kda.make_shape(2, 64, 1, 2), cu=FAKE), 1),          # cu_seqlens needs B = 1
    (dict(shape=kda.make_shape(2, 64, 1, 3)), 1),                   # N must equal B
    (dict(shape=kda.make_shape(1, 64, 1, 1), lb=0.5), 1),           # lower_bound in [-5, 0]
    (dict(shape=kda.make_shape(1, 64, 1, 1), lb=-5.5), 1),
    (dict(shape=kda.make_shape(1, 64, 1, 1), lb=float("nan")), 1),
    (dict(shape=kda.make_shape(1, 64, 1, 1), q=0), 1),              # null input
    (dict(shape=kda.make_shape(1, 64, 1, 1), q=FAKE + 2), 1),       # misaligned input
    (dict(shape=kda.make_shape(1, 64, 1, 1), out=0), 1),
    (dict(shape=kda.make_shape(1, 64, 1, 1), A_log=0), 1),
    (dict(shape=kda.make_shape(1, 64, 1, 1), dt_bias=FAKE + 4), 1),  # dt_bias is read as float4
    (dict(shape=kda.make_shape(1, 64, 1, 1), init=FAKE, init_dt=1, fin=FAKE + (1 << 24), fin_dt=2), 1),
    (dict(shape=kda.make_shape(1, 64, 1, 1), init=FAKE, init_dt=0), 1),   # dtype missing
    (dict(shape=kda.make_shape(1, 64, 2, 1), init=FAKE, init_dt=2, fin=FAKE + 4096, fin_dt=2), 1),  # overlap
    (dict(shape=kda.make_shape(-1, 64, 1, -1)), 1),
    (dict(shape=kda.make_shape(1, 64, 0, 1)), 1),
])
def test_host_side_argument_errors(case, expected):
    shape = case.pop("shape")
    assert _call(shape, **case) == expected


def test_element_aligned_beta_and_out_pass_the_argument_checks():
    # 2-byte aligned beta/out are valid; without a GPU the call then stops at the
    # device query (KDA_ERR_CUDA or KDA_ERR_UNSUPPORTED_DEVICE), not at the checks
    assert _call(kda.make_shape(1, 64, 1, 1), beta=FAKE + 2, out=FAKE + 6) in (4, 5)


def test_python_binding_rejects_softplus_with_a_preactivated_gate():
    with pytest.raises(ValueError):
        kda._flags(False, True, True, safe_gate=False)
    assert kda._flags(True, True, True, safe_gate=False) == kda.KDA_GATE_SOFTPLUS


def test_python_binding_requires_cuda_tensors():
    import torch

    q = torch.zeros(1, 16, 1, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        kda.fwd(q, q, q, q, torch.zeros(1, 16, 1, dtype=torch.bfloat16), 0.1, q.clone(),
                torch.zeros(1), torch.zeros(1, 128), -1.0)


def _decode_call(shape, q=FAKE, out=FAKE, A_log=FAKE, state=FAKE, dtype=2, lb=-1.0, flags=0):
    lib = kda.load_library()
    p = lambda a: ctypes.c_void_p(a) if a else None
    return lib.kda_decode(ctypes.byref(shape), p(q), p(FAKE), p(FAKE), p(FAKE), p(FAKE), ctypes.c_float(0.1),
                          p(out), p(A_log), p(FAKE), ctypes.c_float(lb), p(state), dtype, ctypes.c_uint(flags), None)


@pytest.mark.parametrize("case,expected", [
    (dict(shape=kda.make_shape(4, 1, 2, 4, K=96)), 2),
    (dict(shape=kda.make_shape(4, 1, 2, 3)), 1),                     # N must equal B
    (dict(shape=kda.make_shape(4, 1, 2, 4), lb=0.25), 1),            # lower_bound in [-5, 0]
    (dict(shape=kda.make_shape(4, 1, 2, 4), state=0), 1),            # the state is required
    (dict(shape=kda.make_shape(4, 1, 2, 4), state=FAKE + 8), 1),     # and 16-byte aligned
    (dict(shape=kda.make_shape(4, 1, 2, 4), dtype=0), 1),            # with a dtype
    (dict(shape=kda.make_shape(4, 1, 2, 4), q=0), 1),
    (dict(shape=kda.make_shape(4, 1, 2, 4), out=FAKE + 1), 1),       # 2-byte aligned tokens
    (dict(shape=kda.make_shape(4, 1, 2, 4), A_log=FAKE + 2), 1),
    (dict(shape=kda.make_shape(4, 1, 2, 4), flags=32), 1),           # unknown flag
    (dict(shape=kda.make_shape(4, 1, 2, 4), flags=9), 1),            # preactivated and softplus gates
])
def test_decode_host_side_argument_errors(case, expected):
    shape = case.pop("shape")
    assert _decode_call(shape, **case) == expected


def test_decode_valid_arguments_reach_the_device_query():
    assert _decode_call(kda.make_shape(4, 1, 2, 4), q=FAKE + 2, out=FAKE + 6) in (4, 5)
    # a gate activated by the caller needs neither A_log nor dt_bias, nor a lower bound in range
    assert _decode_call(kda.make_shape(4, 1, 2, 4), A_log=0, lb=7.0, flags=1) in (4, 5)
    # the softplus gate reads A_log and dt_bias but no lower bound
    assert _decode_call(kda.make_shape(4, 1, 2, 4), lb=7.0, flags=8) in (4, 5)
    assert _decode_call(kda.make_shape(4, 1, 2, 4), A_log=0, flags=8) == 1


def _fwd_ex_call(flags, A_log=FAKE, lb=-1.0):
    lib = kda.load_library()
    p = lambda a: ctypes.c_void_p(a) if a else None
    shape = kda.make_shape(1, 64, 1, 1)
    return lib.kda_fwd_ex(ctypes.byref(shape), p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), ctypes.c_float(0.1),
                          p(FAKE), p(A_log), p(A_log), ctypes.c_float(lb), None, 0, None, 0, None,
                          ctypes.c_uint(flags), p(FAKE), ctypes.c_size_t(1 << 30), None)


def test_fwd_ex_flags_on_the_host():
    assert _fwd_ex_call(32) == 1                      # unknown flag
    assert _fwd_ex_call(16) in (4, 5)                 # KDA_PRECISE_STATE passes the host checks
    assert _fwd_ex_call(9) == 1                       # preactivated and softplus gates exclude each other
    assert _fwd_ex_call(8, lb=9.0) in (4, 5)          # the softplus gate reads no lower bound
    assert _fwd_ex_call(8, A_log=0) == 1              # but needs A_log and dt_bias
    assert _fwd_ex_call(8 | 2 | 4) in (4, 5)
    assert _fwd_ex_call(0, A_log=0) == 1              # the in-kernel gate needs its parameters
    assert _fwd_ex_call(1, A_log=0, lb=9.0) in (4, 5)  # a pre-activated gate does not
    assert _fwd_ex_call(6) in (4, 5)


def test_v64_passes_the_shape_checks():
    # V = 64 is accepted (one chain whose last 64 state rows stay zero); V = 32 is not
    assert _call(kda.make_shape(1, 64, 1, 1, V=64)) in (4, 5)
    assert _decode_call(kda.make_shape(4, 1, 2, 4, V=64)) in (4, 5)
    assert _call(kda.make_shape(1, 64, 1, 1, V=32)) == 2
    assert kda.workspace_size(kda.make_shape(1, 64, 2, 1, V=64)) == kda.workspace_size(kda.make_shape(1, 64, 2, 1))


def test_v256_passes_the_shape_checks():
    # V = 256 is accepted (two 128-row chains per head); without a GPU the call stops at the device query
    assert _call(kda.make_shape(1, 64, 1, 1, V=256)) in (4, 5)
    assert _decode_call(kda.make_shape(4, 1, 2, 4, V=256)) in (4, 5)
    assert kda.workspace_size(kda.make_shape(1, 64, 2, 1, V=256)) >= kda.workspace_size(kda.make_shape(1, 64, 2, 1))


def test_k64_passes_the_shape_checks():
    # K = 64 is accepted (key channels 64-127 held at zero), alone and with V = 64 or 256;
    # the workspace does not depend on K
    for V in (64, 128, 256):
        assert _call(kda.make_shape(1, 64, 1, 1, K=64, V=V)) in (4, 5)
        assert _decode_call(kda.make_shape(4, 1, 2, 4, K=64, V=V)) in (4, 5)
        assert kda.workspace_size(kda.make_shape(1, 64, 2, 1, K=64, V=V)) == \
            kda.workspace_size(kda.make_shape(1, 64, 2, 1, V=V))
    assert _call(kda.make_shape(1, 64, 1, 1, K=256)) == 2


def _bwd_call(shape, q=FAKE, dout=FAKE, dq=FAKE, dt_bias=FAKE, lb=-1.0, ws=FAKE, ws_bytes=1 << 40, flags=0,
              init=None, init_dt=0, dh0=FAKE):
    lib = kda.load_library()
    p = lambda a: ctypes.c_void_p(a) if a else None
    return lib.kda_bwd(ctypes.byref(shape), p(q), p(FAKE), p(FAKE), p(FAKE), p(FAKE), ctypes.c_float(0.1),
                       p(FAKE), p(dt_bias), ctypes.c_float(lb), p(init), init_dt, None, p(dout), None, p(dq),
                       p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(dh0), p(FAKE), p(FAKE), ctypes.c_uint(flags),
                       p(ws), ctypes.c_size_t(ws_bytes), None)


@pytest.mark.parametrize("case,expected", [
    (dict(shape=kda.make_shape(1, 64, 2, 1, K=64)), 2),             # the backward takes K = V = 128 only
    (dict(shape=kda.make_shape(1, 64, 2, 1, V=256)), 2),
    (dict(shape=kda.make_shape(1, 64, 2, 1), dout=FAKE + 8), 1),     # dout read four values at a time
    (dict(shape=kda.make_shape(1, 64, 2, 1), dq=FAKE + 4), 1),       # gradients written as float4
    (dict(shape=kda.make_shape(1, 64, 2, 1), dt_bias=FAKE + 4), 1),
    (dict(shape=kda.make_shape(1, 64, 2, 1), dh0=FAKE + 8), 1),
    (dict(shape=kda.make_shape(1, 64, 2, 1), lb=0.5), 1),
    (dict(shape=kda.make_shape(1, 64, 2, 1), flags=9), 1),
    (dict(shape=kda.make_shape(1, 64, 2, 1), init=FAKE, init_dt=0), 1),
    (dict(shape=kda.make_shape(1, 64, 2, 1), ws=FAKE + 16), 1),      # 256-byte aligned workspace
    (dict(shape=kda.make_shape(1, 64, 2, 1), ws_bytes=1024), 3),     # too small
    (dict(shape=kda.make_shape(2, 64, 2, 3)), 1),                    # N must equal B
])
def test_bwd_host_side_argument_errors(case, expected):
    shape = case.pop("shape")
    assert _bwd_call(shape, **case) == expected


def test_bwd_valid_arguments_reach_the_device_query():
    assert _bwd_call(kda.make_shape(1, 64, 2, 1)) in (4, 5)
    assert _bwd_call(kda.make_shape(1, 64, 2, 1), dh0=0, lb=9.0, flags=1, dt_bias=0) in (4, 5)
    # KDA_BWD_RECURRENT selects the backward's form; kda_fwd_ex does not know it, and no
    # higher bit is a flag
    assert _bwd_call(kda.make_shape(1, 64, 2, 1), flags=kda.KDA_BWD_RECURRENT) in (4, 5)
    assert _bwd_call(kda.make_shape(1, 64, 2, 1), flags=64) == 1
    assert _fwd_ex_call(kda.KDA_BWD_RECURRENT) == 1


def test_bwd_workspace_covers_the_chunked_form():
    # the chunked form stores, per 16 tokens and head, S0 and dS1 (bf16, 32 KiB each), Vn and
    # dVn (fp32, 8 KiB each), three 16 x 128 fp32 state products and a 128-float column sum
    for shape in (kda.make_shape(1, 4096, 2, 1), kda.make_shape(3, 100, 4, 3), kda.make_shape(1, 16, 1, 1)):
        slots = shape.B * shape.T // 16 + shape.N + 1
        assert kda.bwd_workspace_size(shape) >= slots * shape.H * (2 * 32768 + 2 * 8192 + 3 * 8192 + 512)


def test_bwd_workspace_holds_a_state_every_eighth_token():
    n1 = kda.bwd_workspace_size(kda.make_shape(1, 4096, 2, 1))
    n2 = kda.bwd_workspace_size(kda.make_shape(1, 8192, 2, 1))
    # per extra 4096 tokens and 2 heads: 512 stored states of 64 KiB per head, the per
    # token-head vectors and four row-slice partials (1552 B x 5), the dA_log terms, and
    # 16 more parameter blocks of 528 B per head (regions are 256-byte aligned)
    expected = 4096 * 2 * (64 * 1024 // 8 + 1552 * 5 + 4) + 16 * 2 * 528
    assert abs((n2 - n1) - expected) <= 6 * 256
