"""Seeded synthetic inputs for the KDA forward pass.

This module only draws random numbers in a fixed order and lays them out in
the shapes of the FlashKDA README "Kernel API" table (q, k, g: [B,T,H,K] bf16;
v: [B,T,H,V] bf16; beta: [B,T,H] bf16 logits; A_log: [H] fp32; dt_bias: [H,K]
fp32; states: [B|N,H,V,K]; cu_seqlens: int64 [N+1]).  It holds none of the
method's arithmetic, so both the CUDA path and the CPU oracle can take their
inputs from it.

Draw order for every workload: sequence lengths, then q, k, v, g, then the
beta logits, then A_log, then dt_bias, then the initial state.  Normals are
drawn in fp32 and rounded to bf16 (round-to-nearest-even) where the dtype is
bf16.  The generator lives on `device` ("cpu" or "cuda"); the two devices give
different (but each reproducible) numbers.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import torch

K_DIM = 128
V_DIM = 128


@dataclasses.dataclass
class Workload:
    """One synthetic workload; the fields mirror the kernel's arguments."""

    name: str
    B: int
    T: int
    H: int
    seq_lens: Optional[List[int]]      # None: fixed-length batch of B rows
    state_dtype: Optional[torch.dtype]  # dtype of initial/final state (None: no state)
    has_initial_state: bool
    has_final_state: bool
    lower_bound: float
    seed: int
    K: int = K_DIM
    V: int = V_DIM
    scale: float = 1.0 / math.sqrt(K_DIM)

    @property
    def N(self) -> int:
        return len(self.seq_lens) if self.seq_lens is not None else self.B

    @property
    def token_heads(self) -> int:
        return self.B * self.T * self.H


def _varlen_lengths_fixed_total(gen: torch.Generator, n: int, total: int, hi: int) -> List[int]:
    """n lengths: n-1 drawn U[1,hi], the last = total - sum, redrawn until in [1,hi]."""
    while True:
        first = torch.randint(1, hi + 1, (n - 1,), generator=gen).tolist()
        last = total - sum(first)
        if 1 <= last <= hi:
            return first + [last]


def _varlen_lengths_fill(gen: torch.Generator, total: int, lo: int, hi: int) -> List[int]:
    """Repeat L ~ U[lo,hi], L = min(L, rem); a remainder below lo joins the last length."""
    lens: List[int] = []
    rem = total
    while rem > 0:
        L = int(torch.randint(lo, hi + 1, (1,), generator=gen).item())
        L = min(L, rem)
        if 0 < rem - L < lo:
            L = rem
        lens.append(L)
        rem -= L
    return lens


def tiny_workload() -> Workload:
    """B=1, T=64, H=1 (four 16-token chunks); no initial state, fp32 final state."""
    return Workload("tiny_B1_T64_H1", 1, 64, 1, None, torch.float32, False, True, -5.0, 0)


def fixed_batch_workload() -> Workload:
    """B=2, T=4096, H=16; fp32 initial and final state; lower_bound -2."""
    return Workload("fixed_B2_T4096_H16", 2, 4096, 16, None, torch.float32, True, True, -2.0, 1)


def varlen_workload(seed: int = 2) -> Workload:
    """B=1, T=32768 split into 8 sequences of U[1,8192] tokens; H=32; bf16 states."""
    gen = torch.Generator().manual_seed(seed)
    lens = _varlen_lengths_fixed_total(gen, 8, 32768, 8192)
    return Workload("varlen_T32768_N8_H32", 1, 32768, 32, lens, torch.bfloat16, True, True, -5.0, seed)


def long_workload() -> Workload:
    """B=1, T=1,048,576, H=8; no initial state, fp32 final state; lower_bound -1."""
    return Workload("long_T1048576_H8", 1, 1 << 20, 8, None, torch.float32, False, True, -1.0, 3)


def decode_workload() -> Workload:
    """One decoding step of a serving batch: B=256 sequences x T=1 token, H=32, fp32 states
    read and written in place (512 MiB, four times L2); lower_bound -5."""
    return Workload("decode_B256_T1_H32", 256, 1, 32, None, torch.float32, True, True, -5.0, 5)


SWEEP_TOTALS = (8192, 32768, 131072, 262144)
SWEEP_HEADS = (32, 64)


def sweep_workload(total: int, H: int) -> Workload:
    """Varlen batch of `total` tokens in lengths U[64,16384]; fp32 states; lower_bound -5."""
    idx = SWEEP_TOTALS.index(total) * len(SWEEP_HEADS) + SWEEP_HEADS.index(H)
    seed = 40 + idx
    gen = torch.Generator().manual_seed(seed)
    lens = _varlen_lengths_fill(gen, total, 64, 16384)
    return Workload(f"sweep_T{total}_H{H}", 1, total, H, lens, torch.float32, True, True, -5.0, seed)


def custom_workload(name: str, B: int, T: int, H: int, seq_lens=None, state_dtype=torch.float32,
                    has_initial_state=True, has_final_state=True, lower_bound=-5.0,
                    seed=1234, V: int = V_DIM, K: int = K_DIM) -> Workload:
    return Workload(name, B, T, H, list(seq_lens) if seq_lens is not None else None,
                    state_dtype, has_initial_state, has_final_state, lower_bound, seed, K=K, V=V,
                    scale=1.0 / math.sqrt(K))


def named_workloads() -> Dict[str, Workload]:
    out = {w.name: w for w in (tiny_workload(), fixed_batch_workload(), varlen_workload(),
                               long_workload(), decode_workload())}
    for total in SWEEP_TOTALS:
        for H in SWEEP_HEADS:
            w = sweep_workload(total, H)
            out[w.name] = w
    return out


def _normal_bf16(gen: torch.Generator, shape, device, std: float = 1.0,
                 rows_per_draw: int = 1 << 22) -> torch.Tensor:
    """N(0, std^2) drawn in fp32 and rounded to bf16, in row blocks to bound memory."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1, shape[-1]) if len(shape) > 1 else out.view(1, -1)
    rows = flat.shape[0]
    for r0 in range(0, rows, rows_per_draw):
        r1 = min(rows, r0 + rows_per_draw)
        blk = torch.randn((r1 - r0, flat.shape[1]), generator=gen, dtype=torch.float32,
                          device=device)
        if std != 1.0:
            blk.mul_(std)
        flat[r0:r1].copy_(blk)
    return out


def make_inputs(w: Workload, device="cpu") -> Dict[str, object]:
    """Draw all inputs of workload `w` on `device`; returns a dict of tensors and scalars."""
    device = torch.device(device)
    gen = torch.Generator(device=device).manual_seed(w.seed)
    if w.seq_lens is not None:
        assert w.B == 1 and sum(w.seq_lens) == w.T
        cu = torch.zeros(len(w.seq_lens) + 1, dtype=torch.int64)
        cu[1:] = torch.cumsum(torch.tensor(w.seq_lens, dtype=torch.int64), 0)
    else:
        cu = None
    B, T, H, K, V = w.B, w.T, w.H, w.K, w.V
    q = _normal_bf16(gen, (B, T, H, K), device)
    k = _normal_bf16(gen, (B, T, H, K), device)
    v = _normal_bf16(gen, (B, T, H, V), device)
    g = _normal_bf16(gen, (B, T, H, K), device)
    beta = _normal_bf16(gen, (B, T, H), device)
    A_log = torch.rand((H,), generator=gen, dtype=torch.float32, device=device) * 2.0 - 1.0
    dt_bias = torch.randn((H, K), generator=gen, dtype=torch.float32, device=device) * 0.1
    init = None
    if w.has_initial_state:
        init = torch.randn((w.N, H, V, K), generator=gen, dtype=torch.float32,
                           device=device) * 0.02
        init = init.to(w.state_dtype)
    return dict(q=q, k=k, v=v, g=g, beta=beta, A_log=A_log, dt_bias=dt_bias,
                scale=w.scale, lower_bound=w.lower_bound, initial_state=init,
                cu_seqlens=cu.to(device) if cu is not None else None)


def random_varlen(gen: torch.Generator, n: int, lo: int, hi: int) -> List[int]:
    """n lengths drawn independently U[lo,hi] (edge-case tests)."""
    return torch.randint(lo, hi + 1, (n,), generator=gen).tolist()
