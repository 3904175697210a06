"""Small helpers shared by the CPU tests (tests only; never imported by the product)."""
from __future__ import annotations

import numpy as np
import torch


def bf16(x) -> torch.Tensor:
    """fp64/fp32 array -> bf16 tensor (RNE)."""
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def as_f64(t) -> np.ndarray:
    return t.to(torch.float64).numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


def rel_fro(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b.ravel())
    return float(np.linalg.norm((a - b).ravel()) / (den if den > 0 else 1.0))


def l2n(x, eps=1e-6):
    """Row-wise L2 normalisation with the epsilon inside the square root."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + eps)
