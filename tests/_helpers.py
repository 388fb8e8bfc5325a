"""Shared test utilities: host<->device conversion and the attention tolerance check."""
from __future__ import annotations

import math

import numpy as np

import oracle as O


def bf16_tensor(bits: np.ndarray, device="cuda"):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def bf16_bits(t) -> np.ndarray:
    import torch

    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_dev(a: np.ndarray, device="cuda"):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def attention_close(got: np.ndarray, ref: np.ndarray, rtol: float = 2e-2) -> tuple[bool, str]:
    """Attention tolerance: per (row set, head) ||got - ref||_F <= rtol ||ref||_F and, per
    element, |got - ref| <= rtol (|ref| + rms(ref)).

    got, ref: [R, H, D] float64 (got already widened from bf16).
    """
    if got.shape != ref.shape:
        return False, f"shape {got.shape} != {ref.shape}"
    if not np.all(np.isfinite(got)):
        return False, "non-finite output"
    worst = 0.0
    for h in range(ref.shape[1]):
        d = got[:, h] - ref[:, h]
        nr = np.linalg.norm(ref[:, h])
        rel = np.linalg.norm(d) / max(nr, 1e-30)
        worst = max(worst, rel)
        if rel > rtol:
            return False, f"head {h}: frobenius rel err {rel:.3e}"
        rms = math.sqrt(float(np.mean(ref[:, h] ** 2)))
        bad = np.abs(d) > rtol * (np.abs(ref[:, h]) + rms)
        if bad.any():
            i = np.argwhere(bad)[0]
            return False, f"head {h} elem {tuple(i)}: got {got[:, h][tuple(i)]} ref {ref[:, h][tuple(i)]}"
    return True, f"worst frobenius rel err {worst:.3e}"


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    return O.widen(bits, "bf16")
