"""Numerics comparator used by every parity test.

It reports the statistics of the kernel-numerics table in vllm.cpp PR #425
('head_dim-128 arm for the warp-split-KV decode kernel', EVIDENCE section):
max_abs, max_rel and the bitwise-identical percentage, plus the indices that
differ, so a failure is localised.

Reading of "max_rel" (the acceptance bound names it without a definition):
normwise, max|g - o| / max|o| over one output tensor.  The elementwise
relative error (denominator floored at 1e-3) is reported alongside.
"""
from __future__ import annotations

import dataclasses

import numpy as np

import synth

# acceptance bounds for bf16 outputs and fp32 LSE
MAX_ABS = 1.5e-2
MAX_REL = 2e-2
LSE_ABS = 1e-4


@dataclasses.dataclass
class Stats:
    n: int
    max_abs: float
    max_rel: float
    max_rel_elem: float
    bitwise_pct: float
    worst_index: int
    differing: np.ndarray

    def ok(self, max_abs=MAX_ABS, max_rel=MAX_REL) -> bool:
        return self.max_abs <= max_abs and self.max_rel <= max_rel

    def __str__(self):
        return (f"n={self.n} max_abs={self.max_abs:.3e} max_rel={self.max_rel:.3e} "
                f"max_rel_elem={self.max_rel_elem:.3e} bitwise={self.bitwise_pct:.4f}% "
                f"worst@{self.worst_index}")


def bf16_bits(x) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return x
    return synth.f32_to_bf16_bits(x.astype(np.float32))


def as_f64(x) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return synth.bf16_bits_to_f32(x).astype(np.float64)
    return x.astype(np.float64)


def compare(got, ref) -> Stats:
    """got: bf16 bit patterns (uint16) or floats; ref: float64 (or bf16 bits for kernel-vs-kernel)."""
    g = as_f64(got).ravel()
    r = as_f64(ref).ravel()
    assert g.shape == r.shape, (g.shape, r.shape)
    n = g.size
    if n == 0:
        return Stats(0, 0.0, 0.0, 0.0, 100.0, -1, np.zeros(0, dtype=np.int64))
    diff = np.abs(g - r)
    diff = np.where(np.isnan(diff), np.inf, diff)
    worst = int(np.argmax(diff))
    max_abs = float(diff[worst])
    scale = float(np.max(np.abs(r))) if np.isfinite(r).any() else 0.0
    max_rel = max_abs / scale if scale > 0 else (0.0 if max_abs == 0 else np.inf)
    max_rel_elem = float(np.max(diff / np.maximum(np.abs(r), 1e-3)))
    gb = bf16_bits(got).ravel() if np.asarray(got).dtype == np.uint16 else bf16_bits(g)
    rb = bf16_bits(ref).ravel() if np.asarray(ref).dtype == np.uint16 else bf16_bits(r)
    same = gb == rb
    differing = np.nonzero(~same)[0]
    return Stats(n, max_abs, max_rel, max_rel_elem, 100.0 * float(same.mean()), worst, differing)


def lse_max_abs(got, ref) -> float:
    g = np.asarray(got, dtype=np.float64).ravel()
    r = np.asarray(ref, dtype=np.float64).ravel()
    both_inf = np.isinf(g) & np.isinf(r) & (np.sign(g) == np.sign(r))
    with np.errstate(invalid="ignore"):
        d = np.where(both_inf, 0.0, np.abs(g - r))
    d = np.where(np.isnan(d), np.inf, d)
    return float(d.max()) if d.size else 0.0
