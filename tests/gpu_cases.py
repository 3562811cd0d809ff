"""Shared helpers for the GPU parity tests: seeded cases, oracle references, tolerances.

Tolerances (floating point; integer/index outputs are compared bit for bit):
  * layer output (bf16 out vs the oracle's fp32 out): max|gpu - oracle| <= 1e-2 * max|oracle|,
    plus an elementwise screen |gpu - oracle| <= 2^-7 |oracle| + 2e-3 max|oracle| that a wrong
    tile or row would fail.
  * route weights: relative 1e-6 (both sides take fp32 exp of the same differences).
  * gate+up stage (bf16 h vs the oracle's fp32 h): bf16 rounding is 2^-9 relative, so the screen
    is 2^-7 |ref| + 2e-3 max|ref|, and the global bound 1e-2 max|ref|.
  * down stage (fp32 y from the same bf16 operands): only the summation order differs:
    1e-3 |ref| + 1e-4 max|ref|.
  * combine (bf16 out from fp32 y): 2^-8 |ref| + 1e-6 max|ref|.
"""
from __future__ import annotations

import numpy as np
import torch

from mixture_experts_grouped_fp32_gb300.workloads import (Workload, bf16_bits, bits_to_bf16, draw_routing,
                                                          draw_weights)


def assert_close(got, ref, rtol, atol_of_max, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    bound = rtol * np.abs(ref) + atol_of_max * scale
    bad = np.abs(got - ref) > bound
    if bad.any():
        i = tuple(int(v) for v in np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} elements off; first at {i}: gpu {got[i]!r} "
                             f"oracle {ref[i]!r} (bound {bound[i]:.3e}, max|ref| {scale:.3e})")


def assert_layer_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = float(np.abs(got - ref).max()) if ref.size else 0.0
    bound = 1e-2 * float(np.abs(ref).max()) if ref.size else 0.0
    assert err <= bound, f"{what}: max|gpu-oracle| = {err:.4e} > 1e-2 * max|oracle| = {bound:.4e}"
    assert_close(got, ref, 2.0 ** -7, 2e-3, what)


def case_inputs(w: Workload, seed: int = 0, weight_device: str = "cpu"):
    logits, x = draw_routing(w.T, w.d, w.E, seed, w.bias)
    wgu, wd = draw_weights(w.d, w.f, w.E, seed, weight_device)
    return logits, x, wgu, wd


def random_bf16(shape, seed, scale=1.0):
    g = torch.Generator("cpu").manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


def to_np_bits(t: torch.Tensor) -> np.ndarray:
    return bf16_bits(t)


def from_np_bits(a: np.ndarray) -> torch.Tensor:
    return bits_to_bf16(a)


def tile_class_tokens(src, offsets, rng, n_random=6, n_extreme=10):
    """Tokens whose outputs reach every class of GEMM tile at full size: the first and last token,
    random ones, the last row of every non-empty expert (its last, usually partial, M-tile; for a
    small expert its swapped chunk), and for the n_extreme largest and smallest non-empty experts
    also the first row of the segment and of its last 128-row and 256-row tiles (single-SM and
    SM-pair tiles)."""
    src = np.asarray(src)
    offsets = np.asarray(offsets)
    T = int(src.max()) + 1 if src.size else 0
    counts = np.diff(offsets)
    active = np.nonzero(counts > 0)[0]
    rows = [offsets[e + 1] - 1 for e in active]
    order = active[np.argsort(counts[active], kind="stable")]
    for e in np.unique(np.concatenate([order[:n_extreme], order[-n_extreme:]])):
        n = int(counts[e])
        rows += [offsets[e], offsets[e] + 128 * ((n - 1) // 128), offsets[e] + 256 * ((n - 1) // 256)]
    tokens = src[np.asarray(rows, np.int64)]
    extra = [0, T - 1] + list(rng.integers(0, T, n_random))
    return np.unique(np.concatenate([tokens, extra])).astype(np.int32)
