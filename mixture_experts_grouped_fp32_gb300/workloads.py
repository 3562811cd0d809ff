"""Seeded synthetic inputs for the MoE layer — shared by the CUDA path's tests/bench and the oracle.

This module draws random numbers and names workload shapes; it holds none of the layer's
arithmetic (no routing, no softmax, no GEMM).  Both sides of every parity check receive the
same tensors from here.

Draw recipe (seed s, default 0):
  * ``torch.Generator('cpu').manual_seed(s)``: router logits fp32 [T,E] ~ N(0,1), plus the
    workload's per-expert logit bias; then x = N(0,1) [T,d] rounded to bf16 (round-to-nearest-even).
  * Weights, with a generator seeded ``s + 1`` on ``weight_device``: W_gate [E,d,f], W_up [E,d,f],
    W_down [E,f,d], each 0.02 * N(0,1) rounded to bf16; W_gate_up = concat(W_gate, W_up) on the
    last axis -> [E, d, 2f].  The full-size layers (1.4 G weights) are drawn on the GPU, where the
    CPU would take ~15 s; small layers are drawn on the CPU.  A CUDA-drawn tensor is reproducible
    for a given torch build, which is all a parity check needs (both sides read the same tensor).

  * The grouped router's selection bias (DeepSeek-V3 workload only): bias_std * N(0,1) [E] from a
    CPU generator seeded ``s + 2``.

Workload shapes are those of the pages' benchmarks: a Mixtral-8x7B-shaped MoE layer (d_model
4096, d_ff 14336, 8 experts, top-2) and a DeepSeek-V3-shaped routed-expert layer (d_model 7168,
d_ff 2048 per expert, 256 experts, top-8) — "Triton-MoE-Dispatch-Kernel erreicht 131 % von
Megablocks" (lumeric.app) names Mixtral-8x7B on an A100 and the DeepSeek-V3 skew regime.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    f: int
    E: int
    k: int
    # Per-expert additive logit bias, as a (kind, parameter) pair:
    #   ("none", 0)          plain N(0,1) logits (near-uniform routing)
    #   ("hot0", b)          +b on expert 0's logit (one over-subscribed expert)
    #   ("zipf", s)          + log(r**-s) with rank r = e + 1 (expert 0 most popular)
    bias: tuple = ("none", 0.0)
    note: str = field(default="", compare=False)
    # Router: ("softmax",) — softmax top-k renormalised; or ("grouped", n_group, topk_group, scale,
    # bias_std) — DeepSeek-V3's sigmoid router with a selection bias drawn N(0, bias_std^2).
    router: tuple = ("softmax",)

    @property
    def M(self) -> int:
        return self.T * self.k


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny", 64, 256, 512, 8, 2,
                 note="tiny MoE layer T=64 d=256 f=512 E=8 k=2"),
        Workload("mixtral_t32", 32, 4096, 14336, 8, 2,
                 note="Mixtral-8x7B-shaped layer, decode-like batch T=32"),
        Workload("mixtral_t512", 512, 4096, 14336, 8, 2,
                 note="Mixtral-8x7B-shaped layer, prefill batch T=512"),
        Workload("mixtral_t512_skew40", 512, 4096, 14336, 8, 2, ("hot0", 1.7053),
                 note="T=512 with expert 0 biased to take ~40% of assignments"),
        Workload("mixtral_t4096", 4096, 4096, 14336, 8, 2,
                 note="Mixtral-8x7B-shaped layer, large batch T=4096"),
        Workload("deepseek_t2048", 2048, 7168, 2048, 256, 8, ("zipf", 1.2),
                 note="DeepSeek-V3-shaped routed experts, Zipf(1.2)-skewed loads, T=2048"),
        Workload("deepseek_e32_t256", 256, 7168, 2048, 32, 8, ("zipf", 1.2),
                 note="profiling-scale DeepSeek-V3-shaped layer: same expert shapes and skew, "
                      "32 experts (2.8 GB of weights, small enough for a full ncu capture)"),
        Workload("deepseek_v3like_e32_t1024", 1024, 7168, 2048, 32, 8, ("zipf", 2.0),
                 note="profiling-scale stand-in for the DeepSeek-V3-router layer: the same expert "
                      "shapes and a row distribution of the same kind (a few experts near T rows, "
                      "a third under 16), 32 experts (2.8 GB of weights)"),
        Workload("deepseek_v3_t2048", 2048, 7168, 2048, 256, 8, ("zipf", 1.2),
                 note="DeepSeek-V3-shaped routed experts with DeepSeek-V3's own router: sigmoid "
                      "affinities, selection bias, 8 groups of 32 experts, 4 groups kept, scale 2.5",
                 router=("grouped", 8, 4, 2.5, 0.1)),
    ]
}


def draw_router_bias(w: Workload, seed: int = 0) -> torch.Tensor:
    """The grouped router's per-expert selection bias, fp32 [E] on the CPU: N(0, bias_std^2) from a
    generator seeded ``seed + 2`` (zeros for the softmax router, which has none)."""
    if w.router[0] != "grouped":
        return torch.zeros(w.E, dtype=torch.float32)
    g = torch.Generator("cpu").manual_seed(seed + 2)
    return (torch.randn(w.E, generator=g, dtype=torch.float32) * float(w.router[4])).contiguous()


def logit_bias(E: int, bias: tuple) -> torch.Tensor:
    kind, p = bias
    b = torch.zeros(E, dtype=torch.float32)
    if kind == "hot0":
        b[0] = float(p)
    elif kind == "zipf":
        b = torch.tensor([-float(p) * math.log(e + 1) for e in range(E)], dtype=torch.float32)
    elif kind != "none":
        raise ValueError(f"unknown bias kind {kind!r}")
    return b


def draw_routing(T: int, d: int, E: int, seed: int = 0, bias: tuple = ("none", 0.0)):
    """logits fp32 [T,E] and x bf16 [T,d], both on the CPU."""
    g = torch.Generator("cpu").manual_seed(seed)
    logits = torch.randn(T, E, generator=g, dtype=torch.float32)
    logits = logits + logit_bias(E, bias)[None, :]
    x = torch.randn(T, d, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return logits.contiguous(), x.contiguous()


def _normal_bf16(shape, g, device, scale=0.02, chunk=1 << 26) -> torch.Tensor:
    """scale * N(0,1) rounded to bf16, drawn in flat chunks to bound the fp32 temporary."""
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = (torch.randn(e - s, generator=g, dtype=torch.float32, device=device) * scale).to(
            torch.bfloat16)
    return out.view(*shape)


def draw_weights(d: int, f: int, E: int, seed: int = 0, device="cpu"):
    """W_gate_up bf16 [E,d,2f] and W_down bf16 [E,f,d] on ``device``."""
    device = torch.device(device)
    g = torch.Generator(device.type if device.type == "cpu" else device).manual_seed(seed + 1)
    wg = _normal_bf16((E, d, f), g, device)
    wu = _normal_bf16((E, d, f), g, device)
    wgu = torch.cat([wg, wu], dim=2).contiguous()
    del wg, wu
    wd = _normal_bf16((E, f, d), g, device)
    return wgu, wd


def default_weight_device(w: Workload) -> str:
    n = 3 * w.E * w.d * w.f
    return "cuda" if n > (1 << 26) and torch.cuda.is_available() else "cpu"


def make_inputs(w: Workload, seed: int = 0, weight_device: str | None = None):
    """All four layer inputs: logits [T,E] fp32 (CPU), x [T,d] bf16 (CPU), W_gate_up, W_down."""
    logits, x = draw_routing(w.T, w.d, w.E, seed, w.bias)
    wgu, wd = draw_weights(w.d, w.f, w.E, seed, weight_device or default_weight_device(w))
    return logits, x, wgu, wd


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (on the CPU)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_bf16(bits: np.ndarray) -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 CPU tensor."""
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16)


def draw_e4m3_codes(shape, seed: int) -> np.ndarray:
    """Uniformly random 8-bit E4M3 codes of the given shape, NaN codes (0x7F, 0xFF) excluded: raw
    operands for the FP8 GEMM stages (no quantisation involved)."""
    rng = np.random.default_rng(seed)
    c = rng.integers(0, 254, size=shape, dtype=np.uint16)  # 254 values: skip 0x7F and 0xFF
    c = c + (c >= 0x7F)
    return c.astype(np.uint8)


def draw_scales(shape, seed: int, lo: float = 1e-3, hi: float = 1e-2) -> np.ndarray:
    """Positive fp32 dequantisation scales, log-uniform in [lo, hi]."""
    rng = np.random.default_rng(seed)
    return np.exp(rng.uniform(np.log(lo), np.log(hi), size=shape)).astype(np.float32)


def draw_pow2_scales(shape, seed: int, lo: int = -12, hi: int = -4) -> np.ndarray:
    """fp32 powers of two 2^e, e uniform in [lo, hi]: raw block scales for the blockwise FP8 stages."""
    rng = np.random.default_rng(seed)
    return np.ldexp(1.0, rng.integers(lo, hi + 1, size=shape)).astype(np.float32)
