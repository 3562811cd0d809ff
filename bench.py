"""Benchmark of the MoE layer forward on GB300: prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                    [--dtype bf16|e4m3|e4m3b] [--flush-l2] [--no-cpu-baseline]

A step is one pass of the whole layer (route -> permute -> gate+up/SwiGLU GEMM -> down GEMM ->
combine) over one batch of seeded synthetic input.  Default (headline) workload: the
Mixtral-8x7B-shaped large batch (T=4096, d=4096, f=14336, E=8, top-2), the largest configuration of
the metric's T=32..4096 range and the tensor-bound one.  The same JSON line carries `per_workload`:
the other configurations (Mixtral T=32, T=512, T=512 with 40 % of assignments on one expert, the
DeepSeek-V3-shaped routed experts with the softmax router and with DeepSeek-V3's own router), each
measured in the same process the same way (steps, roofline, layer roofline, e2e, clocks), one after
the other; `--per-workload none` turns them off.  `timed_region_s` is the headline's timed region
(wall clock), `timed_region_s_all_workloads` the sum over every workload's.

ours (default):
  value        tokens/s with inputs resident in HBM: K steps of moe_forward, CUDA events around each
               step on its stream (K defaults to ~0.5 s of device time; nvidia-smi samples the SM
               clock and throttle reasons every 20 ms during that region).  The weights of every
               workload (>= 2.8 GB) exceed the 129 MB L2, so they stream from HBM each step;
               --flush-l2 also writes 512 MB between steps.
  roofline     the dominant kernel: its algorithmic bytes (or FLOPs) per launch / its mean duration,
               from a second K-step loop that calls the five stage entry points with events between
               them (the same kernels moe_forward launches).  `traffic` is the kernel's DRAM bytes
               per launch from an earlier ncu capture of the same kernel source (`traffic_source`
               says so and names the source hash); null once the source has changed since.
  e2e          tokens/s with x and logits copied from page-locked host memory, the layer and out
               copied back, every step, all inside the timed region: through moe_forward_host_batches
               or its FP8 / DeepSeek-V3-router forms (the K steps as K batches, copies overlapped with
               the layers on two copy streams); with --flush-l2 the binding's copies and layer per
               step on one stream.
  cpu_baseline the CPU oracle on a bounded sample of the same workload (rank 0, N=1 only).
reference:
  the CPU oracle as the reference arm: each step is the oracle's forward on a bounded token
  sample of the same workload (repeated to fill --ref-step-s seconds, by default ~150 s over
  all steps), timed on the host cores.
--dtype e4m3 times the FP8 variant instead (moe_forward_fp8: the grouped GEMMs on E4M3 codes with
per-row / per-output-channel scales; weights quantised once before the timed region), with the
same metric, and the FP8 oracle as CPU baseline and reference arm; --dtype e4m3b the blockwise
variant (moe_forward_fp8b: power-of-two scales per 1x128 activation and 128x128 weight block).
Under torchrun (N > 1) each rank runs an independent replica of the layer on its own GPU (the
layer has no cross-rank exchange); value = tokens of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mixture_experts_grouped_fp32_gb300.workloads import (WORKLOADS, Workload, bf16_bits, draw_router_bias,  # noqa: E402
                                                          make_inputs)

METRIC = "MoE-layer tokens/s and TFLOP/s, % of roofline (1×GB300), T=32..4096"
DEFAULT_WORKLOAD = "mixtral_t4096"
PER_WORKLOAD = ("mixtral_t32", "mixtral_t512", "mixtral_t512_skew40", "deepseek_t2048", "deepseek_v3_t2048")
L2_FLUSH_BYTES = 512 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
STAGES = ("route", "permute", "gateup_swiglu", "down", "combine")
KERNEL_NAMES = {"route": "route_kernel", "permute": "permute_kernel",
                "gateup_swiglu": "grouped_gemm_kernel<0, false, false>",
                "down": "grouped_gemm_kernel<1, false, false>",
                "combine": "combine_kernel"}
# The FP8 layer's stages (moe_forward_fp8) and its GEMM kernels' template instances <KIND, GATHER, FP8>.
STAGES_FP8 = ("route", "permute", "gateup_swiglu", "quantize_h", "down", "combine")
KERNEL_NAMES_FP8 = {"gateup_swiglu": "grouped_gemm_kernel<0, false, true>",
                    "down": "grouped_gemm_kernel<1, false, true>"}
STAGES_FP8B = ("route", "permute", "quantize_x", "gateup_swiglu", "quantize_h", "down", "combine")
# ... when the gate+up GEMM quantises h in its epilogue (moe_fp8b_gemm_quantizes_h).
STAGES_FP8B_FUSED = ("route", "permute", "quantize_x", "gateup_swiglu", "down", "combine")
# <KIND, QH>: QH = h quantised in the gate+up epilogue.
KERNEL_NAMES_FP8B = {"gateup_swiglu": "grouped_gemm_fp8b_kernel<0, false>",
                     "down": "grouped_gemm_fp8b_kernel<1, false>"}
FP8_OVER_BF16 = 2.0  # nominal dense tensor rate ratio (4.5 / 2.25 PFLOP/s) applied to the measured bf16 peak

# Default timed region (no --steps): about this much device time, within these step counts.
AUTO_TIMED_S = 0.5
AUTO_STEPS_MIN, AUTO_STEPS_MAX = 50, 4000

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum per launch) from ncu captures of the
# kernel source with the recorded hash; reported only while the GEMM source still hashes to that
# value, else null.

_TRAFFIC_HASH = "a50adcb350358d68"  # GEMM source hash the captures below were taken at
_TRAFFIC_HASH_FP8B = "cb56d74ba1e13f0f"  # ... and that of the blockwise FP8 kernel's sources
MEASURED_TRAFFIC = {
    ("deepseek_e32_t256", "gateup_swiglu"): (1919805440, _TRAFFIC_HASH),
    ("deepseek_e32_t256", "down"): (1010249216, _TRAFFIC_HASH),
    ("deepseek_v3like_e32_t1024", "gateup_swiglu"): (2392060160, _TRAFFIC_HASH),
    ("deepseek_v3like_e32_t1024", "down"): (1213201152, _TRAFFIC_HASH),
    ("mixtral_t32", "gateup_swiglu"): (1884503296, _TRAFFIC_HASH),
    ("mixtral_t32", "down"): (946020864, _TRAFFIC_HASH),
    ("mixtral_t4096", "gateup_swiglu"): (3273731072, _TRAFFIC_HASH),
    ("mixtral_t4096", "down"): (1626119680, _TRAFFIC_HASH),
    ("mixtral_t512_skew40", "gateup_swiglu"): (1917325056, _TRAFFIC_HASH),
    ("mixtral_t512_skew40", "down"): (984870656, _TRAFFIC_HASH),
    ("mixtral_t512", "gateup_swiglu"): (1917185792, _TRAFFIC_HASH),
    ("mixtral_t512", "down"): (984192000, _TRAFFIC_HASH),
    ("deepseek_e32_t256", "gateup_swiglu_fp8b"): (966629888, _TRAFFIC_HASH_FP8B),
    ("deepseek_e32_t256", "down_fp8b"): (534442240, _TRAFFIC_HASH_FP8B),
    ("deepseek_v3like_e32_t1024", "gateup_swiglu_fp8b"): (1022789120, _TRAFFIC_HASH_FP8B),
    ("deepseek_v3like_e32_t1024", "down_fp8b"): (728637696, _TRAFFIC_HASH_FP8B),
    ("mixtral_t32", "gateup_swiglu_fp8b"): (944861440, _TRAFFIC_HASH_FP8B),
    ("mixtral_t32", "down_fp8b"): (474419968, _TRAFFIC_HASH_FP8B),
    ("mixtral_t4096", "gateup_swiglu_fp8b"): (1090738176, _TRAFFIC_HASH_FP8B),
    ("mixtral_t4096", "down_fp8b"): (776733440, _TRAFFIC_HASH_FP8B),
    ("mixtral_t512_skew40", "gateup_swiglu_fp8b"): (962235136, _TRAFFIC_HASH_FP8B),
    ("mixtral_t512_skew40", "down_fp8b"): (514651392, _TRAFFIC_HASH_FP8B),
    ("mixtral_t512", "gateup_swiglu_fp8b"): (963427840, _TRAFFIC_HASH_FP8B),
    ("mixtral_t512", "down_fp8b"): (591564544, _TRAFFIC_HASH_FP8B),
    ("deepseek_e32_t256", "gateup_swiglu_fp8"): (966086656, _TRAFFIC_HASH),
    ("deepseek_e32_t256", "down_fp8"): (535560192, _TRAFFIC_HASH),
    ("deepseek_v3like_e32_t1024", "gateup_swiglu_fp8"): (1142837248, _TRAFFIC_HASH),
    ("deepseek_v3like_e32_t1024", "down_fp8"): (725435136, _TRAFFIC_HASH),
    ("mixtral_t32", "gateup_swiglu_fp8"): (946222592, _TRAFFIC_HASH),
    ("mixtral_t32", "down_fp8"): (475548416, _TRAFFIC_HASH),
    ("mixtral_t4096", "gateup_swiglu_fp8"): (1215292672, _TRAFFIC_HASH),
    ("mixtral_t4096", "down_fp8"): (788060672, _TRAFFIC_HASH),
    ("mixtral_t512_skew40", "gateup_swiglu_fp8"): (972208384, _TRAFFIC_HASH),
    ("mixtral_t512_skew40", "down_fp8"): (499746560, _TRAFFIC_HASH),
    ("mixtral_t512", "gateup_swiglu_fp8"): (971900672, _TRAFFIC_HASH),
    ("mixtral_t512", "down_fp8"): (499183872, _TRAFFIC_HASH),
}
GEMM_SOURCES = ("mixture_experts_grouped_fp32_gb300/csrc/grouped_gemm.cu",
                "mixture_experts_grouped_fp32_gb300/csrc/grouped_gemm_2sm.cu",
                "mixture_experts_grouped_fp32_gb300/csrc/tcgen05.cuh")


# The blockwise FP8 GEMMs' own kernel (their traffic entries carry this source set's hash).
FP8B_SOURCES = ("mixture_experts_grouped_fp32_gb300/csrc/grouped_gemm_fp8b.cu",
                "mixture_experts_grouped_fp32_gb300/csrc/tcgen05.cuh")


def gemm_source_hash(sources=GEMM_SOURCES) -> str:
    import hashlib
    h = hashlib.sha256()
    for p in sources:
        with open(os.path.join(ROOT, p), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str, stage: str):
    """(bytes per launch, where the figure comes from): a stored ncu capture of this kernel source."""
    rec = MEASURED_TRAFFIC.get((workload, stage))
    sources = FP8B_SOURCES if stage.endswith("_fp8b") else GEMM_SOURCES
    h = gemm_source_hash(sources)
    if rec and rec[1] == h:
        return rec[0], (f"stored ncu capture (dram__bytes_read.sum + dram__bytes_write.sum, one launch) of this "
                        f"kernel source, hash {h}; not measured in this run")
    why = "no capture of this workload" if not rec else f"source changed since the capture (hash {rec[1]} -> {h})"
    return None, f"null: {why}"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------------------------
# Algorithmic work per stage (what the layer must move / compute, not what the kernels happen to)
# ----------------------------------------------------------------------------------------------
def stage_work(w: Workload, n_active: int, fp8: bool = False, blocks: bool = False, fuse_h: bool = False) -> dict:
    T, d, f, E, k = w.T, w.d, w.f, w.E, w.k
    M = T * k
    if blocks:  # 1-byte codes; one 4-byte scale per 128 x 128 weight block and per 128 activation values
        h_out = M * f + M * f // 32 if fuse_h else M * f * 2  # codes + block scales, or bf16 h
        work = {
            "route": {"bytes": T * E * 4 + M * 8, "flops": 0},
            "permute": {"bytes": M * 4 + (E + E + 1 + 2 * M) * 4, "flops": 0},
            "quantize_x": {"bytes": M * 4 + T * d * 2 + M * d + M * d // 32, "flops": 0},
            "gateup_swiglu": {"bytes": n_active * (d * 2 * f + d * 2 * f // 4096) + M * d + M * d // 32 + h_out,
                              "flops": 4 * M * d * f},
            "quantize_h": {"bytes": M * f * 2 + M * f + M * f // 32, "flops": 0},
            "down": {"bytes": n_active * (f * d + f * d // 4096) + M * f + M * f // 32 + M * d * 4,
                     "flops": 2 * M * d * f},
            "combine": {"bytes": M * d * 4 + M * 8 + T * d * 2, "flops": 2 * M * d},
        }
        if fuse_h:
            del work["quantize_h"]
        return work
    if fp8:  # 1-byte codes; weight scales 4 bytes per output column, activation scales per row
        return {
            "route": {"bytes": T * E * 4 + M * 8, "flops": 0},
            "permute": {"bytes": M * 4 + T * d * 2 + M * d + M * 4 + (E + E + 1 + 2 * M) * 4, "flops": 0},
            "gateup_swiglu": {"bytes": n_active * (d * 2 * f + 2 * f * 4) + M * d + M * 4 + M * f * 2,
                              "flops": 4 * M * d * f},
            "quantize_h": {"bytes": M * f * 2 + M * f + M * 4, "flops": 0},
            "down": {"bytes": n_active * (f * d + d * 4) + M * f + M * 4 + M * d * 4, "flops": 2 * M * d * f},
            "combine": {"bytes": M * d * 4 + M * 8 + T * d * 2, "flops": 2 * M * d},
        }
    return {
        "route": {"bytes": T * E * 4 + M * 8, "flops": 0},
        "permute": {"bytes": M * 4 + T * d * 2 + M * d * 2 + (E + E + 1 + 2 * M) * 4, "flops": 0},
        "gateup_swiglu": {"bytes": n_active * d * 2 * f * 2 + M * d * 2 + M * f * 2, "flops": 4 * M * d * f},
        "down": {"bytes": n_active * f * d * 2 + M * f * 2 + M * d * 4, "flops": 2 * M * d * f},
        "combine": {"bytes": M * d * 4 + M * 8 + T * d * 2, "flops": 2 * M * d},
    }


def layer_work(w: Workload, n_active: int, fp8: bool = False, blocks: bool = False) -> dict:
    if blocks:
        wbytes = n_active * (3 * w.d * w.f + 3 * w.d * w.f // 4096)
    elif fp8:
        wbytes = n_active * (3 * w.d * w.f + 4 * (2 * w.f + w.d))
    else:
        wbytes = n_active * 3 * w.d * w.f * 2
    return {"bytes": wbytes + w.T * w.d * 2 + w.T * w.E * 4 + w.T * w.d * 2,
            "flops": 6 * w.T * w.k * w.d * w.f}


# ----------------------------------------------------------------------------------------------
# Clock sampling during the timed region
# ----------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5:
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        t0, t1 = (self.marks[0], self.marks[-1]) if len(self.marks) >= 2 else (0, 1e30)
        rows = [ln for (t, ln) in self.lines if t0 - 0.05 <= t <= t1 + 0.05] or [ln for _, ln in self.lines[-3:]]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------------------------
# Our arm
# ----------------------------------------------------------------------------------------------
def max_over_ranks(value: float, dist, device=None) -> float:
    """The largest of every rank's value (the slowest replica sets the whole job's time)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    on = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=on)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job throughput of independent replicas: all ranks' tokens over the slowest rank's time."""
    return tokens_per_rank * world / (ms_max * 1e-3)


def run_ours(args, w: Workload, rank: int, world: int, dist):
    from mixture_experts_grouped_fp32_gb300 import moe
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    moe.load()

    blocks = args.dtype == "e4m3b"
    fp8 = args.dtype == "e4m3" or blocks
    logits, x, wgu, wd = make_inputs(w, seed=args.seed + rank, weight_device=str(dev))
    x_d, l_d = x.to(dev), logits.to(dev)
    if fp8:
        quant = moe.quantize_weights_fp8b if blocks else moe.quantize_weights_fp8
        w8 = quant(wgu) + quant(wd)  # (wgu8, sgu, wd8, sd), once
        torch.cuda.synchronize(dev)
        wsize = moe.workspace_size_fp8b if blocks else moe.workspace_size_fp8
        ws = torch.empty(wsize(w.T, w.d, w.f, w.E, w.k), dtype=torch.uint8, device=dev)
    else:
        ws = torch.empty(moe.workspace_size(w.T, w.d, w.f, w.E, w.k) + moe.host_staging_size(w.T, w.d, w.E),
                         dtype=torch.uint8, device=dev)
    out = torch.empty(w.T, w.d, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev) if args.flush_l2 else None
    stream = torch.cuda.current_stream(dev)

    grouped = w.router[0] == "grouped"
    bias_d = draw_router_bias(w, seed=args.seed + rank).to(dev)

    def step():
        if fp8 and grouped:  # an FP8 layer with DeepSeek-V3's router as step 1
            _, G, tg, scale, _ = w.router
            moe.forward_grouped_fp8(x_d, l_d, bias_d, *w8, w.k, G, tg, scale, out=out, workspace=ws, blocks=blocks)
        elif blocks:
            moe.forward_fp8b(x_d, l_d, *w8, w.k, out=out, workspace=ws)
        elif fp8:
            moe.forward_fp8(x_d, l_d, *w8, w.k, out=out, workspace=ws)
        elif grouped:  # DeepSeek-V3's router as step 1
            _, G, tg, scale, _ = w.router
            moe.forward_grouped(x_d, l_d, bias_d, wgu, wd, w.k, G, tg, scale, out=out, workspace=ws)
        else:
            moe.forward(x_d, l_d, wgu, wd, w.k, out=out, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if moe.get_device_error(ws) != 0:
        raise RuntimeError("device status word set during warm-up")
    if args.steps is None:
        # No --steps: time enough steps for ~0.5 s of device work, so that the clock sampler
        # (20 ms period) sees the timed region ~25 times; every rank takes the same K.
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(3):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        est = max_over_ranks(e0.elapsed_time(e1) / 3, dist, dev)
        args.steps = int(min(AUTO_STEPS_MAX, max(AUTO_STEPS_MIN, math.ceil(AUTO_TIMED_S * 1e3 / est))))

    views = moe.workspace_views_fp8b if blocks else (moe.workspace_views_fp8 if fp8 else moe.workspace_views)
    v = views(ws, w.T, w.d, w.f, w.E, w.k)
    counts = v["counts"].cpu().numpy()
    n_active = int((counts > 0).sum())

    # ---- timed region: K steps of moe_forward --------------------------------------------------
    sampler = ClockSampler(local) if rank == 0 or world > 1 else None
    if sampler:
        sampler.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.mark()
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    t_wall = time.perf_counter() - t_wall0
    if sampler:
        sampler.mark()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    ms = statistics.mean(step_ms)
    ms_max = max_over_ranks(ms, dist, dev)
    clocks = sampler.stop() if sampler else None

    # ---- per-stage timing: the five stage entry points, events between launches ---------------
    idx, wts = v["idx"], v["w"]
    counts_d, offs, src, dest, h, y = (v["counts"], v["offsets"], v["src"], v["dest"], v["h"], v["y_perm"])
    st = v["status"]
    fuse_h = blocks and moe.fp8b_gemm_quantizes_h(w.T, w.E, w.k)
    stages = (STAGES_FP8B_FUSED if fuse_h else STAGES_FP8B) if blocks else (STAGES_FP8 if fp8 else STAGES)
    if blocks:
        x8, sx, h8, sh = v["x8"], v["sx"], v["h8"], v["sh"]
        route_call = ((lambda: moe.route_grouped(l_d, bias_d, w.k, *w.router[1:4], idx=idx, w=wts)) if grouped else
                      (lambda: moe.route(l_d, w.k, idx=idx, w=wts)))
        calls = [
            route_call,
            lambda: moe.permute(idx, x_d, w.E, status=st, out=(counts_d, offs, src, dest, None)),
            lambda: moe.quantize_rows_fp8b(x_d, src, status=st, out=(x8, sx)),
        ] + ([
            lambda: moe.grouped_gemm_gateup_swiglu_fp8b_q(x8, sx, w8[0], w8[1], offs, h8=h8, sh=sh, status=st),
        ] if fuse_h else [
            lambda: moe.grouped_gemm_gateup_swiglu_fp8b(x8, sx, w8[0], w8[1], offs, h=h, status=st),
            lambda: moe.quantize_rows_fp8b(h, status=st, out=(h8, sh)),
        ]) + [
            lambda: moe.grouped_gemm_down_fp8b(h8, sh, w8[2], w8[3], offs, y_perm=y, status=st, ksplit=v["ksplit"]),
            lambda: moe.combine(y, wts, dest, out=out, status=st, ksplit=v["ksplit"]),
        ]
    elif fp8:
        x8, sx, h8, sh = v["x8"], v["sx"], v["h8"], v["sh"]
        route_call = ((lambda: moe.route_grouped(l_d, bias_d, w.k, *w.router[1:4], idx=idx, w=wts)) if grouped else
                      (lambda: moe.route(l_d, w.k, idx=idx, w=wts)))
        calls = [
            route_call,
            lambda: moe.permute_fp8(idx, x_d, w.E, status=st, out=(counts_d, offs, src, dest, x8, sx)),
            lambda: moe.grouped_gemm_gateup_swiglu_fp8(x8, sx, w8[0], w8[1], offs, h=h, status=st),
            lambda: moe.quantize_rows_fp8(h, status=st, out=(h8, sh)),
            lambda: moe.grouped_gemm_down_fp8(h8, sh, w8[2], w8[3], offs, y_perm=y, status=st, ksplit=v["ksplit"]),
            lambda: moe.combine(y, wts, dest, out=out, status=st, ksplit=v["ksplit"]),
        ]
    else:
        xp = v["x_perm"]
        calls = [
            (lambda: moe.route_grouped(l_d, bias_d, w.k, *w.router[1:4], idx=idx, w=wts)) if grouped else
            (lambda: moe.route(l_d, w.k, idx=idx, w=wts)),
            lambda: moe.permute(idx, x_d, w.E, status=st, out=(counts_d, offs, src, dest, xp)),
            lambda: moe.grouped_gemm_gateup_swiglu(xp, wgu, offs, h=h, status=st),
            lambda: moe.grouped_gemm_down(h, wd, offs, y_perm=y, status=st, ksplit=v["ksplit"]),
            lambda: moe.combine(y, wts, dest, out=out, status=st, ksplit=v["ksplit"]),
        ]
    ns = len(stages)
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(ns + 1)] for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        sev[i][0].record(stream)
        for j, c in enumerate(calls):
            c()
            sev[i][j + 1].record(stream)
    torch.cuda.synchronize(dev)
    stage_ms = {name: statistics.mean(sev[i][j].elapsed_time(sev[i][j + 1]) for i in range(args.steps))
                for j, name in enumerate(stages)}
    staged_step_ms = statistics.mean(sev[i][0].elapsed_time(sev[i][ns]) for i in range(args.steps))

    # ---- e2e: host buffers in, layer, host buffer out, every step ---------------------------------
    # bf16 softmax router: one moe_forward_host_batches call over the K steps (each step's x and
    # logits copied in and its out copied back, on two copy streams beside the layers).  Grouped
    # router and FP8: per step, the host->device copies, the layer and the copy back, each
    # enqueued on the stream by the binding.
    xh, lh = x.pin_memory(), logits.pin_memory()
    oh = torch.empty(w.T, w.d, dtype=torch.bfloat16).pin_memory()
    batched = flush is None
    if batched:
        ohs = [oh, torch.empty_like(oh).pin_memory()]
        wsize = moe.workspace_size_fp8b if blocks else moe.workspace_size_fp8 if fp8 else moe.workspace_size
        ws_b = torch.empty(wsize(w.T, w.d, w.f, w.E, w.k) + 2 * moe.host_staging_size(w.T, w.d, w.E),
                           dtype=torch.uint8, device=dev)
        h2d, d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

        def e2e_run(n):
            outs = [ohs[i & 1] for i in range(n)]
            if grouped:
                G, tg, sc = w.router[1:4]
                if fp8:
                    moe.forward_grouped_fp8_host_batches([xh] * n, [lh] * n, bias_d, *w8, w.k, G, tg, sc, outs, ws_b,
                                                         stream, h2d, d2h, blocks=blocks)
                else:
                    moe.forward_grouped_host_batches([xh] * n, [lh] * n, bias_d, wgu, wd, w.k, G, tg, sc, outs, ws_b,
                                                     stream, h2d, d2h)
            elif fp8:
                fwd = moe.forward_fp8b_host_batches if blocks else moe.forward_fp8_host_batches
                fwd([xh] * n, [lh] * n, *w8, w.k, outs, ws_b, stream, h2d, d2h)
            else:
                moe.forward_host_batches([xh] * n, [lh] * n, wgu, wd, w.k, outs, ws_b, stream, h2d, d2h)

        e2e_run(max(1, args.warmup))
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_run(args.steps)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = e0.elapsed_time(e1) / args.steps
        e2e_api = ("moe_forward_" + ("grouped_" if grouped else "") + ("fp8b_" if blocks else "fp8_" if fp8 else "") +
                   "host_batches: K batches, copies on two copy streams beside the layers")
        if moe.get_device_error(ws_b) != 0:
            raise RuntimeError("device status word set during the e2e run")
    else:
        def e2e_step():
            if grouped or fp8:
                x_d.copy_(xh, non_blocking=True)
                l_d.copy_(lh, non_blocking=True)
                step()
                oh.copy_(out, non_blocking=True)
            else:
                moe.forward_host(xh, lh, wgu, wd, w.k, oh, ws)

        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize(dev)
        eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for i in range(args.steps):
            if flush is not None:
                flush.zero_()
            eev[i][0].record(stream)
            e2e_step()
            eev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = statistics.mean(a.elapsed_time(b) for a, b in eev)
        e2e_api = ("per step on one stream: host-to-device copies, the layer, the copy back" if (grouped or fp8)
                   else "moe_forward_host, one call per step")
    if moe.get_device_error(ws) != 0:
        raise RuntimeError("device status word set during the timed region")

    peaks, peak_src = load_peaks()
    sw = stage_work(w, n_active, fp8, blocks, fuse_h)
    lw = layer_work(w, n_active, fp8, blocks)
    dom = max(("gateup_swiglu", "down"), key=lambda n: stage_ms[n])
    dom_ms = stage_ms[dom]
    tensor_peak = peaks["bf16_tflops"] * (FP8_OVER_BF16 if fp8 else 1.0)
    t_mem = sw[dom]["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_cmp = sw[dom]["flops"] / (tensor_peak * 1e12)
    if t_cmp > t_mem:
        achieved = sw[dom]["flops"] / (dom_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(tensor_peak, 1),
                "unit": "TFLOP/s"}
    else:
        achieved = sw[dom]["bytes"] / (dom_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["traffic"], roof["traffic_source"] = measured_traffic(w.name, dom + ("_fp8b" if blocks else "_fp8" if fp8
                                                                               else ""))
    kname = KERNEL_NAMES_FP8B[dom] if blocks else (KERNEL_NAMES_FP8[dom] if fp8 else KERNEL_NAMES[dom])
    if blocks and fuse_h and dom == "gateup_swiglu":
        kname = "grouped_gemm_fp8b_kernel<0, true>"
    pair_mode = 0 if blocks else (moe.gemm_pair_mode_fp8 if fp8 else moe.gemm_pair_mode)(
        w.T, w.d, w.f, w.E, w.k, 0 if dom == "gateup_swiglu" else 1)
    if pair_mode >= 1:  # SM-pair kernel, template <KIND, SWAPCAP, GATHER, FP8>
        kname = "grouped_gemm_2sm_kernel<%d, %s, false, %s>" % (0 if dom == "gateup_swiglu" else 1,
                                                                "true" if pair_mode == 2 else "false",
                                                                "true" if fp8 else "false")
    psrc = peak_src + " (burst)" + (" x 2 (nominal fp8 / bf16 dense rate)" if fp8 and roof["bound"] == "tensor" else "")
    roof.update({"kernel": kname, "peak_source": psrc,
                 "algorithmic_per_launch": sw[dom]["flops"] if roof["bound"] == "tensor" else sw[dom]["bytes"],
                 "launch_ms": round(dom_ms, 4)})
    layer_roof_ms = 1e3 * max(lw["bytes"] / (peaks["hbm_gbs"] * 1e9), lw["flops"] / (tensor_peak * 1e12))

    return {
        "ms": ms_max, "steps": args.steps, "tokens_per_rank": w.T, "t_wall": t_wall, "clocks": clocks, "stage_ms": stage_ms,
        "staged_step_ms": staged_step_ms, "e2e_ms": e2e_ms, "e2e_api": e2e_api, "roofline": roof, "layer": lw,
        "layer_roof_ms": layer_roof_ms, "n_active": n_active, "max_load": int(counts.max()),
        "host_weights": (wgu, wd), "inputs": (logits, x), "step_ms_p10_p90": (
            float(np.percentile(step_ms, 10)), float(np.percentile(step_ms, 90))),
        "peak_src": peak_src, "peaks": peaks, "ksplit": v["ksplit"],
        # DeepSeek-V3's router never fuses with the permutation: 5 (bf16), 6 (e4m3), 6 or 7 (e4m3b),
        # one fewer for bf16 and e4m3 when the combine is folded into the down GEMM (MOE_FOLD_COMBINE=1).
        "launches_per_step": (((7 - int(fuse_h)) if blocks else
                               (6 if fp8 else 5) - int(os.environ.get("MOE_FOLD_COMBINE", "0") == "1"))
                              if grouped else
                              moe.forward_fp8b_launch_count(w.T, w.E, w.k) if blocks else
                              moe.forward_fp8_launch_count(w.T, w.E, w.k) if fp8 else
                              moe.forward_launch_count(w.T, w.E, w.k)),
    }


# ----------------------------------------------------------------------------------------------
# Oracle timing (CPU baseline and the reference arm)
# ----------------------------------------------------------------------------------------------
def oracle_sample_runner(w: Workload, logits, x, wgu, wd, seed: int = 0, fp8: bool = False, blocks: bool = False):
    import oracle as oracle_pkg
    O = oracle_pkg.Oracle()
    xb = bf16_bits(x)
    ln = logits.numpy()
    wgub, wdb = bf16_bits(wgu), bf16_bits(wd)
    bias = draw_router_bias(w, seed).numpy()
    if blocks:
        w8 = O.quantize_weights_fp8b(wgub) + O.quantize_weights_fp8b(wdb)  # once, untimed
    else:
        w8 = O.quantize_weights_fp8(wgub) + O.quantize_weights_fp8(wdb) if fp8 else None

    def run(S: int) -> float:
        t0 = time.perf_counter()
        if fp8 and w.router[0] == "grouped":
            idx, wts = O.route_grouped(ln[:S], bias, w.k, *w.router[1:4])
            fwd = O.forward_fp8b_tokens_routed if blocks else O.forward_fp8_tokens_routed
            fwd(xb, idx, wts, *w8, np.arange(S, dtype=np.int32))
        elif blocks:
            O.forward_fp8b(xb[:S], ln[:S], *w8, w.k)
        elif fp8:
            O.forward_fp8(xb[:S], ln[:S], *w8, w.k)
        elif w.router[0] == "grouped":
            idx, wts = O.route_grouped(ln[:S], bias, w.k, *w.router[1:4])
            O.forward_routed(xb[:S], idx, wts, wgub, wdb)
        else:
            O.forward(xb[:S], ln[:S], wgub, wdb, w.k)
        return time.perf_counter() - t0

    return O, run


def pick_sample(run, T: int, budget_s: float) -> int:
    """Largest token count S <= T whose oracle forward should take about budget_s."""
    S = min(T, 2)
    t = max(run(S), 1e-4)
    while S < T and t < budget_s / 4:
        S = min(T, S * 4)
        t = max(run(S), 1e-4)
    S = max(1, min(T, int(S * budget_s / t)))
    return S


def passes_for(run, S: int, budget_s: float) -> int:
    """Whole passes over the S-token sample that fill about budget_s (a small batch is run again)."""
    return max(1, int(budget_s / max(run(S), 1e-4)))


def cpu_baseline(w, logits, x, wgu, wd, budget_s: float, seed: int = 0, fp8: bool = False, blocks: bool = False):
    O, run = oracle_sample_runner(w, logits, x, wgu, wd, seed, fp8, blocks)
    S = pick_sample(run, w.T, budget_s)
    R = passes_for(run, S, budget_s)
    dt = sum(run(S) for _ in range(R))
    what = ("FP8 oracle forward (route, permute, x/h quantisation, E4M3 gate+up/SwiGLU and down, combine; "
            f"{'128-wide block' if blocks else 'per-row / per-channel'} scales; weights quantised beforehand, "
            "untimed)" if fp8 else
            "oracle forward (route, permute, gate+up/SwiGLU, down, combine)")
    return {"value": round(R * S / dt, 3), "unit": "tokens/s", "cores": O.num_threads(), "kind": "oracle",
            "sample": f"{what} on the first {S} of {w.T} tokens of the same seeded batch, full weights, "
                      f"{R} pass{'es' if R > 1 else ''}, {dt:.1f} s"}


def run_reference(args, w: Workload, rank: int, world: int):
    if rank != 0:
        return None
    logits, x, wgu, wd = make_inputs(w, seed=args.seed, weight_device="cuda" if torch.cuda.is_available() else "cpu")
    wgu, wd = wgu.cpu(), wd.cpu()
    blocks = args.dtype == "e4m3b"
    fp8 = args.dtype == "e4m3" or blocks
    O, run = oracle_sample_runner(w, logits, x, wgu, wd, args.seed, fp8, blocks)
    n = args.steps + args.warmup
    per_step = args.ref_step_s if args.ref_step_s else max(0.5, min(20.0, 150.0 / max(1, n)))
    S = pick_sample(run, w.T, per_step)
    R = passes_for(run, S, per_step)
    for _ in range(args.warmup):
        run(S)
    times = [sum(run(S) for _ in range(R)) for _ in range(args.steps)]
    ms = 1e3 * statistics.mean(times)
    value = R * S / (ms * 1e-3)
    sample = (f"each step: {'FP8 ' if fp8 else ''}oracle forward on the first {S} of {w.T} tokens of the seeded "
              f"batch, {R} pass{'es' if R > 1 else ''}, full weights, {O.num_threads()} host threads")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded)", "config": config_of(w, args),
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": O.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def config_of(w: Workload, args) -> dict:
    return {"workload": w.name, "T": w.T, "d_model": w.d, "d_ff": w.f, "experts": w.E, "top_k": w.k,
            "logit_bias": list(w.bias), "router": list(w.router), "seed": args.seed, "parallelism": "replicas",
            "gemm_operands": {"e4m3": "e4m3, per-row activation and per-output-channel weight scales",
                              "e4m3b": "e4m3, power-of-two scales per 1x128 activation and 128x128 weight block"}
                             .get(args.dtype, "bf16"),
            "l2": ("flushed between steps (512 MB write, outside the step events)" if args.flush_l2 else
                   "not flushed: inputs larger than L2 (the active experts' weights, >= 2.8 GB, stream "
                   "from HBM every step; L2 is 129 MB)")}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: enough for ~0.5 s of device time, 50..4000; 20 for --impl reference)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-budget-s", type=float, default=12.0, help="oracle CPU-baseline sample size, seconds")
    ap.add_argument("--ref-step-s", type=float, default=None,
                    help="--impl reference: CPU seconds per step (default: ~150 s over all steps, 0.5..20 per step)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "e4m3", "e4m3b"],
                    help="operands of the grouped GEMMs: bf16 (moe_forward), e4m3 (moe_forward_fp8) or e4m3 with "
                         "block scales (moe_forward_fp8b)")
    ap.add_argument("--per-workload", default=",".join(PER_WORKLOAD),
                    help="comma-separated workloads also measured in this process and reported under per_workload "
                         "(default: %(default)s), or 'none'")
    ap.add_argument("--flush-l2", action="store_true",
                    help="write a 512 MB buffer between steps (default: rely on inputs larger than L2)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    w = WORKLOADS[args.workload]
    unknown = [n for n in args.per_workload.split(",") if n and n != "none" and n not in WORKLOADS]
    if unknown:
        ap.error(f"--per-workload: unknown workload(s) {unknown}")

    if args.impl == "reference":
        if args.steps is None:
            args.steps = 20
        line = run_reference(args, w, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    steps_arg = args.steps
    t_bench0 = time.perf_counter()
    r = run_ours(args, w, rank, world, dist)
    line = result_line(r, w, args, world) if rank == 0 else None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        logits, x = r["inputs"]
        wgu, wd = (t.cpu() for t in r["host_weights"])
        line["cpu_baseline"] = cpu_baseline(w, logits, x, wgu, wd, args.cpu_budget_s, args.seed,
                                            args.dtype != "bf16", args.dtype == "e4m3b")
        del wgu, wd
    timed_s = r["t_wall"]
    del r
    names = [] if args.per_workload == "none" else [n for n in args.per_workload.split(",") if n and n != w.name]
    per = {}
    for name in names:
        torch.cuda.empty_cache()
        args.steps = steps_arg  # each workload takes its own K when --steps is not given
        wl = WORKLOADS[name]
        rr = run_ours(args, wl, rank, world, dist)
        timed_s += rr["t_wall"]
        if rank == 0:
            full = result_line(rr, wl, args, world)
            per[name] = {key: full[key] for key in (
                "value", "unit", "ms_per_step", "steps", "tflops", "layer_roofline", "roofline", "e2e", "clocks",
                "stage_ms", "step_ms_p10_p90", "active_experts", "max_expert_load", "gpu_launches")}
            per[name]["config"] = {key: full["config"][key] for key in (
                "T", "d_model", "d_ff", "experts", "top_k", "logit_bias", "router")}
        del rr
    if rank == 0:
        if per:
            line["per_workload"] = per
        line["timed_region_s_all_workloads"] = round(timed_s, 3)
        line["bench_wall_s"] = round(time.perf_counter() - t_bench0, 1)
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def result_line(r: dict, w: Workload, args, world: int) -> dict:
    """The JSON fields of one workload's measurement (rank 0)."""
    tok_s = job_tokens_per_s(r["tokens_per_rank"], world, r["ms"])
    tflops = r["layer"]["flops"] * world / (r["ms"] * 1e-3) / 1e12
    return {
        "metric": METRIC, "value": round(tok_s, 2), "unit": "tokens/s", "n_gpus": world,
        "steps": r["steps"], "warmup": args.warmup, "ms_per_step": round(r["ms"], 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.dtype,
        "data": "synthetic (seeded)", "config": config_of(w, args),
        "tflops": round(tflops, 2),
        "layer_roofline": {"ms": round(r["layer_roof_ms"], 4), "frac": round(r["layer_roof_ms"] / r["ms"], 4),
                           "bytes": r["layer"]["bytes"], "flops": r["layer"]["flops"],
                           "peaks": r["peak_src"]},
        "roofline": r["roofline"],
        "stage_ms": {k: round(v, 4) for k, v in r["stage_ms"].items()},
        "staged_step_ms": round(r["staged_step_ms"], 4),
        "step_ms_p10_p90": [round(v, 4) for v in r["step_ms_p10_p90"]],
        "active_experts": r["n_active"], "max_expert_load": r["max_load"], "down_ksplit": r["ksplit"],
        "e2e": {"value": round(w.T / (r["e2e_ms"] * 1e-3), 2), "unit": "tokens/s",
                "h2d_bytes_per_step": w.T * w.d * 2 + w.T * w.E * 4, "d2h_bytes_per_step": w.T * w.d * 2,
                "ms_per_step": round(r["e2e_ms"], 4), "api": r["e2e_api"]},
        "gpu_launches": r["launches_per_step"] * r["steps"],
        "clocks": r["clocks"],
        "timed_region_s": round(r["t_wall"], 3),
    }


if __name__ == "__main__":
    main()
