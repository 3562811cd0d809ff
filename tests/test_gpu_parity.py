"""GPU parity: every step of the CUDA path against the CPU oracle on the same seeded inputs,
through the C ABI (libmoe.so via its ctypes binding).  Sizes here finish in seconds on the oracle
while spanning several tiles, ragged expert segments, partial N tiles, more work items than
SMs (so the persistent loop wraps its pipeline and both accumulators), and the degenerate cases.
"""
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
from gpu_cases import (assert_close, assert_layer_close, case_inputs, from_np_bits,  # noqa: E402
                       random_bf16, to_np_bits)

from mixture_experts_grouped_fp32_gb300.workloads import WORKLOADS, Workload  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_grouped_fp32_gb300 import moe as m
    m.load()
    return m


# (name, Workload) — the layer shapes checked end to end against the oracle's full forward.
CASES = [
    WORKLOADS["tiny"],
    Workload("ragged_multi_tile", 300, 512, 768, 8, 2),
    Workload("many_items_per_cta", 4096, 256, 2048, 2, 1),
    Workload("partial_n_tiles_k_eq_e", 37, 192, 320, 4, 4),
    Workload("zipf_skew_zero_token_experts", 256, 256, 384, 64, 6, ("zipf", 1.2)),
    Workload("one_hot_expert", 200, 128, 256, 8, 1, ("hot0", 40.0)),
    Workload("single_token", 1, 128, 128, 8, 2),
    Workload("dense_e1_k1", 70, 128, 192, 1, 1),
    Workload("minimal_dims", 50, 64, 64, 3, 2),
    Workload("deepseek_like_wide_d", 40, 1024, 256, 32, 8, ("zipf", 1.2)),
    Workload("hot_expert_mid_experts", 700, 256, 512, 8, 2, ("hot0", 2.2)),
]


def _forward_and_views(moe, w, logits, x, wgu, wd):
    dev = torch.device(DEV)
    ws = torch.empty(moe.workspace_size(w.T, w.d, w.f, w.E, w.k), dtype=torch.uint8, device=dev)
    ws.fill_(0xFF)  # NaN-ish sentinel everywhere: every consumed intermediate must be written
    out = moe.forward(x.to(dev), logits.to(dev), wgu.to(dev), wd.to(dev), w.k, workspace=ws)
    torch.cuda.synchronize()
    return out, moe.workspace_views(ws, w.T, w.d, w.f, w.E, w.k), ws


# GEMM path variants: the default policy (small experts swapped on the 1-SM kernel, SM pairs when
# the average expert has >= 128 rows, few-token down GEMM split over K), the 1-SM kernel with every
# expert in the normal orientation, the SM-pair kernel for every shape in its normal-only form and
# in its swapping form (thresholds 128 and 64 rows; and with its CTA pairs split between normal
# tiles and swapped chunks), a forced 3-way K split, and routing and the permutation as two
# launches where the default fuses them (E <= 32).
MODES = {"default": {}, "noswap": {"MOE_GEMM_SWAP_MAX": "0", "MOE_GEMM_2SM": "0"},
         "pair": {"MOE_GEMM_2SM": "1"}, "pairswap": {"MOE_GEMM_2SM": "2", "MOE_GEMM_PAIR_SPLIT": "0"},
         "pairswap64": {"MOE_GEMM_2SM": "2", "MOE_GEMM_PAIR_SWAP_MAX": "64"},
         "pairsplit": {"MOE_GEMM_2SM": "2", "MOE_GEMM_PAIR_SPLIT": "30"},
         "pairmix": {"MOE_GEMM_2SM": "2", "MOE_GEMM_PAIR_SPLIT": "mix"},
         "pairauto": {"MOE_GEMM_2SM": "2", "MOE_GEMM_PAIR_SPLIT": "auto"},
         "ksplit3": {"MOE_DOWN_KSPLIT": "3"}, "nofuse": {"MOE_FUSE_ROUTE_PERMUTE": "0"},
         "gather": {"MOE_GATHER": "1"}}
ENV_KNOBS = ("MOE_GEMM_SWAP_MAX", "MOE_DOWN_KSPLIT", "MOE_GEMM_2SM", "MOE_GEMM_PAIR_SWAP_MAX", "MOE_GEMM_2SM_DOWN",
             "MOE_FUSE_ROUTE_PERMUTE", "MOE_GEMM_PAIR_LAYOUT", "MOE_GEMM_PAIR_SPLIT", "MOE_GATHER")


@pytest.fixture(params=sorted(MODES))
def mode(request, monkeypatch):
    for k in ENV_KNOBS:
        monkeypatch.delenv(k, raising=False)
    for k, v in MODES[request.param].items():
        monkeypatch.setenv(k, v)
    return request.param


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_forward_matches_oracle(moe, oracle, w, mode):
    logits, x, wgu, wd = case_inputs(w, seed=0)
    out, v, ws = _forward_and_views(moe, w, logits, x, wgu, wd)
    assert moe.get_device_error(ws) == 0
    ln = logits.numpy()
    idx, wt = oracle.route(ln, w.k)
    counts, offsets, src, dest = oracle.permute(idx, w.E)
    assert np.array_equal(v["idx"].cpu().numpy(), idx)
    assert_close(v["w"].cpu().numpy(), wt, 1e-6, 0, "route weights")
    assert np.array_equal(v["counts"].cpu().numpy(), counts)
    assert np.array_equal(v["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(v["src"].cpu().numpy(), src)
    assert np.array_equal(v["dest"].cpu().numpy(), dest)
    if mode != "gather":  # with MOE_GATHER=1 the gate+up GEMM gathers x rows itself; x_perm is unused
        assert np.array_equal(to_np_bits(v["x_perm"].cpu()), to_np_bits(x)[src])
    ref = oracle.forward(to_np_bits(x), ln, to_np_bits(wgu), to_np_bits(wd), w.k)
    assert_layer_close(out.float().cpu().numpy(), ref, w.name)


@pytest.mark.parametrize("mode", ["default", "noswap", "pair", "pairswap", "pairsplit", "ksplit3"])
@pytest.mark.parametrize("w", [CASES[1], CASES[3], CASES[4], CASES[5], CASES[6], CASES[8], CASES[9], CASES[10]],
                         ids=lambda w: w.name)
def test_folded_combine_equals_combine_kernel(moe, w, mode, monkeypatch):
    """The combine folded into the down GEMM (MOE_FOLD_COMBINE=1: the last arrival of a token's
    64-column block sums its k rows in slot order) gives the combine kernel's output bit for bit,
    for every down-GEMM form (1-SM normal and swapped items, SM-pair normal and swapped items, K
    split in three), and in a CUDA graph with the same node count moe_forward_launch_count states."""
    for key in ENV_KNOBS:
        monkeypatch.delenv(key, raising=False)
    for key, val in MODES[mode].items():
        monkeypatch.setenv(key, val)
    logits, x, wgu, wd = case_inputs(w, seed=8)
    dev = torch.device(DEV)
    args = (x.to(dev), logits.to(dev), wgu.to(dev), wd.to(dev), w.k)
    ref = moe.forward(*args)
    monkeypatch.setenv("MOE_FOLD_COMBINE", "1")
    ws = torch.empty(moe.workspace_size(w.T, w.d, w.f, w.E, w.k), dtype=torch.uint8, device=dev)
    ws.fill_(0x7F)  # counters must be zeroed by the permute
    for _ in range(2):  # the second call reuses counters the first one left at their targets
        out = moe.forward(*args, workspace=ws)
        torch.cuda.synchronize()
        assert moe.get_device_error(ws) == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"{w.name} [{mode}]"


def test_forward_is_deterministic(moe):
    w = Workload("det", 300, 512, 768, 8, 2)
    logits, x, wgu, wd = case_inputs(w, seed=3)
    a, _, _ = _forward_and_views(moe, w, logits, x, wgu, wd)
    b, _, _ = _forward_and_views(moe, w, logits, x, wgu, wd)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ------------------------------------------------------------------------------------------
# Stage by stage, each stage fed seeded inputs (never the CUDA path's own outputs).
# ------------------------------------------------------------------------------------------
@pytest.mark.parametrize("T,E,k,ties", [(4096, 8, 2, False), (513, 256, 8, False), (333, 64, 6, True),
                                        (77, 5, 5, True), (1, 8, 1, False), (1000, 33, 3, False),
                                        (64, 8, 2, True)])
def test_route_parity(moe, oracle, T, E, k, ties):
    g = torch.Generator("cpu").manual_seed(T * 7 + E)
    logits = (torch.randint(0, 2, (T, E), generator=g).float() if ties
              else torch.randn(T, E, generator=g))
    idx, w = moe.route(logits.to(DEV), k)
    torch.cuda.synchronize()
    ridx, rw = oracle.route(logits.numpy(), k)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert_close(w.cpu().numpy(), rw, 1e-6, 0, "route weights")


def _nan_logits(T, E, seed):
    """Logits with NaN rows of every kind: one NaN, several, all NaN, -inf beside a NaN, and fewer
    numbers than slots.  The pages define no non-finite logits; both sides rank NaN below every
    number with NaNs by ascending id, so the ids are still compared bit for bit."""
    g = torch.Generator("cpu").manual_seed(seed)
    lg = torch.randn(T, E, generator=g)
    lg[1:9, 2 % E] = float("nan")
    lg[9:13, [0, E - 1]] = float("nan")
    lg[13:15, :] = float("nan")
    lg[15:17, 1] = float("-inf")
    lg[15:17, E - 2] = float("nan")
    lg[17:19, :E - 2] = float("nan")
    return lg


@pytest.mark.parametrize("E,k", [(8, 2), (8, 3), (64, 6), (256, 8)])
def test_route_nan_logits_order(moe, oracle, E, k):
    logits = _nan_logits(64, E, seed=E + k)
    idx, w = moe.route(logits.to(DEV), k)
    torch.cuda.synchronize()
    ridx, rw = oracle.route(logits.numpy(), k)
    gi = idx.cpu().numpy()
    assert np.array_equal(gi, ridx)
    assert all(len(set(r)) == k for r in gi.tolist())  # no expert in two slots of one token
    clean = torch.isfinite(logits).all(dim=1).numpy()
    assert_close(w.cpu().numpy()[clean], rw[clean], 1e-6, 0, "route weights, finite rows")


def test_fused_route_permute_nan_logits_order(moe, oracle, monkeypatch):
    # E <= 32 and T*E <= 8192: moe_forward routes inside the permute kernel (one thread per token).
    w = Workload("nan_fused", 64, 128, 128, 8, 2)
    _, x, wgu, wd = case_inputs(w, seed=5)
    logits = _nan_logits(w.T, w.E, seed=77)
    fused = moe.forward_launch_count(w.T, w.E, w.k)
    monkeypatch.setenv("MOE_FUSE_ROUTE_PERMUTE", "0")
    assert moe.forward_launch_count(w.T, w.E, w.k) == fused + 1
    monkeypatch.delenv("MOE_FUSE_ROUTE_PERMUTE")
    _, v, ws = _forward_and_views(moe, w, logits, x, wgu, wd)
    ridx, rw = oracle.route(logits.numpy(), w.k)
    assert np.array_equal(v["idx"].cpu().numpy(), ridx)
    counts, offsets, src, dest = oracle.permute(ridx, w.E)
    assert np.array_equal(v["src"].cpu().numpy(), src)
    assert np.array_equal(v["dest"].cpu().numpy(), dest)
    clean = torch.isfinite(logits).all(dim=1).numpy()
    assert_close(v["w"].cpu().numpy()[clean], rw[clean], 1e-6, 0, "route weights, finite rows")


@pytest.mark.parametrize("nt", ["", "256", "512", "1024"])
@pytest.mark.parametrize("T,d,E,k", [(4096, 4096, 8, 2), (2048, 256, 256, 8), (37, 64, 4, 4), (1, 128, 8, 2),
                                     (999, 192, 64, 6), (12000, 64, 8, 2), (16000, 64, 64, 8)])
def test_permute_parity(moe, oracle, T, d, E, k, nt, monkeypatch):
    """The permutation bit for bit at every block size (MOE_PERM_THREADS; "" = the default rule),
    including grids at the tokens-per-block cap (T = 12000 and 16000)."""
    if nt:
        monkeypatch.setenv("MOE_PERM_THREADS", nt)
    g = torch.Generator("cpu").manual_seed(T + d)
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).int()
    x = random_bf16((T, d), seed=T)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    counts, offsets, src, dest, x_perm = moe.permute(idx.to(DEV), x.to(DEV), E, status=status)
    torch.cuda.synchronize()
    rc, ro, rs, rd = oracle.permute(idx.numpy(), E)
    assert int(status.item()) == 0
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(src.cpu().numpy(), rs)
    assert np.array_equal(dest.cpu().numpy(), rd)
    assert np.array_equal(to_np_bits(x_perm.cpu()), oracle.gather_rows(to_np_bits(x), rs))


@pytest.mark.parametrize("nt", ["256", "512", "1024"])
def test_fused_route_permute_block_sizes(moe, oracle, nt, monkeypatch):
    """Route + permute in one kernel (E <= 32, T*E <= 8192) at every block size: idx, w, src, dest
    and x_perm against the oracle."""
    monkeypatch.setenv("MOE_PERM_THREADS", nt)
    w = Workload("fused_block_sizes", 1000, 128, 128, 8, 2)
    logits, x, wgu, wd = case_inputs(w, seed=21)
    _, v, ws = _forward_and_views(moe, w, logits, x, wgu, wd)
    ridx, rw = oracle.route(logits.numpy(), w.k)
    assert np.array_equal(v["idx"].cpu().numpy(), ridx)
    assert_close(v["w"].cpu().numpy(), rw, 1e-6, 0, "route weights")
    counts, offsets, src, dest = oracle.permute(ridx, w.E)
    assert np.array_equal(v["src"].cpu().numpy(), src)
    assert np.array_equal(v["dest"].cpu().numpy(), dest)
    assert np.array_equal(to_np_bits(v["x_perm"].cpu()), oracle.gather_rows(to_np_bits(x), src))


def _segments(oracle, T, E, k, seed, bias=("none", 0.0)):
    from mixture_experts_grouped_fp32_gb300.workloads import draw_routing
    logits, _ = draw_routing(T, 64, E, seed, bias)
    idx, _ = oracle.route(logits.numpy(), k)
    counts, offsets, _, _ = oracle.permute(idx, E)
    return offsets


GEMM_CASES = [  # (T, d, f, E, k, bias); row counts per expert at the seeds used below
    (300, 512, 768, 8, 2, ("none", 0.0)),     # 62-90 rows each
    (4096, 256, 2048, 2, 1, ("none", 0.0)),   # ~2048 each: 256-row tiles, one a 1-row remainder
    (37, 192, 320, 4, 4, ("none", 0.0)),      # 37 each, partial N tiles on both GEMMs
    (256, 256, 384, 64, 6, ("zipf", 1.2)),    # 250 down to 0 rows
    (200, 128, 256, 8, 1, ("hot0", 40.0)),    # one expert holds all 200 rows
    (600, 256, 512, 2, 1, ("none", 0.0)),     # 309 / 291: one 256-row tile plus a short remainder
    (700, 256, 512, 8, 2, ("hot0", 2.2)),     # ~630 + 96..143: the pair kernel's 40 KB-stage layout
]


def _set_gemm_env(monkeypatch, swap_max, pair):
    """pair "2:<n>" selects the swapping SM-pair kernel with threshold n (and its default,
    device-chosen schedule), "2:<n>:<p>" fixes the schedule (0 round-robin, p pairs on normal
    tiles, "mix", "auto")."""
    monkeypatch.setenv("MOE_GEMM_SWAP_MAX", swap_max)
    parts = pair.split(":")
    monkeypatch.setenv("MOE_GEMM_2SM", parts[0])
    monkeypatch.delenv("MOE_GEMM_2SM_DOWN", raising=False)
    for name, i in (("MOE_GEMM_PAIR_SWAP_MAX", 1), ("MOE_GEMM_PAIR_SPLIT", 2)):
        if len(parts) > i:
            monkeypatch.setenv(name, parts[i])
        else:
            monkeypatch.delenv(name, raising=False)


@pytest.mark.parametrize("swap_max,pair", [("128", "0"), ("0", "0"), ("64", "1"), ("64", "2:128"),
                                           ("64", "2:64"), ("64", "2:0"), ("64", "2:128:40"), ("64", "2:64:1"),
                                           ("64", "2:128:mix"), ("64", "2:128:auto"),
                                           ("64", "2:128:0")])
@pytest.mark.parametrize("T,d,f,E,k,bias", GEMM_CASES)
def test_gateup_swiglu_parity(moe, oracle, T, d, f, E, k, bias, swap_max, pair, monkeypatch):
    _set_gemm_env(monkeypatch, swap_max, pair)
    offsets = _segments(oracle, T, E, k, seed=11, bias=bias)
    M = T * k
    x_perm = random_bf16((M, d), seed=5)
    _, _, wgu, _ = case_inputs(Workload("g", 1, d, f, E, 1), seed=2)
    extra = 3  # rows past offsets[E] must stay untouched
    h = torch.full((M + extra, f), float("nan"), dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    xp = torch.cat([x_perm, torch.zeros(extra, d, dtype=torch.bfloat16)]).to(DEV)
    moe.grouped_gemm_gateup_swiglu(xp, wgu.to(DEV), torch.from_numpy(offsets).to(DEV), h=h, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.gateup_swiglu(to_np_bits(x_perm), offsets, to_np_bits(wgu))
    got = h[:M].float().cpu().numpy()
    assert np.isfinite(got).all(), "some h rows were not written"
    assert torch.isnan(h[M:].float()).all(), "rows past offsets[E] were written"
    assert float(np.abs(got - ref).max()) <= 1e-2 * float(np.abs(ref).max())
    assert_close(got, ref, 2.0 ** -7, 2e-3, "h")


@pytest.mark.parametrize("swap_max,pair", [("128", "0"), ("0", "0"), ("64", "1"), ("64", "2:128:0"),
                                           ("64", "2:64:0"), ("64", "2:128:auto"), ("64", "2:64:40")])
@pytest.mark.parametrize("T,d,f,E,k,bias", GEMM_CASES)
def test_gateup_swiglu_gather_parity(moe, oracle, T, d, f, E, k, bias, swap_max, pair, monkeypatch):
    """The gate+up GEMM gathering its rows from x by src (what moe_forward runs) against the oracle
    applied to x[src]: every kernel form, with src a random permutation-with-repeats of x's rows."""
    _set_gemm_env(monkeypatch, swap_max, pair)
    offsets = _segments(oracle, T, E, k, seed=11, bias=bias)
    M = T * k
    x = random_bf16((T, d), seed=15)
    g = torch.Generator("cpu").manual_seed(T + d)
    src = torch.randint(0, T, (M,), generator=g, dtype=torch.int32)
    _, _, wgu, _ = case_inputs(Workload("g", 1, d, f, E, 1), seed=2)
    extra = 3
    h = torch.full((M + extra, f), float("nan"), dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    moe.grouped_gemm_gateup_swiglu_gather(x.to(DEV), src.to(DEV), wgu.to(DEV), torch.from_numpy(offsets).to(DEV),
                                          h=h, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    xb = to_np_bits(x)
    ref = oracle.gateup_swiglu(oracle.gather_rows(xb, src.numpy()), offsets, to_np_bits(wgu))
    got = h[:M].float().cpu().numpy()
    assert np.isfinite(got).all(), "some h rows were not written"
    assert torch.isnan(h[M:].float()).all(), "rows past offsets[E] were written"
    assert float(np.abs(got - ref).max()) <= 1e-2 * float(np.abs(ref).max())
    assert_close(got, ref, 2.0 ** -7, 2e-3, "h (gathered)")


@pytest.mark.parametrize("swap_max,ksplit,pair", [("128", 1, "0"), ("0", 1, "0"), ("128", 3, "0"), ("0", 5, "0"),
                                                  ("128", 8, "0"), ("64", 1, "1"), ("64", 3, "1"), ("64", 1, "2:128"),
                                                  ("64", 3, "2:64"), ("64", 2, "2:0"), ("64", 1, "2:128:40"),
                                                  ("64", 2, "2:64:75"), ("64", 1, "2:128:mix"),
                                                  ("64", 1, "2:128:auto"), ("64", 1, "2:128:0")])
@pytest.mark.parametrize("T,d,f,E,k,bias", GEMM_CASES)
def test_down_parity(moe, oracle, T, d, f, E, k, bias, swap_max, ksplit, pair, monkeypatch):
    _set_gemm_env(monkeypatch, swap_max, pair)
    offsets = _segments(oracle, T, E, k, seed=12, bias=bias)
    M = T * k
    h = random_bf16((M, f), seed=6, scale=0.5)
    _, _, _, wd = case_inputs(Workload("g", 1, d, f, E, 1), seed=4)
    y = torch.full((ksplit, M, d), float("nan"), dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    moe.grouped_gemm_down(h.to(DEV), wd.to(DEV), torch.from_numpy(offsets).to(DEV), y_perm=y, status=status,
                          ksplit=ksplit)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.down(to_np_bits(h), offsets, to_np_bits(wd))
    parts = y.cpu().numpy()
    assert np.isfinite(parts).all(), "some partial-sum rows were not written"
    got = parts[0].copy()
    for s_ in range(1, ksplit):  # slice order, as the combine step adds them
        got += parts[s_]
    assert np.isfinite(got).all(), "some y rows were not written"
    assert_close(got, ref, 1e-3, 1e-4, "y_perm")


@pytest.mark.parametrize("T,d,E,k,ksplit", [(4096, 4096, 8, 2, 1), (2048, 7168, 256, 8, 1), (37, 192, 4, 4, 1),
                                             (1, 64, 3, 1, 1), (32, 4096, 8, 2, 5), (300, 512, 8, 2, 8)])
def test_combine_parity(moe, oracle, T, d, E, k, ksplit):
    g = torch.Generator("cpu").manual_seed(T + k)
    logits = torch.randn(T, E, generator=g)
    idx, w = oracle.route(logits.numpy(), k)
    _, _, _, dest = oracle.permute(idx, E)
    y = torch.randn(ksplit, T * k, d, generator=g)
    out = moe.combine(y.to(DEV), torch.from_numpy(w).to(DEV), torch.from_numpy(dest).to(DEV), ksplit=ksplit)
    torch.cuda.synchronize()
    ysum = y[0].numpy().copy()
    for s_ in range(1, ksplit):  # the partial slices are added in slice order before weighting
        ysum += y[s_].numpy()
    ref = oracle.combine(ysum, w, dest)
    assert_close(out.float().cpu().numpy(), ref, 2.0 ** -8, 1e-6, "combine")


# ------------------------------------------------------------------------------------------
# Device-side checks: bad data drives no out-of-bounds access; the status word says what.
# ------------------------------------------------------------------------------------------
def test_status_flags_bad_expert_ids(moe):
    idx = torch.tensor([[0, 1], [2, 9], [3, 3]], dtype=torch.int32, device=DEV)
    x = torch.zeros(3, 64, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    moe.permute(idx, x, 4, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & moe.STATUS_BAD_EXPERT_ID


def test_status_flags_bad_offsets(moe):
    E, d, f = 4, 64, 128
    x_perm = torch.zeros(16, d, dtype=torch.bfloat16, device=DEV)
    wgu = torch.zeros(E, d, 2 * f, dtype=torch.bfloat16, device=DEV)
    h = torch.zeros(16, f, dtype=torch.bfloat16, device=DEV)
    for bad in ([0, 5, 3, 8, 16], [0, 4, 8, 12, 17]):  # decreasing; past M
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        offs = torch.tensor(bad, dtype=torch.int32, device=DEV)
        moe.grouped_gemm_gateup_swiglu(x_perm, wgu, offs, h=h, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) & moe.STATUS_BAD_OFFSETS


def test_status_flags_bad_src(moe):
    """A gathering gate+up GEMM given src indices outside [0, T) reads zero rows for them and sets
    MOE_STATUS_BAD_SRC instead of reading out of bounds."""
    E, d, f, T = 2, 64, 128, 8
    x = torch.ones(T, d, dtype=torch.bfloat16, device=DEV)
    wgu = torch.zeros(E, d, 2 * f, dtype=torch.bfloat16, device=DEV)
    h = torch.zeros(16, f, dtype=torch.bfloat16, device=DEV)
    offs = torch.tensor([0, 8, 16], dtype=torch.int32, device=DEV)
    for bad in (T, -1, 1 << 30):
        src = torch.arange(16, dtype=torch.int32, device=DEV) % T
        src[5] = bad
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        moe.grouped_gemm_gateup_swiglu_gather(x, src, wgu, offs, h=h, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) & moe.STATUS_BAD_SRC
        assert torch.isfinite(h.float()).all()


def test_status_flags_bad_dest(moe):
    y = torch.ones(4, 64, dtype=torch.float32, device=DEV)
    w = torch.full((2, 2), 0.5, dtype=torch.float32, device=DEV)
    dest = torch.tensor([[0, 1], [2, 4]], dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = moe.combine(y, w, dest, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & moe.STATUS_BAD_DEST
    assert torch.allclose(out[0].float(), torch.ones(64, device=DEV))


def test_forward_host_matches_forward(moe):
    w = Workload("host", 97, 256, 512, 8, 2)
    logits, x, wgu, wd = case_inputs(w, seed=9)
    dev = torch.device(DEV)
    wgu_d, wd_d = wgu.to(dev), wd.to(dev)
    ref = moe.forward(x.to(dev), logits.to(dev), wgu_d, wd_d, w.k)
    ws = torch.empty(moe.workspace_size(w.T, w.d, w.f, w.E, w.k) + moe.host_staging_size(w.T, w.d, w.E),
                     dtype=torch.uint8, device=dev)
    xh, lh = x.pin_memory(), logits.pin_memory()
    oh = torch.empty(w.T, w.d, dtype=torch.bfloat16).pin_memory()
    moe.forward_host(xh, lh, wgu_d, wd_d, w.k, oh, ws)
    torch.cuda.synchronize()
    assert torch.equal(oh.view(torch.int16), ref.cpu().view(torch.int16))


@pytest.mark.parametrize("n", [1, 2, 5])
def test_forward_host_batches_matches_forward(moe, n):
    """Batches with copies overlapped on two copy streams give each batch's moe_forward output."""
    w = Workload("host_batches", 97, 256, 512, 8, 2)
    dev = torch.device(DEV)
    _, _, wgu, wd = case_inputs(w, seed=11)
    wgu_d, wd_d = wgu.to(dev), wd.to(dev)
    xs, ls, refs = [], [], []
    for i in range(n):
        logits, x, _, _ = case_inputs(w, seed=20 + i)
        xs.append(x.pin_memory())
        ls.append(logits.pin_memory())
        refs.append(moe.forward(x.to(dev), logits.to(dev), wgu_d, wd_d, w.k).cpu())
    outs = [torch.full((w.T, w.d), -1.0, dtype=torch.bfloat16).pin_memory() for _ in range(n)]
    ws = torch.empty(moe.workspace_size(w.T, w.d, w.f, w.E, w.k) + 2 * moe.host_staging_size(w.T, w.d, w.E),
                     dtype=torch.uint8, device=dev)
    moe.forward_host_batches(xs, ls, wgu_d, wd_d, w.k, outs, ws)
    torch.cuda.current_stream().synchronize()  # the call orders its copies before the stream's end
    assert moe.get_device_error(ws) == 0
    for i in range(n):
        assert torch.equal(outs[i].view(torch.int16), refs[i].view(torch.int16)), f"batch {i}"


def _cudart():
    import ctypes
    import glob
    try:
        return ctypes.CDLL("libcudart.so.13")
    except OSError:
        for c in glob.glob(os.path.join(os.path.dirname(torch.__file__), "..", "nvidia", "*", "lib",
                                        "libcudart.so*")):
            return ctypes.CDLL(c)
    return None


@pytest.mark.parametrize("fuse", ["1", "0"])
def test_forward_launches_and_graph_capture(moe, fuse, monkeypatch):
    """Capture one moe_forward in a CUDA graph: the runtime counts exactly the kernel nodes that
    moe_forward_launch_count() states (4 with route+permute fused, 5 without), and replaying the
    graph reproduces the eager result bit for bit."""
    monkeypatch.setenv("MOE_FUSE_ROUTE_PERMUTE", fuse)
    w = WORKLOADS["tiny"]
    logits, x, wgu, wd = case_inputs(w)
    dev = torch.device(DEV)
    args = (x.to(dev), logits.to(dev), wgu.to(dev), wd.to(dev), w.k)
    ws = torch.empty(moe.workspace_size(w.T, w.d, w.f, w.E, w.k), dtype=torch.uint8, device=dev)
    eager = moe.forward(*args, workspace=ws).clone()
    out = torch.zeros_like(eager)
    torch.cuda.synchronize()
    try:
        g = torch.cuda.CUDAGraph(keep_graph=True)
    except TypeError:  # a torch without keep_graph: replay still checked, nodes not counted
        g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.forward(*args, out=out, workspace=ws)
    raw = None
    try:
        raw = g.raw_cuda_graph()
    except (AttributeError, RuntimeError):
        pass
    kinds = _graph_node_types(raw) if raw else None
    if raw is not None and hasattr(g, "instantiate"):
        g.instantiate()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    if kinds is None:
        pytest.skip("no libcudart / raw_cuda_graph to count graph nodes")
    # cudaGraphNodeTypeKernel == 0
    assert kinds.count(0) == moe.forward_launch_count(w.T, w.E, w.k) == (4 if fuse == "1" else 5), kinds


def _graph_node_types(raw):
    import ctypes
    rt = _cudart()
    if rt is None:
        return None
    g = ctypes.c_void_p(raw)
    n = ctypes.c_size_t(0)
    assert rt.cudaGraphGetNodes(g, None, ctypes.byref(n)) == 0
    nodes = (ctypes.c_void_p * n.value)()
    assert rt.cudaGraphGetNodes(g, nodes, ctypes.byref(n)) == 0
    kinds = []
    for i in range(n.value):
        t = ctypes.c_int(-1)
        assert rt.cudaGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(t)) == 0
        kinds.append(t.value)
    return kinds
