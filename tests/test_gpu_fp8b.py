"""GPU parity of the blockwise FP8 variant (1 x 128 activation blocks, 128 x 128 weight blocks,
power-of-two scales) against the CPU oracle, through the C ABI.

  * quantisers: codes and block scales bit for bit (power-of-two scaling is exact on both sides);
  * GEMMs on random codes and random power-of-two block scales: gate+up (bf16 h) at the gate+up
    stage's tolerance, down (fp32 y) at the down stage's — each block's partial sum is exact
    products summed in fp32, scaled exactly, so only summation order differs;
  * the layer (moe_forward_fp8b): routing, permutation and x codes bit for bit, the output at
    the layer tolerance.
"""
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
from gpu_cases import assert_close, assert_layer_close, case_inputs, random_bf16, to_np_bits  # noqa: E402

from mixture_experts_grouped_fp32_gb300.workloads import (WORKLOADS, Workload, draw_e4m3_codes,  # noqa: E402
                                                          draw_pow2_scales, make_inputs)

pytestmark = pytest.mark.gpu
DEV = "cuda"
KNOBS = ("MOE_GEMM_SWAP_MAX", "MOE_DOWN_KSPLIT", "MOE_FUSE_ROUTE_PERMUTE")


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_grouped_fp32_gb300 import moe as m
    m.load()
    return m


@pytest.fixture(autouse=True)
def _clean_env(monkeypatch):
    for k in KNOBS:
        monkeypatch.delenv(k, raising=False)


def u8(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.uint8)).to(DEV)


def f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(DEV)


def w8(a):
    from mixture_experts_grouped_fp32_gb300.moe import fp8_block
    return u8(fp8_block(a))


def unblock(t):
    from mixture_experts_grouped_fp32_gb300.moe import fp8_unblock
    return fp8_unblock(t.cpu().numpy())


def bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


def spread_blocks(bits, seed, axes):
    """Give every 128-wide block along `axes` its own power-of-two magnitude (block scales differ)."""
    rng = np.random.default_rng(seed)
    v = (bits.astype(np.uint32) << 16).view(np.float32)
    for ax in axes:
        fac = (2.0 ** rng.integers(-8, 8, v.shape[ax] // 128)).repeat(128).astype(np.float32)
        shape = [1] * v.ndim
        shape[ax] = -1
        v = v * fac.reshape(shape)
    u = v.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


@pytest.mark.parametrize("E,K,N", [(2, 256, 384), (3, 128, 128), (1, 512, 256)])
def test_quantize_weights_fp8b_bit_exact(moe, oracle, E, K, N):
    bits = spread_blocks(to_np_bits(random_bf16((E, K, N), seed=K + N)), 3, (1, 2))
    bits[0, :128, :128] = 0  # an all-zero block: scale 1
    q, sc = moe.quantize_weights_fp8b(bf16_dev(bits))
    torch.cuda.synchronize()
    rq, rsc = oracle.quantize_weights_fp8b(bits)
    assert np.array_equal(unblock(q), rq)
    assert np.array_equal(sc.cpu().numpy(), rsc)


@pytest.mark.parametrize("R,C,src_rows", [(37, 256, None), (300, 4096, 150), (5, 128, 5), (2, 14336, 3)])
def test_quantize_rows_fp8b_bit_exact(moe, oracle, R, C, src_rows):
    n_src = src_rows or R
    bits = spread_blocks(to_np_bits(random_bf16((n_src, C), seed=R + C)), R, (1,))
    bits[0, :128] = 0
    if n_src > 2:
        bits[1, 5] = 0x7F7F     # bf16's largest value in a block
        bits[2, 128:] = bits[2, 128:] & 0x807F | 0x0080  # tiny magnitudes
    src = None if src_rows is None else np.random.default_rng(R).integers(0, src_rows, R).astype(np.int32)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    q, sc = moe.quantize_rows_fp8b(bf16_dev(bits), None if src is None else torch.from_numpy(src).to(DEV),
                                   status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rq, rsc = oracle.quantize_rows_fp8b(bits if src is None else bits[src])
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(sc.cpu().numpy(), rsc)


def segments(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


GEMM_CASES = [
    ([5, 0, 64, 1, 17], 256, 512),
    ([130, 3, 257, 64, 65], 256, 384),
    ([700], 512, 256),
    ([33, 128, 1, 0, 200, 96, 7, 15], 384, 640),
    ([120, 9], 128, 128),          # one K block
]


@pytest.mark.parametrize("swap_max", ["64", "0", "128"])
@pytest.mark.parametrize("ci", range(len(GEMM_CASES)))
def test_gemm_fp8b_parity(moe, oracle, monkeypatch, ci, swap_max):
    monkeypatch.setenv("MOE_GEMM_SWAP_MAX", swap_max)
    counts, d, f = GEMM_CASES[ci]
    E = len(counts)
    offsets = segments(counts)
    M = int(offsets[-1]) + 3
    seed = 1000 + 10 * ci + int(swap_max)
    x8, sx = draw_e4m3_codes((M, d), seed), draw_pow2_scales((M, d // 128), seed + 1)
    wgu8, sgu = draw_e4m3_codes((E, 2 * f, d), seed + 2), draw_pow2_scales((E, 2 * f // 128, d // 128), seed + 3)
    h8, sh = draw_e4m3_codes((M, f), seed + 4), draw_pow2_scales((M, f // 128), seed + 5)
    wd8, sd = draw_e4m3_codes((E, d, f), seed + 6), draw_pow2_scales((E, d // 128, f // 128), seed + 7)
    off_t = torch.from_numpy(offsets).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    h = moe.grouped_gemm_gateup_swiglu_fp8b(u8(x8), f32(sx), w8(wgu8), f32(sgu), off_t, status=status)
    y = moe.grouped_gemm_down_fp8b(u8(h8), f32(sh), w8(wd8), f32(sd), off_t, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    n = int(offsets[-1])
    ref_h = oracle.gateup_swiglu_fp8b(x8, sx, offsets, wgu8, sgu)
    ref_hf = (ref_h[:n].astype(np.uint32) << 16).view(np.float32)
    assert_close(h.float().cpu().numpy()[:n], ref_hf, 2.0 ** -7, 2e-3, "blockwise fp8 gate+up h")
    ref_y = oracle.down_fp8b(h8, sh, offsets, wd8, sd)
    assert_close(y.cpu().numpy()[:n], ref_y[:n], 1e-3, 1e-4, "blockwise fp8 down y")


@pytest.mark.parametrize("swap_max", ["64", "0"])
@pytest.mark.parametrize("ci", range(len(GEMM_CASES)))
def test_gemm_gateup_fp8b_quantised_h(moe, oracle, monkeypatch, ci, swap_max):
    """The gate+up GEMM quantising h in its epilogue gives, bit for bit, the codes and block scales
    that quantising its bf16 output gives (normal and swapped items; rows past the experts' untouched)."""
    monkeypatch.setenv("MOE_GEMM_SWAP_MAX", swap_max)
    counts, d, f = GEMM_CASES[ci]
    E = len(counts)
    offsets = segments(counts)
    n = int(offsets[-1])
    M = n + 3
    seed = 2000 + 10 * ci + int(swap_max)
    x8, sx = draw_e4m3_codes((M, d), seed), draw_pow2_scales((M, d // 128), seed + 1)
    wgu8, sgu = draw_e4m3_codes((E, 2 * f, d), seed + 2), draw_pow2_scales((E, 2 * f // 128, d // 128), seed + 3)
    off_t = torch.from_numpy(offsets).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    h = moe.grouped_gemm_gateup_swiglu_fp8b(u8(x8), f32(sx), w8(wgu8), f32(sgu), off_t, status=status)
    h8 = torch.full((M, f), 0x7E, dtype=torch.uint8, device=DEV)
    sh = torch.full((M, f // 128), -1.0, dtype=torch.float32, device=DEV)
    moe.grouped_gemm_gateup_swiglu_fp8b_q(u8(x8), f32(sx), w8(wgu8), f32(sgu), off_t, h8=h8, sh=sh, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref8, refs = oracle.quantize_rows_fp8b(to_np_bits(h[:n].cpu()))
    assert np.array_equal(h8[:n].cpu().numpy(), ref8)
    assert np.array_equal(sh[:n].cpu().numpy(), refs)
    assert bool((h8[n:] == 0x7E).all()) and bool((sh[n:] == -1.0).all())


@pytest.mark.parametrize("ksplit", [2, 3])
def test_gemm_down_fp8b_ksplit(moe, oracle, ksplit):
    counts, d, f = [40, 300, 0, 77], 256, 640
    E = len(counts)
    offsets = segments(counts)
    M = int(offsets[-1])
    h8, sh = draw_e4m3_codes((M, f), 21), draw_pow2_scales((M, f // 128), 22)
    wd8, sd = draw_e4m3_codes((E, d, f), 23), draw_pow2_scales((E, d // 128, f // 128), 24)
    y = moe.grouped_gemm_down_fp8b(u8(h8), f32(sh), w8(wd8), f32(sd), torch.from_numpy(offsets).to(DEV),
                                   ksplit=ksplit)
    torch.cuda.synchronize()
    ref_y = oracle.down_fp8b(h8, sh, offsets, wd8, sd)
    assert_close(y.sum(0).cpu().numpy(), ref_y, 1e-3, 1e-4, f"blockwise fp8 down y, ksplit {ksplit}")


LAYER_CASES = [
    Workload("fp8b_tiny", 64, 256, 512, 8, 2),
    Workload("fp8b_many_rows", 700, 256, 384, 4, 2),
    Workload("fp8b_skewed", 300, 384, 256, 16, 4, ("zipf", 1.2)),
    Workload("fp8b_one_token", 1, 512, 256, 8, 2),
    Workload("fp8b_dense_e1_k1", 70, 128, 256, 1, 1),
    Workload("fp8b_k_eq_e", 37, 256, 384, 4, 4),
    Workload("fp8b_many_experts", 96, 128, 128, 256, 8, ("zipf", 1.2)),
    Workload("fp8b_deepseek_like", 48, 1024, 256, 64, 8, ("zipf", 1.2)),
]


def quantized_weights(moe, oracle, wgu, wd):
    wgu8, sgu = moe.quantize_weights_fp8b(wgu.to(DEV))
    wd8, sd = moe.quantize_weights_fp8b(wd.to(DEV))
    r = oracle.quantize_weights_fp8b(to_np_bits(wgu)) + oracle.quantize_weights_fp8b(to_np_bits(wd))
    torch.cuda.synchronize()
    assert np.array_equal(unblock(wgu8), r[0]) and np.array_equal(sgu.cpu().numpy(), r[1])
    assert np.array_equal(unblock(wd8), r[2]) and np.array_equal(sd.cpu().numpy(), r[3])
    return (wgu8, sgu, wd8, sd), r


@pytest.mark.parametrize("mode", ["default", "noswap", "ksplit3", "nofuse", "fuse_h", "fuse_h_noswap", "unfused_h"])
@pytest.mark.parametrize("w", LAYER_CASES, ids=lambda w: w.name)
def test_forward_fp8b_matches_oracle(moe, oracle, monkeypatch, w, mode):
    if mode.startswith("fuse_h"):  # h quantised in the gate+up GEMM's epilogue whatever the shape
        monkeypatch.setenv("MOE_FP8B_FUSE_H", "1")
        if mode == "fuse_h_noswap":
            monkeypatch.setenv("MOE_GEMM_SWAP_MAX", "0")
    elif mode == "unfused_h":
        monkeypatch.setenv("MOE_FP8B_FUSE_H", "0")
    elif mode == "noswap":
        monkeypatch.setenv("MOE_GEMM_SWAP_MAX", "0")
    elif mode == "ksplit3":
        monkeypatch.setenv("MOE_DOWN_KSPLIT", "3")
    elif mode == "nofuse":
        monkeypatch.setenv("MOE_FUSE_ROUTE_PERMUTE", "0")
    logits, x, wgu, wd = case_inputs(w, seed=2)
    gpu_w, ref_w = quantized_weights(moe, oracle, wgu, wd)
    ws = torch.empty(moe.workspace_size_fp8b(w.T, w.d, w.f, w.E, w.k), dtype=torch.uint8, device=DEV)
    ws.fill_(0xFF)
    out = moe.forward_fp8b(x.to(DEV), logits.to(DEV), *gpu_w, w.k, workspace=ws)
    torch.cuda.synchronize()
    assert moe.get_device_error(ws) == 0
    v = moe.workspace_views_fp8b(ws, w.T, w.d, w.f, w.E, w.k)
    ln, xb = logits.numpy(), to_np_bits(x)
    idx, wt = oracle.route(ln, w.k)
    counts, offsets, src, dest = oracle.permute(idx, w.E)
    assert np.array_equal(v["idx"].cpu().numpy(), idx)
    assert np.array_equal(v["src"].cpu().numpy(), src)
    assert np.array_equal(v["dest"].cpu().numpy(), dest)
    rx8, rsx = oracle.quantize_rows_fp8b(xb[src])
    assert np.array_equal(v["x8"].cpu().numpy(), rx8) and np.array_equal(v["sx"].cpu().numpy(), rsx)
    ref = oracle.forward_fp8b(xb, ln, *ref_w, w.k)
    assert_layer_close(out.float().cpu().numpy(), ref, f"{w.name} blockwise fp8 [{mode}]")


def test_forward_fp8b_launch_count(moe):
    assert moe.forward_fp8b_launch_count(64, 8, 2) == 6       # 16 rows per expert: h quantised apart
    assert moe.forward_fp8b_launch_count(2048, 256, 8) == 7
    assert moe.forward_fp8b_launch_count(512, 8, 2) == 5      # 128 rows: in the gate+up GEMM
    assert moe.forward_fp8b_launch_count(4096, 8, 2) == 6


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mixtral_t32", "mixtral_t512", "mixtral_t4096", "deepseek_t2048"])
def test_forward_fp8b_full_size(moe, oracle, name):
    """The blockwise FP8 layer at full size in the configuration bench.py times: weight codes and
    block scales bit for bit, routing and x codes bit for bit, sampled tokens against the oracle."""
    w = WORKLOADS[name]
    dev = torch.device(DEV)
    logits, x, wgu, wd = make_inputs(w, seed=0, weight_device="cuda")
    wgu8, sgu = moe.quantize_weights_fp8b(wgu)
    wd8, sd = moe.quantize_weights_fp8b(wd)
    torch.cuda.synchronize()
    wgu_bits, wd_bits = to_np_bits(wgu), to_np_bits(wd)
    del wgu, wd
    torch.cuda.empty_cache()
    ws = torch.empty(moe.workspace_size_fp8b(w.T, w.d, w.f, w.E, w.k), dtype=torch.uint8, device=dev)
    out = moe.forward_fp8b(x.to(dev), logits.to(dev), wgu8, sgu, wd8, sd, w.k, workspace=ws)
    torch.cuda.synchronize()
    assert moe.get_device_error(ws) == 0
    v = moe.workspace_views_fp8b(ws, w.T, w.d, w.f, w.E, w.k)
    r_wgu8, r_sgu = oracle.quantize_weights_fp8b(wgu_bits)
    assert np.array_equal(unblock(wgu8), r_wgu8) and np.array_equal(sgu.cpu().numpy(), r_sgu)
    del wgu_bits
    r_wd8, r_sd = oracle.quantize_weights_fp8b(wd_bits)
    assert np.array_equal(unblock(wd8), r_wd8) and np.array_equal(sd.cpu().numpy(), r_sd)
    del wd_bits
    ln, xb = logits.numpy(), to_np_bits(x)
    idx, wt = oracle.route(ln, w.k)
    counts, offsets, src, dest = oracle.permute(idx, w.E)
    assert np.array_equal(v["idx"].cpu().numpy(), idx) and np.array_equal(v["src"].cpu().numpy(), src)
    rx8, rsx = oracle.quantize_rows_fp8b(xb[src])
    assert np.array_equal(v["x8"].cpu().numpy(), rx8) and np.array_equal(v["sx"].cpu().numpy(), rsx)
    rng = np.random.default_rng(5)
    hot = int(np.argmax(counts))
    hot_tokens = src[offsets[hot]:offsets[hot + 1]]
    sample = np.unique(np.concatenate([[0, w.T - 1], rng.integers(0, w.T, 5),
                                       rng.choice(hot_tokens, min(3, hot_tokens.size), replace=False)]))
    ref = oracle.forward_fp8b_tokens_routed(xb, idx[sample], wt[sample], r_wgu8, r_sgu, r_wd8, r_sd,
                                            sample.astype(np.int32))
    got = out[torch.from_numpy(sample).to(dev)].float().cpu().numpy()
    assert_layer_close(got, ref, f"{name} blockwise fp8 sampled tokens {sample.tolist()}")
