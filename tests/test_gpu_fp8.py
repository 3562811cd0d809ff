"""GPU parity of the FP8 (E4M3) variant against the CPU oracle, through the C ABI.

  * quantisers (weights per output column, rows per row, with a src gather): codes and scales
    bit for bit — both sides take absmax, 448 / absmax and the round-to-nearest-even saturating
    E4M3 conversion in fp32 on the same bf16 inputs;
  * FP8 grouped GEMMs on random codes and scales: gate+up (bf16 h) at the gate+up stage's
    tolerance, down (fp32 y) at the down stage's (the products of E4M3 values are exact in fp32,
    so only the summation order differs);
  * the whole FP8 layer (moe_forward_fp8): routing, permutation and the x codes bit for bit, the
    output at the layer tolerance.  h is requantised from bf16 values that may differ from the
    oracle's by one bf16 rounding, so h's codes are not compared bit for bit; the output is.
"""
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
from gpu_cases import assert_close, assert_layer_close, case_inputs, random_bf16, to_np_bits  # noqa: E402

from mixture_experts_grouped_fp32_gb300.workloads import (WORKLOADS, Workload, draw_e4m3_codes,  # noqa: E402
                                                          draw_scales, make_inputs)

pytestmark = pytest.mark.gpu
DEV = "cuda"
KNOBS = ("MOE_GEMM_SWAP_MAX", "MOE_DOWN_KSPLIT", "MOE_FUSE_ROUTE_PERMUTE", "MOE_GEMM_2SM", "MOE_GEMM_2SM_DOWN",
         "MOE_GEMM_PAIR_LAYOUT", "MOE_GEMM_PAIR_SPLIT", "MOE_GEMM_PAIR_SWAP_MAX")
# Grouped-GEMM kernel configurations: the 1-SM kernel (swap thresholds 64, 0, 128) and the SM-pair
# kernel (normal-only; swapping with either shared-memory layout, round-robin or split schedule).
GEMM_MODES = {
    "1sm": {"MOE_GEMM_2SM": "0"},
    "1sm_noswap": {"MOE_GEMM_2SM": "0", "MOE_GEMM_SWAP_MAX": "0"},
    "1sm_swap128": {"MOE_GEMM_2SM": "0", "MOE_GEMM_SWAP_MAX": "128"},
    "pair1": {"MOE_GEMM_2SM": "1"},
    "pair2": {"MOE_GEMM_2SM": "2"},
    "pair2_A": {"MOE_GEMM_2SM": "2", "MOE_GEMM_PAIR_LAYOUT": "A", "MOE_GEMM_PAIR_SPLIT": "0"},
    "pair2_B": {"MOE_GEMM_2SM": "2", "MOE_GEMM_PAIR_LAYOUT": "B", "MOE_GEMM_PAIR_SPLIT": "0"},
    "pair2_split": {"MOE_GEMM_2SM": "2", "MOE_GEMM_PAIR_SPLIT": "30"},
    "pair2_swap64": {"MOE_GEMM_2SM": "2", "MOE_GEMM_PAIR_SWAP_MAX": "64"},
}


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_grouped_fp32_gb300 import moe as m
    m.load()
    return m


@pytest.fixture(autouse=True)
def _clean_env(monkeypatch):
    for k in KNOBS:
        monkeypatch.delenv(k, raising=False)


def w8(a: np.ndarray) -> torch.Tensor:
    """[E, N, K] codes -> the library's blocked weight layout, on the GPU."""
    from mixture_experts_grouped_fp32_gb300.moe import fp8_block
    return u8(fp8_block(a))


def unblock(t: torch.Tensor) -> np.ndarray:
    from mixture_experts_grouped_fp32_gb300.moe import fp8_unblock
    return fp8_unblock(t.cpu().numpy())


def u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.uint8)).to(DEV)


def f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(DEV)


def special_rows(bits: np.ndarray) -> np.ndarray:
    """Rows with the quantiser's edge cases: all zero (scale 1), a -0.0, one dominant value (most
    codes subnormal or zero), tiny magnitudes, values at bf16's largest finite."""
    b = bits.copy()
    b[0] = 0
    b[1, :] = 0
    b[1, 3] = 0x8000                      # -0.0 in an otherwise zero row
    b[2, 5] = 0x4780                      # 65536 among N(0,1) values
    b[3] = (b[3] & 0x807F) | 0x0500       # magnitudes in [2^-117, 2^-116) (448 / absmax still finite)
    b[4, 7] = 0x7F7F                      # bf16 max
    return b


@pytest.mark.parametrize("E,K,N", [(3, 256, 192), (2, 128, 64), (5, 384, 320)])
def test_quantize_weights_fp8_bit_exact(moe, oracle, E, K, N):
    W = random_bf16((E, K, N), seed=E * 7 + K)
    bits = to_np_bits(W)
    bits[0, :, 0] = 0                     # an all-zero output column
    bits[0, 5, 1] = 0x7F7F                # a column with bf16's largest value
    bits[E - 1, :, N - 1] = (bits[E - 1, :, N - 1] & 0x807F) | 0x0500  # a column of tiny values
    Wt = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(DEV)
    q, sc = moe.quantize_weights_fp8(Wt)
    torch.cuda.synchronize()
    rq, rsc = oracle.quantize_weights_fp8(bits)
    assert np.array_equal(unblock(q), rq)
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), rsc.view(np.uint32))


@pytest.mark.parametrize("R,C,src_rows", [(37, 256, None), (300, 4096, 150), (5, 8, 5), (1, 14336, 3),
                                          (6, 16384, None), (4, 20480, 9)])
def test_quantize_rows_fp8_bit_exact(moe, oracle, R, C, src_rows):
    n_src = src_rows or R
    bits = to_np_bits(random_bf16((n_src, C), seed=R + C))
    if n_src >= 5:
        bits = special_rows(bits)
    a = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(DEV)
    src = None
    if src_rows is not None:
        src = np.random.default_rng(R).integers(0, src_rows, R).astype(np.int32)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    q, sc = moe.quantize_rows_fp8(a, None if src is None else torch.from_numpy(src).to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rq, rsc = oracle.quantize_rows_fp8(bits if src is None else bits[src])
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), rsc.view(np.uint32))


def test_quantize_rows_fp8_bad_src(moe, oracle):
    bits = to_np_bits(random_bf16((10, 64), seed=3))
    a = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(DEV)
    src = np.array([0, 9, -1, 10, 4], np.int32)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    q, sc = moe.quantize_rows_fp8(a, torch.from_numpy(src).to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & moe.STATUS_BAD_SRC
    q, sc = q.cpu().numpy(), sc.cpu().numpy()
    assert not q[2].any() and not q[3].any() and sc[2] == 1.0 and sc[3] == 1.0
    rq, rsc = oracle.quantize_rows_fp8(bits[src[[0, 1, 4]]])
    assert np.array_equal(q[[0, 1, 4]], rq) and np.array_equal(sc[[0, 1, 4]], rsc)


@pytest.mark.parametrize("nt", ["", "256", "1024"])
@pytest.mark.parametrize("T,d,E,k", [(1, 256, 8, 2), (300, 256, 8, 2), (2000, 4096, 64, 6), (77, 7168, 16, 4),
                                     (12000, 128, 8, 2)])
def test_permute_fp8_parity(moe, oracle, T, d, E, k, nt, monkeypatch):
    """Step 2 of the FP8 layer: the permutation bit for bit, and each permuted row's codes and
    scale equal to the oracle's quantisation of x[src[r]], at every block size (MOE_PERM_THREADS;
    "" = the default rule)."""
    if nt:
        monkeypatch.setenv("MOE_PERM_THREADS", nt)
    g = torch.Generator("cpu").manual_seed(T + d)
    logits = torch.randn(T, E, generator=g)
    idx, _ = oracle.route(logits.numpy(), k)
    bits = to_np_bits(random_bf16((T, d), seed=T * 3 + E))
    if T >= 5:
        bits = special_rows(bits)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    counts, offsets, src, dest, x8, sx = moe.permute_fp8(torch.from_numpy(idx).to(DEV), x, E, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rc, ro, rs, rd = oracle.permute(idx, E)
    assert np.array_equal(counts.cpu().numpy(), rc) and np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(src.cpu().numpy(), rs) and np.array_equal(dest.cpu().numpy(), rd)
    rq, rsc = oracle.quantize_rows_fp8(bits[rs])
    assert np.array_equal(x8.cpu().numpy(), rq)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), rsc.view(np.uint32))


def segments(counts):
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return offsets


GEMM_CASES = [  # (counts per expert, d, f); rows beyond offsets[E] exist in the buffers (M > offsets[E])
    ([5, 0, 64, 1, 17], 256, 512),          # all swapped (<= 64 rows), an empty expert
    ([130, 3, 257, 64, 65], 256, 384),      # normal tiles with ragged tails, swap both sides of 64
    ([700], 512, 256),                      # one expert, six M-tiles
    ([33, 128, 1, 0, 200, 96, 7, 15], 384, 640),
]


@pytest.mark.parametrize("mode", sorted(GEMM_MODES))
@pytest.mark.parametrize("ci", range(len(GEMM_CASES)))
def test_gemm_fp8_parity(moe, oracle, monkeypatch, ci, mode):
    for k, v in GEMM_MODES[mode].items():
        monkeypatch.setenv(k, v)
    counts, d, f = GEMM_CASES[ci]
    E = len(counts)
    offsets = segments(counts)
    M = int(offsets[-1]) + 3
    seed = 100 * ci + sorted(GEMM_MODES).index(mode)
    x8, sx = draw_e4m3_codes((M, d), seed), draw_scales(M, seed + 1)
    wgu8, sgu = draw_e4m3_codes((E, 2 * f, d), seed + 2), draw_scales((E, 2 * f), seed + 3)
    h8, sh = draw_e4m3_codes((M, f), seed + 4), draw_scales(M, seed + 5)
    wd8, sd = draw_e4m3_codes((E, d, f), seed + 6), draw_scales((E, d), seed + 7)
    off_t = torch.from_numpy(offsets).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    h = moe.grouped_gemm_gateup_swiglu_fp8(u8(x8), f32(sx), w8(wgu8), f32(sgu), off_t, status=status)
    y = moe.grouped_gemm_down_fp8(u8(h8), f32(sh), w8(wd8), f32(sd), off_t, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    n = int(offsets[-1])
    ref_h = oracle.gateup_swiglu_fp8(x8, sx, offsets, wgu8, sgu)
    got_h = h.float().cpu().numpy()[:n]
    ref_hf = (ref_h[:n].astype(np.uint32) << 16).view(np.float32)  # bf16 bits -> fp32, exact
    assert_close(got_h, ref_hf, 2.0 ** -7, 2e-3, "fp8 gate+up h")
    ref_y = oracle.down_fp8(h8, sh, offsets, wd8, sd)
    assert_close(y.cpu().numpy()[:n], ref_y[:n], 1e-3, 1e-4, "fp8 down y")


@pytest.mark.parametrize("mode", ["1sm", "pair1", "pair2"])
@pytest.mark.parametrize("ksplit", [2, 3])
def test_gemm_down_fp8_ksplit(moe, oracle, monkeypatch, ksplit, mode):
    for k, v in GEMM_MODES[mode].items():
        monkeypatch.setenv(k, v)
    counts, d, f = [40, 300, 0, 77], 256, 640  # f = 5 blocks of 128: ksplit 3 leaves slices of 2, 2, 1
    E = len(counts)
    offsets = segments(counts)
    M = int(offsets[-1])
    h8, sh = draw_e4m3_codes((M, f), 11), draw_scales(M, 12)
    wd8, sd = draw_e4m3_codes((E, d, f), 13), draw_scales((E, d), 14)
    y = moe.grouped_gemm_down_fp8(u8(h8), f32(sh), w8(wd8), f32(sd), torch.from_numpy(offsets).to(DEV),
                                  ksplit=ksplit)
    torch.cuda.synchronize()
    ref_y = oracle.down_fp8(h8, sh, offsets, wd8, sd)
    assert_close(y.sum(0).cpu().numpy(), ref_y, 1e-3, 1e-4, f"fp8 down y, ksplit {ksplit}")


LAYER_CASES = [
    Workload("fp8_tiny", 64, 256, 512, 8, 2),
    Workload("fp8_many_rows", 700, 256, 384, 4, 2),
    Workload("fp8_skewed", 300, 384, 256, 16, 4, ("zipf", 1.2)),
    Workload("fp8_hot_expert", 200, 256, 512, 8, 2, ("hot0", 2.2)),
    Workload("fp8_one_token", 1, 512, 256, 8, 2),
    Workload("fp8_dense_e1_k1", 70, 128, 256, 1, 1),
    Workload("fp8_k_eq_e", 37, 256, 384, 4, 4),
    Workload("fp8_many_experts", 96, 128, 128, 256, 8, ("zipf", 1.2)),
    Workload("fp8_deepseek_like", 48, 1024, 256, 64, 8, ("zipf", 1.2)),
]


def quantized_weights(moe, oracle, wgu, wd):
    """GPU-side codes from the library's quantiser, oracle-side codes from the oracle's (checked
    equal, so that both sides start from the same weights)."""
    wgu8, sgu = moe.quantize_weights_fp8(wgu.to(DEV))
    wd8, sd = moe.quantize_weights_fp8(wd.to(DEV))
    r = oracle.quantize_weights_fp8(to_np_bits(wgu)) + oracle.quantize_weights_fp8(to_np_bits(wd))
    torch.cuda.synchronize()
    assert np.array_equal(unblock(wgu8), r[0]) and np.array_equal(sgu.cpu().numpy(), r[1])
    assert np.array_equal(unblock(wd8), r[2]) and np.array_equal(sd.cpu().numpy(), r[3])
    return (wgu8, sgu, wd8, sd), r


@pytest.mark.parametrize("mode", ["default", "noswap", "ksplit3", "nofuse", "pair1", "pair2"])
@pytest.mark.parametrize("w", LAYER_CASES, ids=lambda w: w.name)
def test_forward_fp8_matches_oracle(moe, oracle, monkeypatch, w, mode):
    if mode in GEMM_MODES:
        for k, v in GEMM_MODES[mode].items():
            monkeypatch.setenv(k, v)
    elif mode == "noswap":
        monkeypatch.setenv("MOE_GEMM_SWAP_MAX", "0")
    elif mode == "ksplit3":
        monkeypatch.setenv("MOE_DOWN_KSPLIT", "3")
    elif mode == "nofuse":
        monkeypatch.setenv("MOE_FUSE_ROUTE_PERMUTE", "0")
    logits, x, wgu, wd = case_inputs(w, seed=1)
    gpu_w, ref_w = quantized_weights(moe, oracle, wgu, wd)
    dev = torch.device(DEV)
    ws = torch.empty(moe.workspace_size_fp8(w.T, w.d, w.f, w.E, w.k), dtype=torch.uint8, device=dev)
    ws.fill_(0xFF)
    out = moe.forward_fp8(x.to(dev), logits.to(dev), *gpu_w, w.k, workspace=ws)
    torch.cuda.synchronize()
    assert moe.get_device_error(ws) == 0
    v = moe.workspace_views_fp8(ws, w.T, w.d, w.f, w.E, w.k)
    ln, xb = logits.numpy(), to_np_bits(x)
    idx, wt = oracle.route(ln, w.k)
    counts, offsets, src, dest = oracle.permute(idx, w.E)
    assert np.array_equal(v["idx"].cpu().numpy(), idx)
    assert np.array_equal(v["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(v["src"].cpu().numpy(), src)
    assert np.array_equal(v["dest"].cpu().numpy(), dest)
    rx8, rsx = oracle.quantize_rows_fp8(xb[src])
    assert np.array_equal(v["x8"].cpu().numpy(), rx8)
    assert np.array_equal(v["sx"].cpu().numpy(), rsx)
    ref = oracle.forward_fp8(xb, ln, *ref_w, w.k)
    assert_layer_close(out.float().cpu().numpy(), ref, f"{w.name} fp8 [{mode}]")


def test_forward_fp8_launch_count(moe):
    assert moe.forward_fp8_launch_count(64, 8, 2) == 5      # route+permute fused
    assert moe.forward_fp8_launch_count(2048, 256, 8) == 6
    assert moe.forward_fp8_launch_count(0, 8, 2) == 0


@pytest.mark.slow
@pytest.mark.parametrize("path", ["policy", "other"])
@pytest.mark.parametrize("name", ["mixtral_t32", "mixtral_t512", "mixtral_t4096", "deepseek_t2048"])
def test_forward_fp8_full_size(moe, oracle, monkeypatch, name, path):
    """The FP8 layer at full size in the configuration bench.py times (`policy`), and with another
    grouped-GEMM kernel forced (`other`: single SMs -> swapping SM pairs -> normal-only SM pairs ->
    single SMs): the weight codes and scales bit for bit against the oracle's quantiser, routing,
    permutation and x codes bit for bit, the output on sampled tokens that the oracle computes one
    by one."""
    w = WORKLOADS[name]
    if path == "other":
        rot = {0: "2", 2: "1", 1: "0"}
        monkeypatch.setenv("MOE_GEMM_2SM", rot[moe.gemm_pair_mode_fp8(w.T, w.d, w.f, w.E, w.k, 0)])
        monkeypatch.setenv("MOE_GEMM_2SM_DOWN", rot[moe.gemm_pair_mode_fp8(w.T, w.d, w.f, w.E, w.k, 1)])
    dev = torch.device(DEV)
    logits, x, wgu, wd = make_inputs(w, seed=0, weight_device="cuda")
    wgu8, sgu = moe.quantize_weights_fp8(wgu)
    wd8, sd = moe.quantize_weights_fp8(wd)
    torch.cuda.synchronize()
    wgu_bits, wd_bits = to_np_bits(wgu), to_np_bits(wd)
    del wgu, wd
    torch.cuda.empty_cache()
    ws = torch.empty(moe.workspace_size_fp8(w.T, w.d, w.f, w.E, w.k), dtype=torch.uint8, device=dev)
    out = moe.forward_fp8(x.to(dev), logits.to(dev), wgu8, sgu, wd8, sd, w.k, workspace=ws)
    torch.cuda.synchronize()
    assert moe.get_device_error(ws) == 0
    v = moe.workspace_views_fp8(ws, w.T, w.d, w.f, w.E, w.k)
    r_wgu8, r_sgu = oracle.quantize_weights_fp8(wgu_bits)
    assert np.array_equal(unblock(wgu8), r_wgu8) and np.array_equal(sgu.cpu().numpy(), r_sgu)
    del wgu_bits
    r_wd8, r_sd = oracle.quantize_weights_fp8(wd_bits)
    assert np.array_equal(unblock(wd8), r_wd8) and np.array_equal(sd.cpu().numpy(), r_sd)
    del wd_bits
    ln, xb = logits.numpy(), to_np_bits(x)
    idx, wt = oracle.route(ln, w.k)
    counts, offsets, src, dest = oracle.permute(idx, w.E)
    assert np.array_equal(v["idx"].cpu().numpy(), idx)
    assert np.array_equal(v["src"].cpu().numpy(), src)
    assert np.array_equal(v["dest"].cpu().numpy(), dest)
    rx8, rsx = oracle.quantize_rows_fp8(xb[src])
    assert np.array_equal(v["x8"].cpu().numpy(), rx8) and np.array_equal(v["sx"].cpu().numpy(), rsx)
    rng = np.random.default_rng(3)
    hot = int(np.argmax(counts))
    hot_tokens = src[offsets[hot]:offsets[hot + 1]]
    sample = np.unique(np.concatenate([[0, w.T - 1], rng.integers(0, w.T, 5),
                                       rng.choice(hot_tokens, min(3, hot_tokens.size), replace=False)]))
    ref = oracle.forward_fp8_tokens_routed(xb, idx[sample], wt[sample], r_wgu8, r_sgu, r_wd8, r_sd,
                                           sample.astype(np.int32))
    got = out[torch.from_numpy(sample).to(dev)].float().cpu().numpy()
    assert_layer_close(got, ref, f"{name} fp8 sampled tokens {sample.tolist()}")


@pytest.mark.parametrize("variant", ["fp8", "fp8b"])
def test_forward_fp8_graph_capture(moe, variant):
    """Capture one FP8 layer in a CUDA graph: the kernel nodes equal the stated launch count and
    replaying reproduces the eager result bit for bit."""
    from test_gpu_parity import _graph_node_types
    w = WORKLOADS["tiny"]
    logits, x, wgu, wd = case_inputs(w)
    dev = torch.device(DEV)
    quant = moe.quantize_weights_fp8b if variant == "fp8b" else moe.quantize_weights_fp8
    fwd = moe.forward_fp8b if variant == "fp8b" else moe.forward_fp8
    wsize = moe.workspace_size_fp8b if variant == "fp8b" else moe.workspace_size_fp8
    count = moe.forward_fp8b_launch_count if variant == "fp8b" else moe.forward_fp8_launch_count
    w8 = quant(wgu.to(dev)) + quant(wd.to(dev))
    args = (x.to(dev), logits.to(dev), *w8, w.k)
    ws = torch.empty(wsize(w.T, w.d, w.f, w.E, w.k), dtype=torch.uint8, device=dev)
    eager = fwd(*args, workspace=ws).clone()
    out = torch.zeros_like(eager)
    torch.cuda.synchronize()
    try:
        g = torch.cuda.CUDAGraph(keep_graph=True)
    except TypeError:
        g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fwd(*args, out=out, workspace=ws)
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
    assert kinds.count(0) == count(w.T, w.E, w.k), kinds


@pytest.mark.parametrize("variant", ["fp8", "fp8b"])
def test_forward_fp8_host_batches_matches_forward(moe, variant):
    """FP8 layers over host batches with overlapped copies give each batch's device-call output."""
    w = Workload("fp8_host_batches", 97, 256, 512, 8, 2)
    dev = torch.device(DEV)
    _, _, wgu, wd = case_inputs(w, seed=31)
    quant = moe.quantize_weights_fp8b if variant == "fp8b" else moe.quantize_weights_fp8
    fwd = moe.forward_fp8b if variant == "fp8b" else moe.forward_fp8
    batches = moe.forward_fp8b_host_batches if variant == "fp8b" else moe.forward_fp8_host_batches
    wsize = moe.workspace_size_fp8b if variant == "fp8b" else moe.workspace_size_fp8
    w8 = quant(wgu.to(dev)) + quant(wd.to(dev))
    xs, ls, refs = [], [], []
    for i in range(3):
        logits, x, _, _ = case_inputs(w, seed=40 + i)
        xs.append(x.pin_memory())
        ls.append(logits.pin_memory())
        refs.append(fwd(x.to(dev), logits.to(dev), *w8, w.k).cpu())
    outs = [torch.full((w.T, w.d), -1.0, dtype=torch.bfloat16).pin_memory() for _ in range(3)]
    ws = torch.empty(wsize(w.T, w.d, w.f, w.E, w.k) + 2 * moe.host_staging_size(w.T, w.d, w.E),
                     dtype=torch.uint8, device=dev)
    batches(xs, ls, *w8, w.k, outs, ws)
    torch.cuda.current_stream().synchronize()
    assert moe.get_device_error(ws) == 0
    for i in range(3):
        assert torch.equal(outs[i].view(torch.int16), refs[i].view(torch.int16)), f"{variant} batch {i}"


def test_fp8_status_flags(moe):
    """Bad offsets reach the FP8 and blockwise FP8 GEMMs' status bit; a bad expert id reaches the
    FP8 permute's; nothing is read out of bounds."""
    E, d, f = 4, 128, 128
    M = 16
    x8 = torch.zeros(M, d, dtype=torch.uint8, device=DEV)
    sx = torch.ones(M, dtype=torch.float32, device=DEV)
    sxb = torch.ones(M, d // 128, dtype=torch.float32, device=DEV)
    w8 = torch.zeros(E, 2 * f // 64, d // 128, 64, 128, dtype=torch.uint8, device=DEV)
    sw = torch.ones(E, 2 * f, dtype=torch.float32, device=DEV)
    swb = torch.ones(E, 2 * f // 128, d // 128, dtype=torch.float32, device=DEV)
    h = torch.zeros(M, f, dtype=torch.bfloat16, device=DEV)
    for bad in ([0, 5, 3, 8, 16], [0, 4, 8, 12, 17]):
        offs = torch.tensor(bad, dtype=torch.int32, device=DEV)
        for call in (lambda st: moe.grouped_gemm_gateup_swiglu_fp8(x8, sx, w8, sw, offs, h=h, status=st),
                     lambda st: moe.grouped_gemm_gateup_swiglu_fp8b(x8, sxb, w8, swb, offs, h=h, status=st)):
            status = torch.zeros(1, dtype=torch.int32, device=DEV)
            call(status)
            torch.cuda.synchronize()
            assert int(status.item()) & moe.STATUS_BAD_OFFSETS
    idx = torch.tensor([[0, 1], [2, 9], [3, 3]], dtype=torch.int32, device=DEV)
    x = torch.zeros(3, 128, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    moe.permute_fp8(idx, x, 4, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & moe.STATUS_BAD_EXPERT_ID
