"""GPU parity at the full workload sizes, in the launch configuration bench.py times
(moe_forward, one call, five launches).  Routing and the permutation are compared in full and bit
for bit; the layer output is compared on sampled tokens that the oracle computes one by one
(first, last, random, tokens routed to the busiest expert, the last row of every expert's segment,
and the first rows of the segment and of its last 128- and 256-row tiles for the largest and
smallest experts)."""
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
from gpu_cases import assert_close, assert_layer_close, tile_class_tokens, to_np_bits  # noqa: E402

from mixture_experts_grouped_fp32_gb300.workloads import WORKLOADS, make_inputs  # noqa: E402

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
FULL = ["mixtral_t32", "mixtral_t512", "mixtral_t512_skew40", "mixtral_t4096", "deepseek_t2048"]


@pytest.mark.parametrize("path", ["policy", "other"])
@pytest.mark.parametrize("name", FULL)
def test_full_size_forward(oracle, name, path, monkeypatch):
    """`policy`: the GEMM path moe_forward picks for the shape; `other`: another kernel forced
    (single SMs -> swapping SM pairs -> normal-only SM pairs -> single SMs), so every kernel is
    checked at full size."""
    from mixture_experts_grouped_fp32_gb300 import moe
    w = WORKLOADS[name]
    if path == "other":
        rot = {0: "2", 2: "1", 1: "0"}
        monkeypatch.setenv("MOE_GEMM_2SM", rot[moe.gemm_pair_mode(w.T, w.d, w.f, w.E, w.k, 0)])
        monkeypatch.setenv("MOE_GEMM_2SM_DOWN", rot[moe.gemm_pair_mode(w.T, w.d, w.f, w.E, w.k, 1)])
    dev = torch.device("cuda")
    logits, x, wgu, wd = make_inputs(w, seed=0, weight_device="cuda")
    ws = torch.empty(moe.workspace_size(w.T, w.d, w.f, w.E, w.k), dtype=torch.uint8, device=dev)
    out = moe.forward(x.to(dev), logits.to(dev), wgu, wd, w.k, workspace=ws)
    torch.cuda.synchronize()
    assert moe.get_device_error(ws) == 0
    v = moe.workspace_views(ws, w.T, w.d, w.f, w.E, w.k)

    ln = logits.numpy()
    idx, wt = oracle.route(ln, w.k)
    counts, offsets, src, dest = oracle.permute(idx, w.E)
    assert np.array_equal(v["idx"].cpu().numpy(), idx)
    assert_close(v["w"].cpu().numpy(), wt, 1e-6, 0, "route weights")
    assert np.array_equal(v["counts"].cpu().numpy(), counts)
    assert np.array_equal(v["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(v["src"].cpu().numpy(), src)
    assert np.array_equal(v["dest"].cpu().numpy(), dest)
    xb = to_np_bits(x)
    if os.environ.get("MOE_GATHER") != "1":  # with MOE_GATHER=1 the gate+up GEMM gathers x rows itself
        assert np.array_equal(to_np_bits(v["x_perm"].cpu()), xb[src])

    rng = np.random.default_rng(1)
    hot = int(np.argmax(counts))
    hot_tokens = src[offsets[hot]:offsets[hot + 1]]
    sample = np.unique(np.concatenate([tile_class_tokens(src, offsets, rng),
                                       rng.choice(hot_tokens, min(4, hot_tokens.size), replace=False)]))
    ref = oracle.forward_tokens(xb, ln, to_np_bits(wgu), to_np_bits(wd), w.k, sample.astype(np.int32))
    got = out[torch.from_numpy(sample).to(dev)].float().cpu().numpy()
    assert_layer_close(got, ref, f"{name} sampled tokens {sample.tolist()}")
