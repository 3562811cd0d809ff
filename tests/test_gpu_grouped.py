"""GPU parity of DeepSeek-V3's router (moe_route_grouped) and of the layer built on it
(moe_forward_grouped) against the CPU oracle, through the C ABI.

Both sides choose experts by comparing fp32 scores s + bias with s = sigmoid(logit); the GPU's
expf and the host's expf may round the same affinity one ulp apart, so where two candidates'
scores lie within that distance the two choices can differ and both are valid top-k selections.
How often: a token takes about three such decisions (the kept groups, the top-2 inside a group,
the k-th expert); with ~128 candidate scores spread over a range of ~1, the chance that a decision's
gap is under two ulps (1.2e-7) is ~1.2e-7 * 128 ~ 1.5e-5, so ~5e-5 per token, ~0.1 tokens at
T = 2048 (0 observed in every case here).  The tests allow at most MAX_DIFFERING_TOKENS = 2 (the
Poisson tail beyond that at 0.1 expected is ~1.5e-4) and print the count.  Every differing token is
checked in full: its choice against a float64 evaluation (the GPU's groups and experts optimal to
within 1e-6), its weights against scale * s / sum(s) over the GPU's own ids in float64 (1e-6
relative), and its layer output against the oracle fed the GPU's routing for that token.  Weights of
matching tokens agree to 1e-6 relative (both sides evaluate scale * s / sum(s) in fp32).
"""
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
from gpu_cases import assert_close, assert_layer_close, case_inputs, tile_class_tokens, to_np_bits  # noqa: E402

from mixture_experts_grouped_fp32_gb300.workloads import WORKLOADS, Workload, draw_router_bias  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_grouped_fp32_gb300 import moe as m
    m.load()
    return m


def valid_grouped_choice(logits_row, bias, ids, k, G, tg, tol=1e-6):
    """Is `ids` a top-k choice of DeepSeek-V3's router for this token, up to score ties within tol?"""
    E = logits_row.shape[0]
    gs = E // G
    q = min(gs, max(1, k // tg))
    s = 1.0 / (1.0 + np.exp(-logits_row.astype(np.float64)))
    c = s + bias.astype(np.float64)
    gsc = np.array([np.sort(c[g * gs:(g + 1) * gs])[::-1][:q].sum() for g in range(G)])
    ids = list(ids)
    if len(set(ids)) != k:
        return False
    used = {e // gs for e in ids}
    if len(used) > tg:
        return False
    # Some set of tg groups containing the used ones must be as good as the best tg groups.
    others = sorted((g for g in range(G) if g not in used), key=lambda g: -gsc[g])
    kept = sorted(used) + others[:tg - len(used)]
    if gsc[kept].sum() < np.sort(gsc)[::-1][:tg].sum() - tol * tg:
        return False
    rest = [e for e in range(E) if e // gs in kept and e not in ids]
    if rest and c[ids].min() < c[rest].max() - tol:
        return False
    return bool(np.all(np.diff(c[ids]) <= tol))  # slot order: descending score


MAX_DIFFERING_TOKENS = 2


def check_routing(idx, w, ref_idx, ref_w, logits, bias, k, G, tg, scale):
    """ids equal except near-ties (each differing token's ids and weights validated); weights of
    equal tokens close.  Returns the mask of tokens routed like the oracle."""
    same = np.all(idx == ref_idx, axis=1)
    n_diff = int((~same).sum())
    print(f"grouped router: {n_diff} of {len(same)} tokens routed differently from the oracle")
    assert n_diff <= MAX_DIFFERING_TOKENS, f"{n_diff} of {len(same)} tokens routed differently"
    for t in np.nonzero(~same)[0]:
        assert valid_grouped_choice(logits[t], bias, idx[t], k, G, tg), (t, idx[t], ref_idx[t])
        s64 = 1.0 / (1.0 + np.exp(-logits[t].astype(np.float64)[idx[t]]))
        np.testing.assert_allclose(w[t], scale * s64 / s64.sum(), rtol=1e-6, atol=0,
                                   err_msg=f"weights of differing token {t}")
    assert_close(w[same], ref_w[same], 1e-6, 0, "grouped route weights")
    return same


def merged_routing(idx, w, ref_idx, ref_w, same):
    """The oracle's routing, with the GPU's (validated) routing for the tokens that differ: the
    routing to feed the oracle's steps 2-5 so that every token's output can be compared."""
    return np.where(same[:, None], ref_idx, idx).astype(np.int32), np.where(same[:, None], ref_w, w).astype(np.float32)


ROUTE_CASES = [  # (T, E, k, n_group, topk_group, scale, bias_std)
    (2048, 256, 8, 8, 4, 2.5, 0.1),   # DeepSeek-V3's own setting
    (513, 256, 8, 8, 4, 2.5, 0.0),
    (300, 64, 6, 4, 2, 1.0, 0.3),
    (77, 16, 3, 4, 3, 1.5, 0.2),
    (64, 32, 4, 1, 1, 1.0, 0.0),      # one group, no bias: plain top-k of the logits
    (33, 8, 2, 8, 2, 2.0, 0.5),       # one expert per group
    (1, 128, 8, 32, 8, 2.5, 0.1),
    (200, 128, 4, 4, 4, 1.0, 0.2),    # 32-expert groups, one score per group (q = 1)
    (150, 64, 2, 2, 1, 1.5, 0.1),     # 32-expert groups, q = 2
]


@pytest.mark.parametrize("T,E,k,G,tg,scale,bstd", ROUTE_CASES)
def test_route_grouped_parity(moe, oracle, T, E, k, G, tg, scale, bstd):
    g = torch.Generator("cpu").manual_seed(T * 31 + E)
    logits = torch.randn(T, E, generator=g)
    bias = torch.randn(E, generator=g) * bstd
    idx, w = moe.route_grouped(logits.to(DEV), bias.to(DEV), k, G, tg, scale)
    torch.cuda.synchronize()
    ref_idx, ref_w = oracle.route_grouped(logits.numpy(), bias.numpy(), k, G, tg, scale)
    check_routing(idx.cpu().numpy(), w.cpu().numpy(), ref_idx, ref_w, logits.numpy(), bias.numpy(), k, G, tg,
                  scale)


def test_route_grouped_exact_ties(moe, oracle):
    """All logits 0 (s = 1/2 exactly) and dyadic biases: group and expert ties are exact on both
    sides and must resolve identically (lower group, then lower id)."""
    logits = torch.zeros(5, 8)
    for b in ([.5, -.25, -.25, -.25, .125, .125, -.5, -.5], [.5, -.25, -.25, -.25, .25, .125, -.5, -.5],
              [0, 0, 0, 0, 0, 0, 0, 0]):
        bias = torch.tensor(b, dtype=torch.float32)
        idx, w = moe.route_grouped(logits.to(DEV), bias.to(DEV), 2, 2, 1, 2.5)
        torch.cuda.synchronize()
        ref_idx, ref_w = oracle.route_grouped(logits.numpy(), bias.numpy(), 2, 2, 1, 2.5)
        assert np.array_equal(idx.cpu().numpy(), ref_idx)
        assert np.array_equal(w.cpu().numpy(), ref_w)


LAYER_CASES = [
    Workload("grouped_small", 64, 256, 512, 32, 4, router=("grouped", 4, 2, 1.0, 0.1)),
    Workload("grouped_dsv3_like", 40, 1024, 256, 64, 8, ("zipf", 1.2), router=("grouped", 8, 4, 2.5, 0.1)),
    Workload("grouped_many_rows", 700, 256, 512, 16, 4, router=("grouped", 4, 2, 2.5, 0.2)),
]


@pytest.mark.parametrize("w", LAYER_CASES, ids=lambda w: w.name)
def test_forward_grouped_matches_oracle(moe, oracle, w):
    _, G, tg, scale, _ = w.router
    logits, x, wgu, wd = case_inputs(w, seed=0)
    bias = draw_router_bias(w, seed=0)
    dev = torch.device(DEV)
    ws = torch.empty(moe.workspace_size(w.T, w.d, w.f, w.E, w.k), dtype=torch.uint8, device=dev)
    ws.fill_(0xFF)
    out = moe.forward_grouped(x.to(dev), logits.to(dev), bias.to(dev), wgu.to(dev), wd.to(dev), w.k, G, tg, scale,
                              workspace=ws)
    torch.cuda.synchronize()
    assert moe.get_device_error(ws) == 0
    v = moe.workspace_views(ws, w.T, w.d, w.f, w.E, w.k)
    ln, bn = logits.numpy(), bias.numpy()
    ref_idx, ref_w = oracle.route_grouped(ln, bn, w.k, G, tg, scale)
    gidx, gw = v["idx"].cpu().numpy(), v["w"].cpu().numpy()
    same = check_routing(gidx, gw, ref_idx, ref_w, ln, bn, w.k, G, tg, scale)
    midx, mw = merged_routing(gidx, gw, ref_idx, ref_w, same)
    ref = oracle.forward_routed(to_np_bits(x), midx, mw, to_np_bits(wgu), to_np_bits(wd))
    assert_layer_close(out.float().cpu().numpy(), ref, w.name)


@pytest.mark.slow
def test_forward_grouped_full_size(moe, oracle):
    """DeepSeek-V3's layer shape and router at full size (22.5 GB of weights), in the launch
    configuration bench.py times: the routing of every token is checked, the output on sampled
    tokens that the oracle computes one by one."""
    from mixture_experts_grouped_fp32_gb300.workloads import make_inputs
    w = WORKLOADS["deepseek_v3_t2048"]
    _, G, tg, scale, _ = w.router
    dev = torch.device(DEV)
    logits, x, wgu, wd = make_inputs(w, seed=0, weight_device="cuda")
    bias = draw_router_bias(w, seed=0)
    ws = torch.empty(moe.workspace_size(w.T, w.d, w.f, w.E, w.k), dtype=torch.uint8, device=dev)
    out = moe.forward_grouped(x.to(dev), logits.to(dev), bias.to(dev), wgu, wd, w.k, G, tg, scale, workspace=ws)
    torch.cuda.synchronize()
    assert moe.get_device_error(ws) == 0
    v = moe.workspace_views(ws, w.T, w.d, w.f, w.E, w.k)
    ln, bn = logits.numpy(), bias.numpy()
    ref_idx, ref_w = oracle.route_grouped(ln, bn, w.k, G, tg, scale)
    gidx, gw = v["idx"].cpu().numpy(), v["w"].cpu().numpy()
    same = check_routing(gidx, gw, ref_idx, ref_w, ln, bn, w.k, G, tg, scale)
    gc, go, gs, gd = (v[n].cpu().numpy() for n in ("counts", "offsets", "src", "dest"))
    if same.all():  # the permutation is then the oracle's, bit for bit
        counts, offsets, src, dest = oracle.permute(ref_idx, w.E)
        assert np.array_equal(gc, counts) and np.array_equal(go, offsets)
        assert np.array_equal(gs, src) and np.array_equal(gd, dest)
    else:  # a near-tie changed some ids: check the properties that define the permutation
        flat = gidx.reshape(-1)
        assert np.array_equal(gc, np.bincount(flat, minlength=w.E))
        assert np.array_equal(go, np.concatenate([[0], np.cumsum(gc)]))
        assert np.array_equal(gs, np.argsort(flat, kind="stable") // w.k)
        assert np.array_equal(gs[gd.reshape(-1)], np.repeat(np.arange(w.T), w.k))
    rng = np.random.default_rng(2)
    sample = np.unique(np.concatenate([tile_class_tokens(gs, go, rng, n_random=8), np.nonzero(~same)[0]]))
    midx, mw = merged_routing(gidx, gw, ref_idx, ref_w, same)
    ref = oracle.forward_tokens_routed(to_np_bits(x), midx[sample], mw[sample], to_np_bits(wgu),
                                       to_np_bits(wd), sample.astype(np.int32))
    got = out[torch.from_numpy(sample).to(dev)].float().cpu().numpy()
    assert_layer_close(got, ref, f"deepseek_v3_t2048 sampled tokens {sample.tolist()}")


def _quantised(moe, oracle, wgu, wd, blocks):
    """GPU weight codes and the oracle's (checked equal, so that both sides use the same weights)."""
    from mixture_experts_grouped_fp32_gb300.moe import fp8_unblock
    gq = moe.quantize_weights_fp8b if blocks else moe.quantize_weights_fp8
    oq = oracle.quantize_weights_fp8b if blocks else oracle.quantize_weights_fp8
    g = gq(wgu.to(DEV)) + gq(wd.to(DEV))
    r = oq(to_np_bits(wgu)) + oq(to_np_bits(wd))
    torch.cuda.synchronize()
    assert np.array_equal(fp8_unblock(g[0].cpu().numpy()), r[0]) and np.array_equal(g[1].cpu().numpy(), r[1])
    assert np.array_equal(fp8_unblock(g[2].cpu().numpy()), r[2]) and np.array_equal(g[3].cpu().numpy(), r[3])
    return g, r


@pytest.mark.parametrize("blocks", [False, True], ids=["fp8", "fp8b"])
@pytest.mark.parametrize("w", LAYER_CASES, ids=lambda w: w.name)
def test_forward_grouped_fp8_matches_oracle(moe, oracle, w, blocks):
    """The FP8 layers with DeepSeek-V3's router: routing as for the bf16 layer, the output of every
    token routed like the oracle's against the FP8 oracle at the layer tolerance."""
    _, G, tg, scale, _ = w.router
    logits, x, wgu, wd = case_inputs(w, seed=4)
    bias = draw_router_bias(w, seed=4)
    gw, rw = _quantised(moe, oracle, wgu, wd, blocks)
    size = moe.workspace_size_fp8b if blocks else moe.workspace_size_fp8
    views = moe.workspace_views_fp8b if blocks else moe.workspace_views_fp8
    ws = torch.empty(size(w.T, w.d, w.f, w.E, w.k), dtype=torch.uint8, device=DEV)
    out = moe.forward_grouped_fp8(x.to(DEV), logits.to(DEV), bias.to(DEV), *gw, w.k, G, tg, scale, workspace=ws,
                                  blocks=blocks)
    torch.cuda.synchronize()
    assert moe.get_device_error(ws) == 0
    v = views(ws, w.T, w.d, w.f, w.E, w.k)
    ln, bn = logits.numpy(), bias.numpy()
    ref_idx, ref_w = oracle.route_grouped(ln, bn, w.k, G, tg, scale)
    gidx, gwt = v["idx"].cpu().numpy(), v["w"].cpu().numpy()
    same = check_routing(gidx, gwt, ref_idx, ref_w, ln, bn, w.k, G, tg, scale)
    midx, mw = merged_routing(gidx, gwt, ref_idx, ref_w, same)
    fwd = oracle.forward_fp8b_tokens_routed if blocks else oracle.forward_fp8_tokens_routed
    tokens = np.arange(w.T, dtype=np.int32)
    ref = fwd(to_np_bits(x), midx, mw, *rw, tokens)
    assert_layer_close(out.float().cpu().numpy(), ref, f"{w.name} grouped router, {'fp8b' if blocks else 'fp8'}")


@pytest.mark.slow
@pytest.mark.parametrize("blocks", [False, True], ids=["fp8", "fp8b"])
def test_forward_grouped_fp8_full_size(moe, oracle, blocks):
    """DeepSeek-V3's layer shape and router at full size on the FP8 layers: weight codes bit for bit,
    routing checked for every token, the output on sampled tokens against the FP8 oracle."""
    from mixture_experts_grouped_fp32_gb300.moe import fp8_unblock
    from mixture_experts_grouped_fp32_gb300.workloads import make_inputs
    w = WORKLOADS["deepseek_v3_t2048"]
    _, G, tg, scale, _ = w.router
    logits, x, wgu, wd = make_inputs(w, seed=0, weight_device="cuda")
    bias = draw_router_bias(w, seed=0)
    gq = moe.quantize_weights_fp8b if blocks else moe.quantize_weights_fp8
    gw = gq(wgu) + gq(wd)
    torch.cuda.synchronize()
    wgu_bits, wd_bits = to_np_bits(wgu), to_np_bits(wd)
    del wgu, wd
    torch.cuda.empty_cache()
    size = moe.workspace_size_fp8b if blocks else moe.workspace_size_fp8
    views = moe.workspace_views_fp8b if blocks else moe.workspace_views_fp8
    ws = torch.empty(size(w.T, w.d, w.f, w.E, w.k), dtype=torch.uint8, device=DEV)
    out = moe.forward_grouped_fp8(x.to(DEV), logits.to(DEV), bias.to(DEV), *gw, w.k, G, tg, scale, workspace=ws,
                                  blocks=blocks)
    torch.cuda.synchronize()
    assert moe.get_device_error(ws) == 0
    v = views(ws, w.T, w.d, w.f, w.E, w.k)
    oq = oracle.quantize_weights_fp8b if blocks else oracle.quantize_weights_fp8
    r_gu = oq(wgu_bits)
    assert np.array_equal(fp8_unblock(gw[0].cpu().numpy()), r_gu[0]) and np.array_equal(gw[1].cpu().numpy(), r_gu[1])
    del wgu_bits
    r_d = oq(wd_bits)
    assert np.array_equal(fp8_unblock(gw[2].cpu().numpy()), r_d[0]) and np.array_equal(gw[3].cpu().numpy(), r_d[1])
    del wd_bits
    ln, bn = logits.numpy(), bias.numpy()
    ref_idx, ref_w = oracle.route_grouped(ln, bn, w.k, G, tg, scale)
    gidx, gwt = v["idx"].cpu().numpy(), v["w"].cpu().numpy()
    same = check_routing(gidx, gwt, ref_idx, ref_w, ln, bn, w.k, G, tg, scale)
    midx, mw = merged_routing(gidx, gwt, ref_idx, ref_w, same)
    rng = np.random.default_rng(7)
    go, gs = v["offsets"].cpu().numpy(), v["src"].cpu().numpy()
    sample = np.unique(np.concatenate([tile_class_tokens(gs, go, rng), np.nonzero(~same)[0]])).astype(np.int32)
    fwd = oracle.forward_fp8b_tokens_routed if blocks else oracle.forward_fp8_tokens_routed
    ref = fwd(to_np_bits(x), midx[sample], mw[sample], *r_gu, *r_d, sample)
    got = out[torch.from_numpy(sample).long().to(DEV)].float().cpu().numpy()
    assert_layer_close(got, ref, f"deepseek_v3_t2048 {'fp8b' if blocks else 'fp8'} sampled tokens {sample.tolist()}")


@pytest.mark.parametrize("variant", ["bf16", "fp8", "fp8b"])
def test_forward_grouped_host_batches_matches_forward(moe, variant):
    """DeepSeek-V3's router over host batches with overlapped copies: each batch's output equals
    the device call's."""
    w = LAYER_CASES[0]
    _, G, tg, scale, _ = w.router
    dev = torch.device(DEV)
    _, _, wgu, wd = case_inputs(w, seed=50)
    bias = draw_router_bias(w, seed=50).to(dev)
    if variant == "bf16":
        wts = (wgu.to(dev), wd.to(dev))
        fwd = lambda x, l: moe.forward_grouped(x, l, bias, *wts, w.k, G, tg, scale)
        size = moe.workspace_size
    else:
        blocks = variant == "fp8b"
        quant = moe.quantize_weights_fp8b if blocks else moe.quantize_weights_fp8
        wts = quant(wgu.to(dev)) + quant(wd.to(dev))
        fwd = lambda x, l: moe.forward_grouped_fp8(x, l, bias, *wts, w.k, G, tg, scale, blocks=blocks)
        size = moe.workspace_size_fp8b if blocks else moe.workspace_size_fp8
    xs, ls, refs = [], [], []
    for i in range(3):
        logits, x, _, _ = case_inputs(w, seed=60 + i)
        xs.append(x.pin_memory())
        ls.append(logits.pin_memory())
        refs.append(fwd(x.to(dev), logits.to(dev)).cpu())
    outs = [torch.full((w.T, w.d), -1.0, dtype=torch.bfloat16).pin_memory() for _ in range(3)]
    ws = torch.empty(size(w.T, w.d, w.f, w.E, w.k) + 2 * moe.host_staging_size(w.T, w.d, w.E), dtype=torch.uint8,
                     device=dev)
    if variant == "bf16":
        moe.forward_grouped_host_batches(xs, ls, bias, *wts, w.k, G, tg, scale, outs, ws)
    else:
        moe.forward_grouped_fp8_host_batches(xs, ls, bias, *wts, w.k, G, tg, scale, outs, ws, blocks=variant == "fp8b")
    torch.cuda.current_stream().synchronize()
    assert moe.get_device_error(ws) == 0
    for i in range(3):
        assert torch.equal(outs[i].view(torch.int16), refs[i].view(torch.int16)), f"{variant} batch {i}"
