"""Pins for the CPU oracle: checks against facts that do not come from the oracle itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises ``AssertionError`` when the oracle disagrees
with a closed form, a hand-worked example, a library routine (numpy / scipy) or a float64
brute force written here from the layer's definition.  ``test_oracle_pins.py`` runs them on the
real oracle; ``test_oracle_mutants.py`` runs them on deliberately broken copies of the oracle
and expects each copy to fail at least one pin.

The layer (per token t, chosen experts e_j, weights w_j):
    out[t] = sum_j w_j * ( silu(x W_gate[e_j]) * (x W_up[e_j]) ) W_down[e_j]
with W_gate_up[e] = [W_gate[e] | W_up[e]] ([d, 2f]) and silu(z) = z * sigmoid(z).
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import expit, softmax

from oracle import bf16_bits_to_f32


def sigma(z: float) -> float:
    return 1.0 / (1.0 + math.exp(-z))


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest even) and return the bit patterns."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


# --------------------------------------------------------------------------------------------
# Hand-worked example: E = 3 experts, top-2, d = f = 2, T = 4 tokens.
#   W_gate[e] = a_e * I with a = (1, 2, 0.5);  W_up[e] = I;  W_down[e] = c_e * I with c = (1, 0.5, -1)
#   so expert e maps x to y_i = c_e * silu(a_e x_i) * x_i = c_e * a_e * x_i^2 * sigma(a_e x_i).
#   Per expert: e0: y_i = x_i^2 sigma(x_i);  e1: y_i = x_i^2 sigma(2 x_i);  e2: y_i = -x_i^2 sigma(x_i/2) / 2.
# Tokens (x; logits) and the hand derivation:
#   t0 x=[1,-1];  logits [0,0,0]: three-way tie -> lowest ids first: idx [0,1], w [1/2, 1/2].
#       e0 -> [s(1), s(-1)], e1 -> [s(2), s(-2)]  => out = [(s1+s2)/2, (s(-1)+s(-2))/2]
#   t1 x=[2,0];   logits [1,0,2]: order e2 (2) > e0 (1) > e1 (0): idx [2,0];
#       w = softmax over {2,1} = [s(1), s(-1)].  e2 -> [-2 s(1), 0], e0 -> [4 s(2), 0]
#       => out = [-2 s(1)^2 + 4 s(-1) s(2), 0]
#   t2 x=[1,2];   logits [0,1,1]: tie for first between e1, e2 -> idx [1,2], w [1/2,1/2].
#       e1 -> [s(2), 4 s(4)], e2 -> [-s(1/2)/2, -2 s(1)]  => out = [(s2 - s(1/2)/2)/2, 2 s(4) - s(1)]
#   t3 x=[-2,1];  logits [3,1,1]: e0 first, tie e1/e2 for second -> idx [0,1];
#       w = softmax over {3,1} = [s(2), s(-2)].  e0 -> [4 s(-2), s(1)], e1 -> [4 s(-4), s(2)]
#       => out = [4 s(2) s(-2) + 4 s(-2) s(-4), s(2) s(1) + s(-2) s(2)]
#   Counting sort by expert then token: e0 <- t0,t1,t3 (rows 0,1,2); e1 <- t0,t2,t3 (rows 3,4,5);
#   e2 <- t1,t2 (rows 6,7).  counts [3,3,2], offsets [0,3,6,8], src [0,1,3,0,2,3,1,2],
#   dest [[0,3],[6,1],[4,7],[2,5]].
# Every weight and x value is exactly representable in bf16.
# --------------------------------------------------------------------------------------------
HAND_X = np.array([[1, -1], [2, 0], [1, 2], [-2, 1]], np.float32)
HAND_LOGITS = np.array([[0, 0, 0], [1, 0, 2], [0, 1, 1], [3, 1, 1]], np.float32)
HAND_A = (1.0, 2.0, 0.5)
HAND_C = (1.0, 0.5, -1.0)


def hand_weights():
    E, d, f = 3, 2, 2
    wgu = np.zeros((E, d, 2 * f), np.float32)
    wd = np.zeros((E, f, d), np.float32)
    for e in range(E):
        wgu[e, :, :f] = HAND_A[e] * np.eye(2)
        wgu[e, :, f:] = np.eye(2)
        wd[e] = HAND_C[e] * np.eye(2)
    return f32_to_bf16_bits(wgu), f32_to_bf16_bits(wd)


def hand_expected():
    s = sigma
    idx = np.array([[0, 1], [2, 0], [1, 2], [0, 1]], np.int32)
    w = np.array([[0.5, 0.5], [s(1), s(-1)], [0.5, 0.5], [s(2), s(-2)]])
    out = np.array([
        [(s(1) + s(2)) / 2, (s(-1) + s(-2)) / 2],
        [-2 * s(1) ** 2 + 4 * s(-1) * s(2), 0.0],
        [(s(2) - s(0.5) / 2) / 2, 2 * s(4) - s(1)],
        [4 * s(2) * s(-2) + 4 * s(-2) * s(-4), s(2) * s(1) + s(-2) * s(2)],
    ])
    counts = np.array([3, 3, 2], np.int32)
    offsets = np.array([0, 3, 6, 8], np.int32)
    src = np.array([0, 1, 3, 0, 2, 3, 1, 2], np.int32)
    dest = np.array([[0, 3], [6, 1], [4, 7], [2, 5]], np.int32)
    return idx, w, out, counts, offsets, src, dest


def pin_hand_example(O):
    idx_e, w_e, out_e, counts_e, offsets_e, src_e, dest_e = hand_expected()
    x_bits = f32_to_bf16_bits(HAND_X)
    wgu, wd = hand_weights()
    idx, w = O.route(HAND_LOGITS, 2)
    assert np.array_equal(idx, idx_e), (idx, idx_e)
    np.testing.assert_allclose(w, w_e, rtol=1e-6, atol=0)
    counts, offsets, src, dest = O.permute(idx, 3)
    assert np.array_equal(counts, counts_e)
    assert np.array_equal(offsets, offsets_e)
    assert np.array_equal(src, src_e)
    assert np.array_equal(dest, dest_e)
    out = O.forward(x_bits, HAND_LOGITS, wgu, wd, 2)
    np.testing.assert_allclose(out, out_e, rtol=1e-6, atol=1e-7)
    out_rows = O.forward_tokens(x_bits, HAND_LOGITS, wgu, wd, 2, np.array([3, 0], np.int32))
    np.testing.assert_allclose(out_rows, out_e[[3, 0]], rtol=1e-6, atol=1e-7)


# --------------------------------------------------------------------------------------------
# Random small layers and a float64 brute force written from the definition: per token, pick the
# k largest logits (stable, lower id first on ties), softmax-renormalise, run each chosen
# expert's dense SwiGLU FFN in float64 with numpy matmuls, and sum.  No permutation.
# --------------------------------------------------------------------------------------------
def random_layer(rng, T, d, f, E, tie_logits=False):
    if tie_logits:
        logits = rng.integers(0, 3, size=(T, E)).astype(np.float32)
    else:
        logits = rng.standard_normal((T, E)).astype(np.float32)
    x_bits = f32_to_bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    wgu_bits = f32_to_bf16_bits((0.3 * rng.standard_normal((E, d, 2 * f))).astype(np.float32))
    wd_bits = f32_to_bf16_bits((0.3 * rng.standard_normal((E, f, d))).astype(np.float32))
    return logits, x_bits, wgu_bits, wd_bits


def brute_force_forward(logits, x_bits, wgu_bits, wd_bits, k):
    T, E = logits.shape
    f = wgu_bits.shape[2] // 2
    x = bf16_bits_to_f32(x_bits).astype(np.float64)
    wgu = bf16_bits_to_f32(wgu_bits).astype(np.float64)
    wd = bf16_bits_to_f32(wd_bits).astype(np.float64)
    out = np.zeros((T, x.shape[1]))
    for t in range(T):
        chosen = np.argsort(-logits[t].astype(np.float64), kind="stable")[:k]
        p = softmax(logits[t].astype(np.float64))
        wts = p[chosen] / p[chosen].sum()
        for e, wt in zip(chosen, wts):
            g = x[t] @ wgu[e][:, :f]
            u = x[t] @ wgu[e][:, f:]
            out[t] += wt * ((g * expit(g) * u) @ wd[e])
    return out


BRUTE_SHAPES = [  # (T, d, f, E, k, tie_logits)
    (16, 32, 24, 6, 2, False),
    (9, 16, 32, 5, 3, True),
    (12, 8, 8, 4, 4, False),
    (7, 24, 16, 6, 1, True),
    (1, 32, 32, 3, 2, False),
]


def pin_brute_force(O, seed=1234):
    rng = np.random.default_rng(seed)
    for T, d, f, E, k, ties in BRUTE_SHAPES:
        logits, x_bits, wgu, wd = random_layer(rng, T, d, f, E, ties)
        ref = brute_force_forward(logits, x_bits, wgu, wd, k)
        out = O.forward(x_bits, logits, wgu, wd, k)
        err = np.abs(out - ref).max()
        assert err <= 1e-5 * max(1.0, np.abs(ref).max()), (T, d, f, E, k, err)
        tok = np.arange(T - 1, -1, -2, dtype=np.int32)
        rows = O.forward_tokens(x_bits, logits, wgu, wd, k, tok)
        err = np.abs(rows - ref[tok]).max()
        assert err <= 1e-5 * max(1.0, np.abs(ref).max()), ("tokens", T, d, f, E, k, err)


def pin_dense_e1_k1(O, seed=7):
    """E = 1, k = 1: the layer is the dense SwiGLU FFN silu(x Wg) * (x Wu) @ Wd (numpy matmul)."""
    rng = np.random.default_rng(seed)
    T, d, f = 10, 48, 40
    logits, x_bits, wgu_bits, wd_bits = random_layer(rng, T, d, f, 1)
    x = bf16_bits_to_f32(x_bits).astype(np.float64)
    wg = bf16_bits_to_f32(wgu_bits[0, :, :f]).astype(np.float64)
    wu = bf16_bits_to_f32(wgu_bits[0, :, f:]).astype(np.float64)
    wd = bf16_bits_to_f32(wd_bits[0]).astype(np.float64)
    g = x @ wg
    ref = (g * expit(g) * (x @ wu)) @ wd
    out = O.forward(x_bits, logits, wgu_bits, wd_bits, 1)
    assert np.abs(out - ref).max() <= 1e-5 * np.abs(ref).max()
    _, w = O.route(logits, 1)
    assert np.all(w == 1.0)


def pin_route_library(O, seed=11):
    """Top-k ids equal numpy's stable argsort of -logits; weights equal scipy's softmax renormalised."""
    rng = np.random.default_rng(seed)
    for T, E, k, ties in [(64, 8, 2, False), (50, 7, 3, True), (33, 40, 8, False), (20, 256, 8, True),
                          (5, 5, 5, False), (17, 6, 6, True)]:
        logits = (rng.integers(0, 4, (T, E)) if ties else rng.standard_normal((T, E))).astype(np.float32)
        idx, w = O.route(logits, k)
        ref_idx = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :k]
        assert np.array_equal(idx, ref_idx), (T, E, k)
        p = softmax(logits.astype(np.float64), axis=1)
        pk = np.take_along_axis(p, ref_idx, axis=1)
        np.testing.assert_allclose(w, pk / pk.sum(axis=1, keepdims=True), rtol=1e-6, atol=0)
        np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-6)
        if k == E:  # all experts kept: the weights are the full softmax
            np.testing.assert_allclose(np.take_along_axis(w, np.argsort(idx, axis=1), 1), p,
                                       rtol=1e-6, atol=0)


def pin_route_nan_order(O, seed=13):
    """Rows with NaN logits: the ids equal numpy's stable argsort of -logits, which sorts NaN after
    every number (-inf included) and keeps ascending id among NaNs; rows without a NaN keep their
    weights.  (The pages define no non-finite logits; this is the order both sides take.)"""
    rng = np.random.default_rng(seed)
    T, E, k = 40, 8, 3
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[1:8, 2] = np.nan                      # one NaN
    logits[8:12, [0, 5]] = np.nan                # two NaNs, below everything
    logits[12:14, :] = np.nan                    # all NaN -> ids 0, 1, 2
    logits[14:16, 3] = -np.inf                   # -inf still ranks above NaN
    logits[14:16, 6] = np.nan
    logits[16:18, :6] = np.nan                   # only two numbers left for three slots
    idx, w = O.route(logits, k)
    ref_idx = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :k]
    assert np.array_equal(idx, ref_idx)
    assert np.array_equal(idx[12], [0, 1, 2]) and np.array_equal(idx[16][:2], [6, 7])
    clean = ~np.isnan(logits).any(axis=1) & ~np.isinf(logits).any(axis=1)
    p = softmax(logits[clean].astype(np.float64), axis=1)
    pk = np.take_along_axis(p, ref_idx[clean], axis=1)
    np.testing.assert_allclose(w[clean], pk / pk.sum(axis=1, keepdims=True), rtol=1e-6, atol=0)


def pin_permute_library(O, seed=5):
    """The permutation equals numpy's stable argsort of the flattened expert ids."""
    rng = np.random.default_rng(seed)
    for T, E, k in [(40, 8, 2), (31, 16, 4), (1, 3, 3), (64, 256, 8), (25, 1, 1)]:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        counts, offsets, src, dest = O.permute(idx, E)
        flat = idx.reshape(-1)
        order = np.argsort(flat, kind="stable")
        assert np.array_equal(counts, np.bincount(flat, minlength=E))
        assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
        assert np.array_equal(src, order // k)
        ref_dest = np.empty(T * k, np.int64)
        ref_dest[order] = np.arange(T * k)
        assert np.array_equal(dest.reshape(-1), ref_dest)


def pin_invariants(O, seed=3):
    """Layer invariants on a random layer: counts sum to T*k, src/dest are inverse bijections,
    each row lies in its expert's segment, tokens ascend within a segment, weights sum to 1."""
    rng = np.random.default_rng(seed)
    T, E, k = 57, 9, 3
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx, w = O.route(logits, k)
    assert all(len(set(r)) == k for r in idx.tolist())
    assert np.all(np.diff(np.take_along_axis(logits, idx, 1), axis=1) <= 0)
    np.testing.assert_allclose(w.sum(1), 1.0, atol=1e-6, rtol=0)
    counts, offsets, src, dest = O.permute(idx, E)
    assert counts.sum() == T * k and np.all(np.diff(offsets) >= 0)
    for t in range(T):
        for j in range(k):
            r = dest[t, j]
            assert src[r] == t
            assert offsets[idx[t, j]] <= r < offsets[idx[t, j] + 1]
    for e in range(E):
        seg = src[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)
    assert np.array_equal(np.sort(dest.reshape(-1)), np.arange(T * k))


def pin_stages(O, seed=9):
    """The stage entry points compose to the one-call forward, and each stage matches its own
    library-routine statement (gather = fancy indexing, down = per-row matmul in float64,
    combine = weighted sum of gathered rows)."""
    rng = np.random.default_rng(seed)
    T, d, f, E, k = 13, 16, 24, 4, 2
    logits, x_bits, wgu, wd = random_layer(rng, T, d, f, E)
    idx, w = O.route(logits, k)
    counts, offsets, src, dest = O.permute(idx, E)
    xp = O.gather_rows(x_bits, src)
    assert np.array_equal(xp, x_bits[src])
    h = O.gateup_swiglu(xp, offsets, wgu)
    expert_of_row = np.repeat(np.arange(E), counts)
    xpf = bf16_bits_to_f32(xp).astype(np.float64)
    wguf = bf16_bits_to_f32(wgu).astype(np.float64)
    g_ref = np.stack([xpf[r] @ wguf[expert_of_row[r]][:, :f] for r in range(T * k)])
    u_ref = np.stack([xpf[r] @ wguf[expert_of_row[r]][:, f:] for r in range(T * k)])
    h_ref = g_ref * expit(g_ref) * u_ref
    assert np.abs(h - h_ref).max() <= 1e-5 * np.abs(h_ref).max()
    y = O.down(h, offsets, wd)
    wdf = bf16_bits_to_f32(wd).astype(np.float64)
    y_ref = np.stack([h[r].astype(np.float64) @ wdf[expert_of_row[r]] for r in range(T * k)])
    assert np.abs(y - y_ref).max() <= 1e-5 * np.abs(y_ref).max()
    hb = f32_to_bf16_bits(h)
    y16 = O.down(hb, offsets, wd)
    y16_ref = np.stack([bf16_bits_to_f32(hb[r]).astype(np.float64) @ wdf[expert_of_row[r]]
                        for r in range(T * k)])
    assert np.abs(y16 - y16_ref).max() <= 1e-5 * np.abs(y16_ref).max()
    out = O.combine(y, w, dest)
    out_ref = np.einsum("tk,tkd->td", w.astype(np.float64), y.astype(np.float64)[dest])
    assert np.abs(out - out_ref).max() <= 1e-6 * np.abs(out_ref).max()
    full = O.forward(x_bits, logits, wgu, wd, k)
    assert np.array_equal(full, out)


# --------------------------------------------------------------------------------------------
# The second router (DeepSeek-V3's): s = sigmoid(logit), selection score c = s + bias, experts in
# G equal groups, group score = sum of the group's q = k / topk_group largest c, keep the
# topk_group best groups (equal -> lower group), then the k largest c among their experts (equal
# -> lower id), w = scale * s / sum(s over the chosen).
# --------------------------------------------------------------------------------------------
def pin_grouped_hand_example(O):
    """Hand-worked cases with exact fp32 values (all logits 0, so s = 1/2 everywhere, and
    dyadic biases).  E = 8 in G = 2 groups {0..3}, {4..7}; topk_group = 1; k = 2 (q = 2); scale 2.5.
      bias A = [.5, -.25, -.25, -.25, .125, .125, -.5, -.5] -> c = [1, .25, .25, .25, .625, .625, 0, 0]
        group scores 1 + .25 = 1.25 and .625 + .625 = 1.25: a tie, the lower group (0) is kept;
        inside it c = 1 first, then a three-way tie at .25 -> id 1.  idx [0, 1], w = 2.5 * [.5, .5].
      bias B = A with bias[4] = .25 -> group 1 scores .75 + .625 = 1.375 > 1.25: group 1 is kept and
        idx = [4, 5] although expert 0 has the largest c overall (plain top-2 would give [0, 4]).
      The bias moves the selection only: w = 2.5 * [.5, .5] = [1.25, 1.25] in both cases."""
    logits = np.zeros((2, 8), np.float32)
    bias_a = np.array([.5, -.25, -.25, -.25, .125, .125, -.5, -.5], np.float32)
    bias_b = bias_a.copy()
    bias_b[4] = .25
    idx, w = O.route_grouped(logits, bias_a, 2, 2, 1, 2.5)
    assert idx.tolist() == [[0, 1], [0, 1]], idx
    assert w.tolist() == [[1.25, 1.25], [1.25, 1.25]], w
    idx, w = O.route_grouped(logits, bias_b, 2, 2, 1, 2.5)
    assert idx.tolist() == [[4, 5], [4, 5]], idx
    assert w.tolist() == [[1.25, 1.25], [1.25, 1.25]], w
    # Weights from distinct affinities (no bias, one group, k = 3 of 4): closed form in float64.
    lg = np.array([[math.log(3.0), 0.0, -math.log(3.0), math.log(7.0)]], np.float32)
    idx, w = O.route_grouped(lg, np.zeros(4, np.float32), 3, 1, 1, 1.0)
    assert idx.tolist() == [[3, 0, 1]], idx  # sigma: 7/8 > 3/4 > 1/2 > 1/4
    ref = np.array([7 / 8, 3 / 4, 1 / 2]) / (7 / 8 + 3 / 4 + 1 / 2)
    np.testing.assert_allclose(w[0], ref, rtol=1e-6, atol=0)


def pin_grouped_reduces_to_topk(O, seed=21):
    """One group and no bias: sigmoid is increasing, so the chosen ids are the k largest logits —
    the softmax router's ids (pinned to numpy's argsort above) — and the weights are scipy's
    expit of those logits, normalised and scaled."""
    rng = np.random.default_rng(seed)
    for T, E, k, scale in [(40, 8, 2, 1.0), (25, 64, 6, 2.5), (16, 256, 8, 2.5), (9, 5, 5, 0.5)]:
        logits = rng.standard_normal((T, E)).astype(np.float32)
        idx, w = O.route_grouped(logits, np.zeros(E, np.float32), k, 1, 1, scale)
        ref_idx, _ = O.route(logits, k)
        assert np.array_equal(idx, np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :k])
        assert np.array_equal(idx, ref_idx)
        s = expit(np.take_along_axis(logits, idx, 1).astype(np.float64))
        np.testing.assert_allclose(w, scale * s / s.sum(1, keepdims=True), rtol=1e-6, atol=0)


def grouped_brute_force(logits, bias, k, G, topk_group, scale):
    """float64 brute force over every set of topk_group groups and every k-subset of their experts.
    Returns (idx, w, margin): margin = the smallest score gap a decision rested on, so callers can
    skip decisions that float32 rounding could flip."""
    import itertools
    T, E = logits.shape
    gs = E // G
    q = min(gs, max(1, k // topk_group))
    idx = np.empty((T, k), np.int64)
    w = np.empty((T, k))
    margin = np.empty(T)
    for t in range(T):
        s = 1.0 / (1.0 + np.exp(-logits[t].astype(np.float64)))
        c = s + bias.astype(np.float64)
        gsc = [sum(sorted(c[g * gs:(g + 1) * gs], reverse=True)[:q]) for g in range(G)]
        best = max(itertools.combinations(range(G), topk_group), key=lambda gg: sum(gsc[g] for g in gg))
        allowed = [e for e in range(E) if e // gs in best]
        pick = max(itertools.combinations(allowed, k), key=lambda es: sum(c[e] for e in es))
        pick = sorted(pick, key=lambda e: -c[e])
        idx[t] = pick
        w[t] = scale * s[pick] / s[pick].sum()
        kept_g = sorted(gsc[g] for g in best)
        rest_g = [gsc[g] for g in range(G) if g not in best]
        rest_e = [c[e] for e in allowed if e not in pick]
        gaps = [kept_g[0] - max(rest_g)] if rest_g else [1.0]
        gaps += [min(c[pick]) - max(rest_e)] if rest_e else []
        gaps += list(-np.diff(c[pick]))
        margin[t] = min(gaps)
    return idx, w, margin


def pin_grouped_brute_force(O, seed=23):
    """Random layers against the float64 brute force: the same groups, ids and slot order, and
    the same weights to 1e-6, wherever the decision margin is wider than float32 rounding."""
    rng = np.random.default_rng(seed)
    checked = 0
    for T, E, k, G, tg, scale in [(30, 8, 2, 2, 1, 2.5), (30, 16, 4, 4, 2, 1.0), (20, 16, 3, 4, 3, 1.5),
                                  (20, 12, 4, 3, 2, 2.5), (10, 32, 8, 8, 4, 2.5)]:
        logits = rng.standard_normal((T, E)).astype(np.float32)
        bias = (0.2 * rng.standard_normal(E)).astype(np.float32)
        idx, w = O.route_grouped(logits, bias, k, G, tg, scale)
        ref_idx, ref_w, margin = grouped_brute_force(logits, bias, k, G, tg, scale)
        ok = margin > 1e-5
        assert ok.mean() > 0.9
        assert np.array_equal(idx[ok], ref_idx[ok]), (T, E, k, G, tg)
        np.testing.assert_allclose(w[ok], ref_w[ok], rtol=1e-6, atol=0)
        checked += int(ok.sum())
    assert checked > 100


def pin_grouped_invariants(O, seed=29):
    """DeepSeek-V3-shaped routing (E = 256, 8 groups of 32, 4 groups kept, top-8): distinct ids
    from at most 4 groups, weights summing to the scale, weights proportional to sigmoid(logit),
    and no unchosen expert of a kept group beating a chosen one on s + bias."""
    rng = np.random.default_rng(seed)
    T, E, k, G, tg, scale = 64, 256, 8, 8, 4, 2.5
    logits = rng.standard_normal((T, E)).astype(np.float32)
    bias = (0.1 * rng.standard_normal(E)).astype(np.float32)
    idx, w = O.route_grouped(logits, bias, k, G, tg, scale)
    s = expit(logits.astype(np.float64))
    c = s + bias
    for t in range(T):
        ids = idx[t].tolist()
        assert len(set(ids)) == k and all(0 <= e < E for e in ids)
        groups = {e // 32 for e in ids}
        assert len(groups) <= tg
        np.testing.assert_allclose(w[t].sum(), scale, rtol=1e-6)
        np.testing.assert_allclose(w[t] / w[t].sum(), s[t, ids] / s[t, ids].sum(), rtol=1e-6)
        assert np.all(np.diff(c[t, ids]) <= 1e-7)  # slot order: descending selection score
        kept = [e for e in range(E) if e // 32 in groups and e not in ids]
        assert max(c[t, kept]) <= min(c[t, ids]) + 1e-7


# --------------------------------------------------------------------------------------------
# The FP8 variant: E4M3 (OCP 8-bit float, E4M3: bias 7, 3 mantissa bits, no infinities, S.1111.111
# NaN, largest finite 448), per-row / per-output-channel scales absmax / 448.
# --------------------------------------------------------------------------------------------
def e4m3_table():
    """Value of every code, written from the format definition (float64; NaN for the two NaN codes)."""
    vals = np.empty(256)
    for c in range(256):
        sgn, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            vals[c] = np.nan
        elif e == 0:
            vals[c] = (m / 8) * 2.0 ** -6
        else:
            vals[c] = (1 + m / 8) * 2.0 ** (e - 7)
        if sgn:
            vals[c] = -vals[c]
    return vals


def pin_e4m3_decode_table(O):
    """All 256 codes decode to the format's values; the landmarks of the format."""
    tab = e4m3_table()
    dec = O.e4m3_decode(np.arange(256, dtype=np.uint8)).astype(np.float64)
    assert np.array_equal(np.isnan(dec), np.isnan(tab))
    ok = ~np.isnan(tab)
    assert np.array_equal(dec[ok], tab[ok])
    assert dec[0x7E] == 448 and dec[0x08] == 2.0 ** -6 and dec[0x01] == 2.0 ** -9 and dec[0x38] == 1.0
    assert np.isnan(dec[0x7F]) and np.isnan(dec[0xFF])


def e4m3_brute_encode(x):
    """Nearest E4M3 code by search over every finite value, ties to the even (lsb 0) code, values
    above 448 saturating to +-448; NaN -> 0x7F."""
    tab = e4m3_table()
    pos = [c for c in range(128) if not np.isnan(tab[c])]
    pv = np.array([tab[c] for c in pos])
    out = np.empty(x.shape, np.uint8)
    for i, v in enumerate(np.asarray(x, np.float64).reshape(-1)):
        if np.isnan(v):
            out.reshape(-1)[i] = 0x7F
            continue
        a = min(abs(v), 448.0)
        dist = np.abs(pv - a)
        best = np.flatnonzero(dist == dist.min())
        c = pos[best[0]] if len(best) == 1 else next(pos[b] for b in best if pos[b] % 2 == 0)
        out.reshape(-1)[i] = c | (0x80 if np.signbit(v) else 0)
    return out


def pin_e4m3_encode_rne(O, seed=41):
    """Encoding = nearest-value search with ties to even and saturation: on every representable
    value, every midpoint between neighbours (the ties), just above and below each midpoint, and
    random magnitudes across the whole range (subnormals and saturation included)."""
    tab = e4m3_table()
    fin = np.array(sorted({abs(v) for v in tab if not np.isnan(v)}))
    mids = (fin[:-1] + fin[1:]) / 2
    rng = np.random.default_rng(seed)
    rand = np.exp(rng.uniform(np.log(2.0 ** -12), np.log(600.0), 4000)) * rng.choice([-1, 1], 4000)
    xs = np.concatenate([fin, -fin, mids, -mids, np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
                         np.nextafter(mids.astype(np.float32), np.float32(0)), rand, [460.0, 464.0, 470.0, 1e6]])
    xs = xs.astype(np.float32)
    assert np.array_equal(O.e4m3_encode(xs), e4m3_brute_encode(xs))


def pin_quantize_rows_fp8(O, seed=43):
    """Per-row quantisation: scale = absmax / 448, the absmax element maps to +-448 exactly, every
    value is within half a quantum of its code's value times the scale, and a zero row gives
    scale 1 and zero codes."""
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((20, 300)).astype(np.float32) * np.exp(rng.uniform(-6, 6, (20, 1))).astype(np.float32)
    a[3] = 0.0
    bits = f32_to_bf16_bits(a)
    af = bf16_bits_to_f32(bits).astype(np.float64)
    q, sc = O.quantize_rows_fp8(bits)
    tab = e4m3_table()
    for r in range(a.shape[0]):
        amax = np.abs(af[r]).max()
        if amax == 0:
            assert sc[r] == 1.0 and not q[r].any()
            continue
        assert sc[r] == np.float32(np.float32(amax) / np.float32(448.0))
        j = int(np.argmax(np.abs(af[r])))
        assert abs(tab[q[r, j]]) == 448.0
        rec = tab[q[r]] * sc[r]
        # half a quantum: 2^-4 relative for normals, 2^-10 * scale in the subnormal range
        bound = np.maximum(np.abs(af[r]) * 2.0 ** -4, 2.0 ** -10 * sc[r]) * (1 + 1e-6)
        assert np.all(np.abs(rec - af[r]) <= bound), r


def pin_fp8_forward(O, seed=47):
    """The FP8 layer against a float64 statement of it built from the pinned pieces (router,
    E4M3 quantiser): dequantised operands, per-row and per-channel scales, h rounded to bf16 and
    requantised per row, slot-ordered combine."""
    rng = np.random.default_rng(seed)
    T, d, f, E, k = 9, 32, 48, 4, 2
    logits, x_bits, wgu, wd = random_layer(rng, T, d, f, E)
    wgu8, sgu = O.quantize_weights_fp8(wgu)
    wd8, sdn = O.quantize_weights_fp8(wd)
    # The weight quantiser is the row quantiser on the transposed weights.
    for e in range(E):
        q, sc = O.quantize_rows_fp8(np.ascontiguousarray(wgu[e].T))
        assert np.array_equal(q, wgu8[e]) and np.array_equal(sc, sgu[e])
    out = O.forward_fp8(x_bits, logits, wgu8, sgu, wd8, sdn, k)
    idx, w = O.route(logits, k)
    tab = e4m3_table()
    ref = np.zeros((T, d))
    for t in range(T):
        x8, sx = O.quantize_rows_fp8(x_bits[t:t + 1])
        xd = tab[x8[0]]
        for j in range(k):
            e = idx[t, j]
            gu = (tab[wgu8[e]] @ xd) * (np.float64(sx[0]) * sgu[e].astype(np.float64))
            g, u = gu[:f], gu[f:]
            hb = f32_to_bf16_bits((g / (1 + np.exp(-g)) * u).astype(np.float32))[None, :]
            h8, sh = O.quantize_rows_fp8(hb)
            y = (tab[wd8[e]] @ tab[h8[0]]) * (np.float64(sh[0]) * sdn[e].astype(np.float64))
            ref[t] += w[t, j] * y
    err = np.abs(out - ref).max()
    assert err <= 2e-3 * np.abs(ref).max(), err


def pin_fp8_stages(O, seed=53):
    """The FP8 stage functions composed in the layer's order (permute, quantise x_perm rows,
    gate+up, quantise h rows, down, combine) give the FP8 layer's output exactly (the same fp32
    operations in the same order), on a layer where one expert receives no token."""
    rng = np.random.default_rng(seed)
    T, d, f, E, k = 11, 32, 48, 5, 2
    logits, x_bits, wgu, wd = random_layer(rng, T, d, f, E)
    logits[:, 3] = -30.0  # expert 3 never chosen: an empty segment
    wgu8, sgu = O.quantize_weights_fp8(wgu)
    wd8, sdn = O.quantize_weights_fp8(wd)
    out = O.forward_fp8(x_bits, logits, wgu8, sgu, wd8, sdn, k)
    idx, w = O.route(logits, k)
    counts, offsets, src, dest = O.permute(idx, E)
    assert counts[3] == 0
    x8, sx = O.quantize_rows_fp8(x_bits[src])
    h = O.gateup_swiglu_fp8(x8, sx, offsets, wgu8, sgu)
    h8, sh = O.quantize_rows_fp8(h)
    y = O.down_fp8(h8, sh, offsets, wd8, sdn)
    got = O.combine(y, w, dest)
    assert np.array_equal(got, out)


# --------------------------------------------------------------------------------------------
# Blockwise FP8: 1 x 128 activation blocks, 128 x 128 weight blocks, power-of-two block scales.
# --------------------------------------------------------------------------------------------
def pow2_scale_ref(amax):
    """The block scale stated on its own: the smallest power of two P with fl32(amax / 448) <= P,
    clamped below at 2^-126; 1 for amax == 0 (float64 search over exponents)."""
    if amax == 0:
        return 1.0
    q = float(np.float32(np.float32(amax) / np.float32(448.0)))
    e = -126
    while 2.0 ** e < q:
        e += 1
    return 2.0 ** e


def pin_pow2_block_scale(O, seed=59):
    """Powers of two times 448 (exact ratios), their neighbours, tiny and huge magnitudes, random ones."""
    rng = np.random.default_rng(seed)
    vals = [0.0, 448.0, 224.0, 896.0, 1.0, 3.0e38, 1e-30, 1e-40]
    for e in range(-20, 21, 5):
        v = np.float32(448.0 * 2.0 ** e)
        vals += [float(v), float(np.nextafter(v, np.float32(np.inf))), float(np.nextafter(v, np.float32(0)))]
    vals += list(np.exp(rng.uniform(-60, 60, 40)).astype(np.float32).astype(float))
    for a in vals:
        a32 = float(np.float32(a))
        assert O.pow2_block_scale(a32) == pow2_scale_ref(a32), a32


def block_quantise_ref(O, vals, B=128):
    """Rows of float values quantised in consecutive blocks of B: the pinned scale rule per block,
    the pinned E4M3 encoder on value / scale."""
    R, C = vals.shape
    q = np.empty((R, C), np.uint8)
    sc = np.empty((R, C // B))
    for r in range(R):
        for b in range(C // B):
            blk = vals[r, b * B:(b + 1) * B]
            P = pow2_scale_ref(float(np.abs(blk).max()))
            sc[r, b] = P
            q[r, b * B:(b + 1) * B] = O.e4m3_encode((blk.astype(np.float32) * np.float32(1.0 / P)).astype(np.float32))
    return q, sc


def pin_quantize_fp8b(O, seed=61):
    """Row blocks and weight blocks against the block rule stated with numpy: each 128-wide block of
    a row (each 128 x 128 block of a weight matrix) gets its own power-of-two scale; codes are the
    encoder's on value / scale; a zero block gets scale 1; dequantised values are within half a
    quantum."""
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((6, 384)).astype(np.float32)
    a[:, 128:256] *= 1000.0   # blocks of very different magnitude in one row
    a[2, 256:] = 0.0          # a zero block
    a[3, :128] *= 1e-20
    bits = f32_to_bf16_bits(a)
    af = bf16_bits_to_f32(bits)
    q, sc = O.quantize_rows_fp8b(bits)
    rq, rsc = block_quantise_ref(O, af)
    assert np.array_equal(q, rq) and np.array_equal(sc.astype(np.float64), rsc)
    tab = e4m3_table()
    rec = tab[q] * np.repeat(sc.astype(np.float64), 128, axis=1)
    bound = np.maximum(np.abs(af) * 2.0 ** -4, 2.0 ** -10 * np.repeat(sc, 128, axis=1)) * (1 + 1e-6)
    assert np.all(np.abs(rec - af) <= bound)
    # weights: W [E, K, N] -> codes [E, N, K], scales [E, N/128, K/128]
    W = (0.05 * rng.standard_normal((2, 256, 384))).astype(np.float32)
    W[1, :128, 128:256] *= 64.0
    wbits = f32_to_bf16_bits(W)
    wf = bf16_bits_to_f32(wbits)
    wq, wsc = O.quantize_weights_fp8b(wbits)
    assert wq.shape == (2, 384, 256) and wsc.shape == (2, 3, 2)
    for e in range(2):
        for bn in range(3):
            for bk in range(2):
                blk = wf[e, bk * 128:(bk + 1) * 128, bn * 128:(bn + 1) * 128].T  # [n, k]
                P = pow2_scale_ref(float(np.abs(blk).max()))
                assert wsc[e, bn, bk] == P
                codes = O.e4m3_encode((blk.astype(np.float32) * np.float32(1.0 / P)).astype(np.float32))
                assert np.array_equal(wq[e, bn * 128:(bn + 1) * 128, bk * 128:(bk + 1) * 128], codes)


def pin_fp8b_forward(O, seed=67):
    """The blockwise FP8 layer against a float64 statement built from dequantised operands (codes
    times their block scales), h rounded to bf16 and requantised in 128-wide blocks, slot-ordered
    combine."""
    rng = np.random.default_rng(seed)
    T, d, f, E, k = 7, 256, 384, 3, 2
    logits, x_bits, wgu, wd = random_layer(rng, T, d, f, E)
    # Give every 128 x 128 weight block (and every 128-wide x block) its own magnitude, so that the
    # block scales differ and a wrongly indexed scale changes the result.
    def spread(bits, axes, lo=-6, hi=6):
        v = bf16_bits_to_f32(bits).astype(np.float32)
        for ax in axes:
            fac = (2.0 ** rng.integers(lo, hi, v.shape[ax] // 128)).repeat(128).astype(np.float32)
            shape = [1] * v.ndim
            shape[ax] = -1
            v = v * fac.reshape(shape)
        return f32_to_bf16_bits(v)
    wgu, wd, x_bits = spread(wgu, (1, 2)), spread(wd, (1, 2)), spread(x_bits, (1,), -3, 3)
    wgu8, sgu = O.quantize_weights_fp8b(wgu)   # [E, 2f, d], [E, 2f/128, d/128]
    wd8, sdn = O.quantize_weights_fp8b(wd)     # [E, d, f], [E, d/128, f/128]
    assert len(np.unique(sgu)) > 4 and len(np.unique(sdn)) > 2
    out = O.forward_fp8b(x_bits, logits, wgu8, sgu, wd8, sdn, k)
    idx, w = O.route(logits, k)
    tab = e4m3_table()

    def deq_w(codes, sc):  # [N, K] codes, [N/128, K/128] scales
        return tab[codes] * np.kron(sc.astype(np.float64), np.ones((128, 128)))

    ref = np.zeros((T, d))
    for t in range(T):
        x8, sx = O.quantize_rows_fp8b(x_bits[t:t + 1])
        xd = tab[x8[0]] * np.repeat(sx[0].astype(np.float64), 128)
        for j in range(k):
            e = idx[t, j]
            gu = deq_w(wgu8[e], sgu[e]) @ xd
            g, u = gu[:f], gu[f:]
            hb = f32_to_bf16_bits((g / (1 + np.exp(-g)) * u).astype(np.float32))[None, :]
            h8, sh = O.quantize_rows_fp8b(hb)
            hd = tab[h8[0]] * np.repeat(sh[0].astype(np.float64), 128)
            ref[t] += w[t, j] * (deq_w(wd8[e], sdn[e]) @ hd)
    err = np.abs(out - ref).max()
    assert err <= 2e-3 * np.abs(ref).max(), err


def pin_fp8b_stages(O, seed=71):
    """The blockwise FP8 stage functions composed in the layer's order give its output exactly."""
    rng = np.random.default_rng(seed)
    T, d, f, E, k = 9, 256, 256, 4, 2
    logits, x_bits, wgu, wd = random_layer(rng, T, d, f, E)
    logits[:, 1] = -30.0  # expert 1 never chosen: an empty segment
    wgu8, sgu = O.quantize_weights_fp8b(wgu)
    wd8, sdn = O.quantize_weights_fp8b(wd)
    out = O.forward_fp8b(x_bits, logits, wgu8, sgu, wd8, sdn, k)
    idx, w = O.route(logits, k)
    counts, offsets, src, dest = O.permute(idx, E)
    x8, sx = O.quantize_rows_fp8b(x_bits[src])
    h = O.gateup_swiglu_fp8b(x8, sx, offsets, wgu8, sgu)
    h8, sh = O.quantize_rows_fp8b(h)
    y = O.down_fp8b(h8, sh, offsets, wd8, sdn)
    assert np.array_equal(O.combine(y, w, dest), out)


ALL_PINS = [pin_hand_example, pin_brute_force, pin_dense_e1_k1, pin_route_library, pin_route_nan_order,
            pin_permute_library, pin_invariants, pin_stages, pin_grouped_hand_example,
            pin_grouped_reduces_to_topk, pin_grouped_brute_force, pin_grouped_invariants,
            pin_e4m3_decode_table, pin_e4m3_encode_rne, pin_quantize_rows_fp8, pin_fp8_forward,
            pin_fp8_stages, pin_pow2_block_scale, pin_quantize_fp8b, pin_fp8b_forward, pin_fp8b_stages]
