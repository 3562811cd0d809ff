"""Plant plausible mistakes in a copy of the oracle and check that the pins catch every one.

Each mutant is a one-line textual edit of ``oracle/moe_oracle.cpp`` (a dropped term, a wrong
sign, index or operand), compiled to a temporary library and run through ``oracle_pins`` in a
child process.  A mutant that passes every pin would mean the pins cannot see that mistake.
CPU only; the real oracle is never modified.
"""
import json
import os
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.cpp")

MUTANTS = {
    "silu_sign": ("return z / (1.0f + std::exp(-z));", "return z / (1.0f + std::exp(z));"),
    "gate_reads_up": ("g[n] += xi * bf16_to_f32(wrow[n]);", "g[n] += xi * bf16_to_f32(wrow[f + n]);"),
    "swiglu_swapped": ("h[n] = silu(g[n]) * u[n];", "h[n] = silu(u[n]) * g[n];"),
    "down_transposed": ("y[m] += hn * bf16_to_f32(wrow[m]);",
                        "y[m] += hn * bf16_to_f32(Wd_e[static_cast<size_t>(m) * f + n]);"),
    "ties_to_higher_id": ("            return l[a] > l[b];\n        });",
                          "            return l[a] > l[b] || (l[a] == l[b] && a > b);\n        });"),
    "no_renormalise": ("w[static_cast<size_t>(t) * k + j] = p[order[j]] / s;",
                       "w[static_cast<size_t>(t) * k + j] = p[order[j]];"),
    "tokens_descending": ("const int r = cursor[e]++;",
                          "const int r = offsets[e + 1] - 1 - (cursor[e]++ - offsets[e]);"),
    "combine_drops_slot": ("const float wj = w[static_cast<size_t>(t) * k + j];",
                           "const float wj = (j + 1 < k) ? w[static_cast<size_t>(t) * k + j] : 0.0f;"),
    "combine_slot_mismatch": ("y + static_cast<size_t>(dest[static_cast<size_t>(t) * k + j]) * d;",
                              "y + static_cast<size_t>(dest[static_cast<size_t>(t) * k + (k - 1 - j)]) * d;"),
    "down_wrong_expert": ("const uint16_t* We = Wd + static_cast<size_t>(e) * f * d;\n#pragma omp parallel for",
                          "const uint16_t* We = Wd + static_cast<size_t>((e + 1) % E) * f * d;\n#pragma omp parallel for"),
    "gather_wrong_row": ("x + static_cast<size_t>(src[r]) * d,", "x + static_cast<size_t>(src[M - 1 - r]) * d,"),
    # the DeepSeek-V3 router
    "grouped_bias_in_weights": ("w[static_cast<size_t>(t) * k + j] = scale * (sc[eorder[j]] / ssum);",
                                "w[static_cast<size_t>(t) * k + j] = scale * (c[eorder[j]] / ssum);"),
    "grouped_no_bias": ("c[e] = sc[e] + bias[e];", "c[e] = sc[e];"),
    "grouped_top1_group_score": ("const int q = std::min(gs, std::max(1, k / topk_group));", "const int q = 1;"),
    "grouped_no_group_limit": ("for (int i = 0; i < topk_group; ++i) kept[gorder[i]] = 1;",
                               "for (int i = 0; i < n_group; ++i) kept[gorder[i]] = 1;"),
    "grouped_no_scale": ("= scale * (sc[eorder[j]] / ssum);", "= (sc[eorder[j]] / ssum);"),
    "grouped_group_ties_higher": ("return gscore[a] > gscore[b]; });",
                                  "return gscore[a] > gscore[b] || (gscore[a] == gscore[b] && a > b); });"),
    "grouped_affinity_sign": ("sc[e] = 1.0f / (1.0f + std::exp(-l[e]));", "sc[e] = 1.0f / (1.0f + std::exp(l[e]));"),
    # the FP8 variant
    "e4m3_ties_away": ("const double q = std::nearbyint(a / quantum);", "const double q = std::round(a / quantum);"),
    "e4m3_no_saturation": ("if (v > 448.0) v = 448.0;", "if (v > 480.0) v = 480.0;"),
    "fp8_row_scale_dropped": ("scale[r] = amax > 0.0f ? amax / 448.0f : 1.0f;", "scale[r] = 1.0f;"),
    "fp8_weight_scale_dropped": ("const float v = acc * (sx * se[n]);", "const float v = acc * sx;"),
    "fp8_h_unquantised": ("oracle_quantize_rows_fp8(hb.data(), 1, f, h8.data(), &sh);\n"
                          "            for (int n = 0; n < f; ++n) hd[n] = e4m3_decode(h8[n]);",
                          "oracle_quantize_rows_fp8(hb.data(), 1, f, h8.data(), &sh);\n"
                          "            for (int n = 0; n < f; ++n) hd[n] = bf16_to_f32(hb[n]) / sh;"),
    # the blockwise FP8 variant
    "fp8b_scale_rounds_down": ("const float p = (m == 0.5f) ? q : std::ldexp(1.0f, e);",
                               "const float p = (m == 0.5f) ? q : std::ldexp(1.0f, e - 1);"),
    "fp8b_weight_scale_transposed": ("acc += part * (sx[b] * se[static_cast<size_t>(n / 128) * nb + b]);",
                                     "acc += part * (sx[b] * se[static_cast<size_t>(b) * (2 * f / 128) + n / 128]);"),
    "fp8b_first_block_scale_only": ("acc += part * (sh[b] * sde[static_cast<size_t>(m / 128) * nb + b]);",
                                    "acc += part * (sh[0] * sde[static_cast<size_t>(m / 128) * nb + b]);"),
    "fp8b_weight_block_one_row": ("for (int n = bn * 128; n < (bn + 1) * 128; ++n)\n                    for (int k = bk * 128; k < (bk + 1) * 128; ++k)\n                        amax",
                                  "for (int n = bn * 128; n < bn * 128 + 1; ++n)\n                    for (int k = bk * 128; k < (bk + 1) * 128; ++k)\n                        amax"),
    "fp8b_block_absmax_half": ("for (int c = b * B; c < (b + 1) * B; ++c) amax",
                               "for (int c = b * B; c < b * B + B / 2; ++c) amax"),
}

_CHILD = textwrap.dedent("""
    import json, sys
    sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
    import oracle, oracle_pins
    O = oracle.Oracle(oracle.load_library({lib!r}))
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(O)
        except Exception as exc:  # AssertionError or a rejected input
            failed.append(pin.__name__)
    print(json.dumps(failed))
""")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor for {name} must occur exactly once"
    src = tmp_path / "mutant.cpp"
    src.write_text(text.replace(old, new))
    sys.path.insert(0, ROOT)
    import oracle
    lib = oracle.build(str(src), str(tmp_path / "libmutant.so"))
    code = _CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=lib)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    if res.returncode != 0:
        return  # the mutant crashed the pins' process: caught
    failed = json.loads(res.stdout.strip().splitlines()[-1])
    assert failed, f"mutant {name} passed every pin"
