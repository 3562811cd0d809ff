"""libmoe.so without a GPU: it loads, exports every symbol include/moe.h declares, and rejects
bad arguments with the documented codes before making any CUDA call.  CPU only."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_grouped_fp32_gb300 import build, moe
    if not os.path.exists(moe.LIB_PATH):
        build.build()
    return moe.load()


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)


def test_header_declares_the_stage_calls():
    names = set(declared_symbols())
    for n in ["moe_route", "moe_permute", "moe_grouped_gemm_gateup_swiglu", "moe_grouped_gemm_down",
              "moe_combine", "moe_forward"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_version_and_launch_count(lib):
    assert lib.moe_version() >= 100
    assert lib.moe_forward_launch_count(32, 8, 2) == 4       # route+permute fused
    assert lib.moe_forward_launch_count(1024, 8, 2) == 4     # T*E = 8192
    assert lib.moe_forward_launch_count(1025, 8, 2) == 5
    assert lib.moe_forward_launch_count(4096, 8, 2) == 5
    assert lib.moe_forward_launch_count(2048, 256, 8) == 5   # E > 32
    assert lib.moe_forward_launch_count(0, 8, 2) == 0
    assert lib.moe_forward_launch_count(4, 8, 9) == -1
    os.environ["MOE_FUSE_ROUTE_PERMUTE"] = "0"
    try:
        assert lib.moe_forward_launch_count(32, 8, 2) == 5
    finally:
        del os.environ["MOE_FUSE_ROUTE_PERMUTE"]
    os.environ["MOE_FOLD_COMBINE"] = "1"  # the combine folded into the down GEMM: one launch fewer
    try:
        assert lib.moe_forward_launch_count(32, 8, 2) == 3 and lib.moe_forward_launch_count(4096, 8, 2) == 4
        assert lib.moe_forward_fp8_launch_count(32, 8, 2) == 4
    finally:
        del os.environ["MOE_FOLD_COMBINE"]


def _err(lib):
    return lib.moe_last_error_string().decode()


def test_workspace_layout_matches_the_documented_order(lib):
    from mixture_experts_grouped_fp32_gb300 import moe
    T, d, f, E, k = 300, 512, 768, 8, 2
    L = moe.workspace_layout(T, d, f, E, k)
    M = T * k

    def up(v):
        return (v + 255) // 256 * 256

    S = moe.down_ksplit(T, d, f, E, k)
    assert 1 <= S <= 8
    expect, o = {}, 0
    for name, nbytes in [("status", 256), ("idx", M * 4), ("w", M * 4), ("counts", E * 4),
                         ("offsets", (E + 1) * 4), ("src", M * 4), ("dest", M * 4),
                         ("x_perm", M * d * 2), ("h", M * f * 2), ("y_perm", S * M * d * 4)]:
        expect[name] = o
        o = up(o + nbytes)
    o = up(o + T * (d // 64) * 4)  # the combine-fold counters, one per token and 64 output columns
    expect["total"] = o
    assert L == expect
    assert moe.workspace_size(T, d, f, E, k) == o
    assert moe.workspace_size(T, 100, f, E, k) == 0  # invalid shape


@pytest.mark.parametrize("args,fragment", [
    ((-1, 64, 128, 8, 2), "T = -1"),
    ((4, 64, 128, 0, 1), "E = 0"),
    ((4, 64, 128, 257, 2), "E = 257"),
    ((4, 64, 128, 8, 9), "top_k = 9"),
    ((4, 64, 128, 4, 5), "top_k = 5"),
    ((4, 96, 128, 8, 2), "d = 96"),
    ((4, 64, 100, 8, 2), "f = 100"),
])
def test_forward_rejects_bad_shapes(lib, args, fragment):
    T, d, f, E, k = args
    p = ctypes.c_void_p(1 << 20)
    rc = lib.moe_forward(p, p, p, p, T, d, f, E, k, p, p, 1 << 40, None)
    assert rc == -1
    assert fragment in _err(lib)


def test_forward_rejects_null_and_small_workspace(lib):
    p = ctypes.c_void_p(1 << 20)
    assert lib.moe_forward(None, p, p, p, 4, 64, 128, 8, 2, p, p, 1 << 40, None) == -1
    assert lib.moe_forward(p, p, p, p, 4, 64, 128, 8, 2, p, p, 16, None) == -3
    assert "workspace" in _err(lib)
    assert lib.moe_forward(p, p, p, p, 4, 64, 128, 8, 2, p, ctypes.c_void_p((1 << 20) + 16), 1 << 40,
                           None) == -3
    assert lib.moe_forward(p, p, ctypes.c_void_p((1 << 20) + 2), p, 4, 64, 128, 8, 2, p, p, 1 << 40,
                           None) == -1


def test_forward_host_batches_validates(lib):
    p = ctypes.c_void_p(1 << 20)
    arr = (ctypes.c_void_p * 2)(1 << 20, 1 << 21)
    nul = (ctypes.c_void_p * 2)(1 << 20, None)
    f = lib.moe_forward_host_batches
    assert f(arr, arr, p, p, 0, 4, 64, 128, 8, 2, arr, p, 1 << 40, None, None, None) == 0   # no batches
    assert f(arr, arr, p, p, 2, 0, 64, 128, 8, 2, arr, p, 1 << 40, None, None, None) == 0   # T = 0
    assert f(arr, arr, p, p, -1, 4, 64, 128, 8, 2, arr, p, 1 << 40, None, None, None) == -1
    assert f(None, arr, p, p, 2, 4, 64, 128, 8, 2, arr, p, 1 << 40, None, None, None) == -1
    assert f(arr, nul, p, p, 2, 4, 64, 128, 8, 2, arr, p, 1 << 40, None, None, None) == -1
    assert "batch 1" in _err(lib)
    need = lib.moe_workspace_size(4, 64, 128, 8, 2) + 2 * lib.moe_host_staging_size(4, 64, 8)
    assert f(arr, arr, p, p, 2, 4, 64, 128, 8, 2, arr, p, need - 1, None, None, None) == -3
    assert f(arr, arr, p, p, 2, 4, 64, 100, 8, 2, arr, p, 1 << 40, None, None, None) == -1   # f % 64


@pytest.mark.parametrize("sym", ["moe_forward_fp8_host_batches", "moe_forward_fp8b_host_batches"])
def test_forward_fp8_host_batches_validates(lib, sym):
    p = ctypes.c_void_p(1 << 20)
    arr = (ctypes.c_void_p * 2)(1 << 20, 1 << 21)
    f = getattr(lib, sym)
    assert f(arr, arr, p, p, p, p, 0, 4, 128, 128, 8, 2, arr, p, 1 << 40, None, None, None) == 0
    assert f(arr, arr, p, p, p, p, -1, 4, 128, 128, 8, 2, arr, p, 1 << 40, None, None, None) == -1
    assert f(arr, arr, p, None, p, p, 2, 4, 128, 128, 8, 2, arr, p, 1 << 40, None, None, None) == -1
    assert f(arr, arr, p, p, p, p, 2, 4, 64, 128, 8, 2, arr, p, 1 << 40, None, None, None) == -1    # d % 128
    assert f(arr, arr, p, p, p, p, 2, 4, 128, 128, 8, 2, arr, p, 4096, None, None, None) == -3
    assert "workspace" in _err(lib)


def test_forward_grouped_host_batches_validates(lib):
    p = ctypes.c_void_p(1 << 20)
    arr = (ctypes.c_void_p * 2)(1 << 20, 1 << 21)
    f = lib.moe_forward_grouped_host_batches
    assert f(arr, arr, p, p, p, 0, 4, 64, 128, 8, 2, 4, 2, 1.0, arr, p, 1 << 40, None, None, None) == 0
    assert f(arr, arr, None, p, p, 2, 4, 64, 128, 8, 2, 4, 2, 1.0, arr, p, 1 << 40, None, None, None) == -1  # bias
    assert f(arr, arr, p, p, p, 2, 4, 64, 128, 8, 2, 3, 2, 1.0, arr, p, 1 << 40, None, None, None) == -1  # 8 % 3
    g8 = lib.moe_forward_grouped_fp8b_host_batches
    assert g8(arr, arr, p, p, p, p, p, 2, 4, 128, 128, 8, 2, 4, 5, 1.0, arr, p, 1 << 40, None, None, None) == -1
    assert g8(arr, arr, p, p, p, p, p, 2, 4, 128, 128, 8, 2, 4, 2, 1.0, arr, p, 4096, None, None, None) == -3


def test_stage_calls_reject_bad_arguments(lib):
    p = ctypes.c_void_p(1 << 20)
    assert lib.moe_route(None, 4, 8, 2, p, p, None) == -1
    assert lib.moe_route(p, 4, 8, 0, p, p, None) == -1
    assert lib.moe_permute(p, None, 4, 64, 8, 2, p, p, p, p, p, None, None) == -1
    assert lib.moe_permute(p, ctypes.c_void_p((1 << 20) + 8), 4, 64, 8, 2, p, p, p, p, p, None, None) == -1
    assert lib.moe_grouped_gemm_gateup_swiglu(p, p, None, 8, 64, 128, 8, p, None, None) == -1
    assert lib.moe_grouped_gemm_gateup_swiglu(p, p, p, -1, 64, 128, 8, p, None, None) == -1
    assert lib.moe_grouped_gemm_down(p, p, p, 8, 64, 96, 8, 1, p, None, None) == -1
    assert lib.moe_grouped_gemm_down(p, p, p, 8, 64, 128, 8, 9, p, None, None) == -1
    assert "ksplit" in _err(lib)
    assert lib.moe_combine(p, p, p, 4, 64, 0, 1, p, None, None) == -1
    assert lib.moe_combine(p, p, p, 4, 64, 2, 0, p, None, None) == -1
    assert lib.moe_get_device_error(None, None) == -1


def test_grouped_router_rejects_bad_groups(lib):
    p = ctypes.c_void_p(1 << 20)
    f = ctypes.c_float
    assert lib.moe_route_grouped(p, None, 4, 256, 8, 8, 4, f(2.5), p, p, None) == -1   # null bias
    assert "bias" in _err(lib)
    assert lib.moe_route_grouped(p, p, 4, 256, 8, 7, 4, f(2.5), p, p, None) == -1      # 7 does not divide 256
    assert lib.moe_route_grouped(p, p, 4, 256, 8, 64, 4, f(2.5), p, p, None) == -1     # more than 32 groups
    assert lib.moe_route_grouped(p, p, 4, 256, 8, 8, 9, f(2.5), p, p, None) == -1      # topk_group > n_group
    assert lib.moe_route_grouped(p, p, 4, 16, 8, 8, 2, f(1.0), p, p, None) == -1       # k > 2 groups x 2
    assert "kept groups" in _err(lib)
    assert lib.moe_route_grouped(p, p, 4, 256, 8, 8, 4, f(0.0), p, p, None) == -1      # scale
    assert lib.moe_route_grouped(p, p, 0, 256, 8, 8, 4, f(2.5), p, p, None) == 0       # empty batch
    assert lib.moe_forward_grouped(p, p, p, p, p, 4, 64, 128, 16, 8, 8, 2, f(1.0), p, p, 1 << 40, None) == -1
    assert lib.moe_forward_grouped(p, p, p, p, p, 0, 64, 128, 256, 8, 8, 4, f(2.5), p, p, 1 << 40, None) == 0


def test_empty_batch_is_a_no_op(lib):
    # T = 0 (and M = 0) launch nothing and succeed, so they need no device.
    p = ctypes.c_void_p(1 << 20)
    assert lib.moe_forward(p, p, p, p, 0, 64, 128, 8, 2, p, p, 1 << 40, None) == 0
    assert lib.moe_route(p, 0, 8, 2, p, p, None) == 0
    assert lib.moe_permute(p, p, 0, 64, 8, 2, p, p, p, p, p, None, None) == 0
    assert lib.moe_grouped_gemm_down(p, p, p, 0, 64, 128, 8, 1, p, None, None) == 0
    assert lib.moe_combine(p, p, p, 0, 64, 2, 1, p, None, None) == 0


def test_binding_fails_loudly_without_the_library(tmp_path):
    from mixture_experts_grouped_fp32_gb300 import moe
    saved = moe._lib
    moe._lib = None
    try:
        with pytest.raises(RuntimeError, match="missing"):
            moe.load(str(tmp_path / "libmoe.so"))
    finally:
        moe._lib = saved


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "mixture_experts_grouped_fp32_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in text and "from oracle" not in text, fn
                assert "liboracle" not in text and "moe_oracle" not in text, fn


def test_down_ksplit_policy(lib):
    """Few tokens -> the down projection is split over K; many tokens -> no split; never an empty
    slice; the environment override is honoured and clamped."""
    from mixture_experts_grouped_fp32_gb300 import moe
    assert moe.down_ksplit(32, 4096, 14336, 8, 2) == 1
    assert moe.down_ksplit(512, 4096, 14336, 8, 2) == 1  # SM-pair kernel: unsplit
    assert moe.down_ksplit(256, 4096, 14336, 8, 2) == 2  # 1-SM kernel, 1-2 waves of items
    assert moe.down_ksplit(4096, 4096, 14336, 8, 2) == 1
    assert moe.down_ksplit(2048, 7168, 2048, 256, 8) == 1
    for T, d, f, E, k in [(1, 64, 64, 8, 2), (64, 256, 512, 8, 2), (37, 192, 320, 4, 4), (512, 4096, 14336, 8, 2)]:
        S = moe.down_ksplit(T, d, f, E, k)
        nkb = f // 64
        per = -(-nkb // S)
        assert 1 <= S <= min(8, nkb) and (S - 1) * per < nkb
    os.environ["MOE_DOWN_KSPLIT"] = "3"
    try:
        assert moe.down_ksplit(4096, 4096, 14336, 8, 2) == 3
        assert moe.down_ksplit(4, 64, 128, 8, 2) == 2  # clamped to f/64 = 2 K blocks
    finally:
        del os.environ["MOE_DOWN_KSPLIT"]


def test_gemm_pair_mode_policy(lib):
    from mixture_experts_grouped_fp32_gb300 import moe
    mx = (4096, 14336)  # Mixtral-8x7B-shaped d, f
    for kind, big in ((0, 2), (1, 1)):
        assert moe.gemm_pair_mode(4096, *mx, 8, 2, kind) == big   # 1024 rows per expert on average
        assert moe.gemm_pair_mode(512, *mx, 8, 2, kind) == big    # 128
        assert moe.gemm_pair_mode(32, *mx, 8, 2, kind) == 0       # 8
        assert moe.gemm_pair_mode(4, *mx, 8, 9, kind) == -1
        assert moe.gemm_pair_mode(256, 7168, 2048, 32, 8, kind) == 0   # 64 rows, few slots
        assert moe.gemm_pair_mode(2048, 7168, 2048, 256, 8, kind) == 2  # 64 rows, many slots
        assert moe.gemm_pair_mode(1000, 7168, 2048, 256, 8, kind) == 0  # 31.25 rows
    assert moe.gemm_pair_mode(512, *mx, 8, 2, 2) == -1
    os.environ["MOE_GEMM_2SM_DOWN"] = "0"
    try:
        assert moe.gemm_pair_mode(4096, *mx, 8, 2, 1) == 0 and moe.gemm_pair_mode(4096, *mx, 8, 2, 0) == 2
    finally:
        del os.environ["MOE_GEMM_2SM_DOWN"]


def test_fp8_workspace_layout_and_validation(lib):
    from mixture_experts_grouped_fp32_gb300 import moe
    T, d, f, E, k = 300, 512, 768, 8, 2
    L = moe.workspace_layout_fp8(T, d, f, E, k)
    M = T * k

    def up(v):
        return (v + 255) // 256 * 256

    S = moe.down_ksplit_fp8(T, d, f, E, k)
    assert 1 <= S <= 8
    expect, o = {}, 0
    for name, nbytes in [("status", 256), ("idx", M * 4), ("w", M * 4), ("counts", E * 4),
                         ("offsets", (E + 1) * 4), ("src", M * 4), ("dest", M * 4), ("x8", M * d),
                         ("sx", M * 4), ("h", M * f * 2), ("h8", M * f), ("sh", M * 4),
                         ("y_perm", S * M * d * 4)]:
        expect[name] = o
        o = up(o + nbytes)
    o = up(o + T * (d // 64) * 4)  # the combine-fold counters
    expect["total"] = o
    assert L == expect
    assert moe.workspace_size_fp8(T, d, f, E, k) == o
    assert moe.workspace_size_fp8(T, 192, f, E, k) == 0       # d not a multiple of 128
    assert lib.moe_forward_fp8_launch_count(32, 8, 2) == 5
    assert lib.moe_forward_fp8_launch_count(2048, 256, 8) == 6
    assert lib.moe_forward_fp8_launch_count(0, 8, 2) == 0
    p = ctypes.c_void_p(1 << 20)
    assert lib.moe_forward_fp8(p, p, p, p, p, p, 4, 192, 256, 8, 2, p, p, 1 << 40, None) == -1
    assert "multiples of 128" in _err(lib)
    assert lib.moe_forward_fp8(p, p, None, p, p, p, 4, 256, 256, 8, 2, p, p, 1 << 40, None) == -1
    assert lib.moe_forward_fp8(p, p, p, p, p, p, 4, 256, 256, 8, 2, p, p, 16, None) == -3
    assert lib.moe_forward_fp8(p, p, p, p, p, p, 0, 256, 256, 8, 2, p, p, 1 << 40, None) == 0
    assert lib.moe_quantize_weights_fp8(p, 8, 192, 256, p, p, None) == -1        # K % 128
    assert lib.moe_quantize_weights_fp8(None, 8, 256, 256, p, p, None) == -1
    assert lib.moe_quantize_rows_fp8(p, None, 4, 12, 4, p, p, None, None) == -1   # C % 8
    assert lib.moe_quantize_rows_fp8(p, None, 4, 64, 3, p, p, None, None) == -1   # src_rows < R, no src
    assert lib.moe_quantize_rows_fp8(p, None, 0, 64, 0, p, p, None, None) == 0    # nothing to do
    assert lib.moe_grouped_gemm_gateup_swiglu_fp8(p, None, p, p, p, 8, 256, 256, 8, p, None, None) == -1
    assert lib.moe_grouped_gemm_down_fp8(p, p, p, p, p, 8, 256, 256, 8, 9, p, None, None) == -1
    assert lib.moe_grouped_gemm_down_fp8(p, p, p, p, p, 0, 256, 256, 8, 1, p, None, None) == 0


def test_fp8_block_layout_round_trip():
    """The blocked FP8 weight layout helpers are inverse index permutations, and the block of
    (n, k) is at [n // 64][k // 128][n % 64][k % 128]."""
    import numpy as np
    import torch
    from mixture_experts_grouped_fp32_gb300.moe import fp8_block, fp8_unblock
    a = np.random.default_rng(0).integers(0, 255, (3, 192, 256), dtype=np.uint8)
    b = fp8_block(a)
    assert b.shape == (3, 3, 2, 64, 128)
    assert np.array_equal(fp8_unblock(b), a)
    for e, n, k in [(0, 0, 0), (1, 65, 130), (2, 191, 255)]:
        assert b[e, n // 64, k // 128, n % 64, k % 128] == a[e, n, k]
    t = torch.from_numpy(a)
    assert torch.equal(fp8_unblock(fp8_block(t)), t)
    assert np.array_equal(fp8_block(t).numpy(), b)


def test_gemm_pair_mode_fp8_policy(lib):
    for v in ("MOE_GEMM_2SM", "MOE_GEMM_2SM_DOWN"):
        os.environ.pop(v, None)
    f = lib.moe_gemm_pair_mode_fp8
    assert f(32, 4096, 14336, 8, 2, 0) == 0 and f(32, 4096, 14336, 8, 2, 1) == 0       # Mixtral, T=32
    assert f(512, 4096, 14336, 8, 2, 0) == 2 and f(512, 4096, 14336, 8, 2, 1) == 1     # 128 rows per expert
    assert f(4096, 4096, 14336, 8, 2, 0) == 2 and f(4096, 4096, 14336, 8, 2, 1) == 1   # 1024 rows per expert
    assert f(2048, 7168, 2048, 256, 8, 0) == 2 and f(2048, 7168, 2048, 256, 8, 1) == 0  # DeepSeek-V3 shape
    assert f(256, 7168, 2048, 32, 8, 0) == 0 and f(256, 7168, 2048, 32, 8, 1) == 0     # 32 experts
    assert f(32, 4096, 14336, 8, 2, 2) == -1 and f(32, 4000, 14336, 8, 2, 0) == -1


def test_fp8b_quantised_h_policy(lib, monkeypatch):
    monkeypatch.delenv("MOE_FP8B_FUSE_H", raising=False)
    f = lib.moe_fp8b_gemm_quantizes_h
    assert f(32, 8, 2) == 0 and f(256, 8, 2) == 0        # 8 / 64 rows per expert on average
    assert f(512, 8, 2) == 1 and f(4096, 8, 2) == 1      # 128 / 1024
    assert f(2048, 256, 8) == 0                          # DeepSeek-V3 shape: 64
    assert f(4, 8, 9) == -1
    assert lib.moe_forward_fp8b_launch_count(4096, 8, 2) == 6 and lib.moe_forward_fp8b_launch_count(2048, 256, 8) == 7
    monkeypatch.setenv("MOE_FP8B_FUSE_H", "1")
    assert f(32, 8, 2) == 1 and lib.moe_forward_fp8b_launch_count(32, 8, 2) == 5
    monkeypatch.setenv("MOE_FP8B_FUSE_H", "0")
    assert f(4096, 8, 2) == 0


def test_fp8b_entry_points_validate(lib):
    from mixture_experts_grouped_fp32_gb300 import moe
    T, d, f, E, k = 300, 512, 768, 8, 2
    L = moe.workspace_layout_fp8b(T, d, f, E, k)
    M = T * k
    assert L["sh"] - L["h8"] >= M * f and L["y_perm"] - L["sh"] >= M * (f // 128) * 4
    assert L["h"] - L["sx"] >= M * (d // 128) * 4
    assert moe.workspace_size_fp8b(T, d, f, E, k) == L["total"]
    assert moe.down_ksplit_fp8b(T, d, f, E, k) >= 1
    assert lib.moe_forward_fp8b_launch_count(32, 8, 2) == 6      # h quantised by its own launch
    assert lib.moe_forward_fp8b_launch_count(512, 8, 2) == 5     # h quantised in the gate+up GEMM
    p = ctypes.c_void_p(1 << 20)
    assert lib.moe_quantize_weights_fp8b(p, 8, 256, 192, p, p, None) == -1      # N % 128
    assert lib.moe_quantize_rows_fp8b(p, None, 4, 64, 4, p, p, None, None) == -1  # C % 128
    assert lib.moe_forward_fp8b(p, p, p, p, p, p, 4, 192, 256, 8, 2, p, p, 1 << 40, None) == -1
    assert lib.moe_forward_fp8b(p, p, p, p, p, p, 4, 256, 256, 8, 2, p, p, 16, None) == -3
    assert lib.moe_grouped_gemm_down_fp8b(p, p, p, p, p, 0, 256, 256, 8, 1, p, None, None) == 0
