"""moe_forward_noalloc: the layer for callers that cannot allocate device memory (graph-capture
code, pre-planned serving memory, plugins without access to an allocator).  It keeps its
intermediates in a fixed device array inside libmoe.so instead of a caller workspace.

Checked through the C ABI against moe_forward (the entry point with a caller workspace), on two
calls in a row with different inputs and shapes so that a stale or shared-scratch mistake shows.
This file is collected last; it builds its own inputs and needs no other test to run first.
"""
import ctypes
import os
import sys

import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
from gpu_cases import assert_layer_close, case_inputs  # noqa: E402

from mixture_experts_grouped_fp32_gb300.workloads import Workload  # noqa: E402

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 * 1024 * 1024


def _noalloc(lib, x, logits, wgu, wd, k, out):
    T, d = x.shape
    E, _, f2 = wgu.shape
    return lib.moe_forward_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(logits.data_ptr()),
                                   ctypes.c_void_p(wgu.data_ptr()), ctypes.c_void_p(wd.data_ptr()),
                                   T, d, f2 // 2, E, k, ctypes.c_void_p(out.data_ptr()),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_forward_on_two_calls_in_a_row():
    from mixture_experts_grouped_fp32_gb300 import moe
    lib = moe.load()
    lib.moe_forward_noalloc.restype = ctypes.c_int
    dev = torch.device("cuda")
    cases = [Workload("noalloc_a", 300, 512, 768, 8, 2), Workload("noalloc_b", 77, 256, 384, 16, 4)]
    for seed, w in enumerate(cases):
        logits, x, wgu, wd = (t.to(dev) for t in case_inputs(w, seed=seed + 20))
        ref = moe.forward(x, logits, wgu, wd, w.k)
        out = torch.full_like(ref, float("nan"))
        rc = _noalloc(lib, x, logits, wgu, wd, w.k, out)
        assert rc == 0, lib.moe_last_error_string().decode()
        torch.cuda.synchronize()
        assert_layer_close(out.float().cpu().numpy(), ref.float().cpu().numpy(), w.name)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    from mixture_experts_grouped_fp32_gb300 import moe
    lib = moe.load()
    T, d, f, E, k = 4096, 4096, 14336, 8, 2
    assert moe.workspace_size(T, d, f, E, k) > SCRATCH_BYTES
    p = ctypes.c_void_p(1 << 20)
    rc = lib.moe_forward_noalloc(p, p, p, p, T, d, f, E, k, p, None)
    assert rc == -3
    assert "scratch" in lib.moe_last_error_string().decode()
