"""moe_forward_noalloc: the layer for callers that cannot allocate device memory when they run it
(servers whose device memory is carved into fixed pools at start-up, plugins that cannot reach
their host framework's allocator, latency-critical paths that cannot afford a cudaMalloc).  It
keeps its intermediates in a fixed device array inside libmoe.so instead of a caller workspace.

Checked through the C ABI on two calls in a row with different inputs and shapes, so that a stale
or shared-scratch mistake shows: bit for bit against moe_forward (the same launches on the same
inputs are deterministic), and against the CPU oracle at the layer tolerance.  The array's status
word is read back through moe_get_device_error(NULL, ...), clean after a normal call and set after
a call whose pipeline wait was made to run out (the MOE_INJECT_STALL host hook; nothing faults).
This file is collected last; it builds its own inputs and needs no other test to run first.
"""
import ctypes
import os
import sys

import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
from gpu_cases import assert_layer_close, case_inputs  # noqa: E402

from mixture_experts_grouped_fp32_gb300.workloads import Workload, bf16_bits  # noqa: E402

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 * 1024 * 1024


def _noalloc(lib, x, logits, wgu, wd, k, out):
    T, d = x.shape
    E, _, f2 = wgu.shape
    return lib.moe_forward_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(logits.data_ptr()),
                                   ctypes.c_void_p(wgu.data_ptr()), ctypes.c_void_p(wd.data_ptr()),
                                   T, d, f2 // 2, E, k, ctypes.c_void_p(out.data_ptr()),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _noalloc_status(lib) -> int:
    code = ctypes.c_int32(-1)
    rc = lib.moe_get_device_error(None, ctypes.byref(code))
    assert rc == 0, lib.moe_last_error_string().decode()
    return int(code.value)


def test_noalloc_matches_forward_and_oracle_on_two_calls_in_a_row():
    from oracle import Oracle

    from mixture_experts_grouped_fp32_gb300 import moe
    lib = moe.load()
    dev = torch.device("cuda")
    cases = [Workload("noalloc_a", 300, 512, 768, 8, 2), Workload("noalloc_b", 77, 256, 384, 16, 4)]
    O = Oracle()
    for seed, w in enumerate(cases):
        logits, x, wgu, wd = case_inputs(w, seed=seed + 20)
        ref_cpu = O.forward(bf16_bits(x), logits.numpy(), bf16_bits(wgu), bf16_bits(wd), w.k)
        logits_d, x_d, wgu_d, wd_d = (t.to(dev) for t in (logits, x, wgu, wd))
        ref = moe.forward(x_d, logits_d, wgu_d, wd_d, w.k)
        out = torch.full_like(ref, float("nan"))
        rc = _noalloc(lib, x_d, logits_d, wgu_d, wd_d, w.k, out)
        assert rc == 0, lib.moe_last_error_string().decode()
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"{w.name}: noalloc output differs from moe_forward's"
        assert _noalloc_status(lib) == 0
        assert_layer_close(out.float().cpu().numpy(), ref_cpu, w.name + " vs oracle")


def test_noalloc_status_word_reports_an_expired_wait(monkeypatch):
    from mixture_experts_grouped_fp32_gb300 import moe
    lib = moe.load()
    dev = torch.device("cuda")
    w = Workload("noalloc_stall", 64, 256, 512, 8, 2)
    logits, x, wgu, wd = (t.to(dev) for t in case_inputs(w, seed=31))
    out = torch.empty(w.T, w.d, dtype=torch.bfloat16, device=dev)
    monkeypatch.setenv("MOE_INJECT_STALL", "1")
    assert _noalloc(lib, x, logits, wgu, wd, w.k, out) == 0, lib.moe_last_error_string().decode()
    torch.cuda.synchronize()
    assert _noalloc_status(lib) & moe.STATUS_WAIT_TIMEOUT
    monkeypatch.delenv("MOE_INJECT_STALL")
    assert _noalloc(lib, x, logits, wgu, wd, w.k, out) == 0, lib.moe_last_error_string().decode()
    torch.cuda.synchronize()
    assert _noalloc_status(lib) == 0  # the next call's first kernel clears it
    assert torch.equal(out, moe.forward(x, logits, wgu, wd, w.k))


def test_noalloc_rejects_shapes_beyond_its_scratch():
    from mixture_experts_grouped_fp32_gb300 import moe
    lib = moe.load()
    T, d, f, E, k = 4096, 4096, 14336, 8, 2
    assert moe.workspace_size(T, d, f, E, k) > SCRATCH_BYTES
    p = ctypes.c_void_p(1 << 20)
    rc = lib.moe_forward_noalloc(p, p, p, p, T, d, f, E, k, p, None)
    assert rc == -3
    assert "scratch" in lib.moe_last_error_string().decode()
