"""Failure detection on the GPU without a fault: a grouped-GEMM pipeline wait is made to run out
(the host arms one stage for bytes that never arrive, MOE_INJECT_STALL=1).  The kernel must give
up after its ~1 s limit, set MOE_STATUS_WAIT_TIMEOUT in the status word, free its tensor memory and
return — and the same process must then run the layer correctly."""
import os
import sys
import time

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
from gpu_cases import assert_close, random_bf16  # noqa: E402

from mixture_experts_grouped_fp32_gb300.workloads import Workload  # noqa: E402

pytestmark = pytest.mark.gpu


def _down_case():
    from mixture_experts_grouped_fp32_gb300.workloads import draw_routing, draw_weights
    from oracle import Oracle
    T, d, f, E, k = 300, 256, 512, 8, 2
    logits, _ = draw_routing(T, 64, E, 12)
    idx, _ = Oracle().route(logits.numpy(), k)
    _, offsets, _, _ = Oracle().permute(idx, E)
    h = random_bf16((T * k, f), seed=6, scale=0.5)
    _, wd = draw_weights(d, f, E, 4, "cpu")
    return offsets, h, wd, T * k, d


def test_expired_wait_reports_status_and_context_survives(monkeypatch, oracle):
    from mixture_experts_grouped_fp32_gb300 import moe
    offsets, h, wd, M, d = _down_case()
    dev = torch.device("cuda")
    offs, hd, wdd = torch.from_numpy(offsets).to(dev), h.to(dev), wd.to(dev)

    monkeypatch.setenv("MOE_INJECT_STALL", "1")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    y = torch.zeros(M, d, dtype=torch.float32, device=dev)
    t0 = time.time()
    moe.grouped_gemm_down(hd, wdd, offs, y_perm=y, status=status)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert int(status.item()) & moe.STATUS_WAIT_TIMEOUT
    assert 0.5 < elapsed < 20, elapsed

    monkeypatch.delenv("MOE_INJECT_STALL")
    status.zero_()
    y2 = moe.grouped_gemm_down(hd, wdd, offs, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.down(h.view(torch.int16).numpy().view(np.uint16), offsets,
                      wd.view(torch.int16).numpy().view(np.uint16))
    assert_close(y2.cpu().numpy(), ref, 1e-3, 1e-4, "down after an expired wait")
