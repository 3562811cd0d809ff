"""Write ``oracle_small.json``: the oracle's outputs on one small seeded layer.

This script calls only ``oracle/`` (and the seeded input generators).  The fixture is a
regression record, not a pin: it shows that the oracle built on another host (the x86 build
machine, the Arm GPU host) still computes what it computed when the fixture was written.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from mixture_experts_grouped_fp32_gb300.workloads import bf16_bits, draw_routing, draw_weights  # noqa: E402
from oracle import Oracle  # noqa: E402

CASE = dict(T=24, d=64, f=64, E=6, k=2, seed=17)


def compute():
    c = CASE
    logits, x = draw_routing(c["T"], c["d"], c["E"], c["seed"])
    wgu, wd = draw_weights(c["d"], c["f"], c["E"], c["seed"], "cpu")
    O = Oracle()
    idx, w = O.route(logits.numpy(), c["k"])
    counts, offsets, src, dest = O.permute(idx, c["E"])
    out = O.forward(bf16_bits(x), logits.numpy(), bf16_bits(wgu), bf16_bits(wd), c["k"])
    return dict(case=c, idx=idx.tolist(), w=[float(v) for v in w.reshape(-1)],
                counts=counts.tolist(), offsets=offsets.tolist(), src=src.tolist(),
                dest=dest.tolist(), out=[float(v) for v in out.reshape(-1)])


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_small.json"), "w") as fh:
        json.dump(compute(), fh)
    print("wrote oracle_small.json")
