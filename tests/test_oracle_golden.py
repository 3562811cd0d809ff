"""The oracle still reproduces its recorded outputs (tests/golden/oracle_small.json, written by
tests/golden/make_golden.py from the oracle alone).  A regression record across hosts and
compilers, not a pin."""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))


def test_oracle_matches_recorded_outputs():
    import make_golden
    rec = json.load(open(os.path.join(HERE, "golden", "oracle_small.json")))
    now = make_golden.compute()
    for key in ("idx", "counts", "offsets", "src", "dest"):
        assert now[key] == rec[key], key
    np.testing.assert_allclose(now["w"], rec["w"], rtol=1e-6, atol=0)
    np.testing.assert_allclose(now["out"], rec["out"], rtol=1e-5, atol=1e-6)
