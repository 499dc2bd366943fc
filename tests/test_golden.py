"""Regression check of the oracle against the fixture that
tests/golden/make_golden.py wrote from the oracle alone (quickstart shape of
"Fast Attention Residuals", section "Quickstart: standard AttnRes")."""
import json
import os

import numpy as np

from attention_residuals_gb300.workloads import make_workload
from oracle import attnres_oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def test_quickstart_fixture():
    with open(os.path.join(HERE, "golden", "quickstart_oracle.json")) as f:
        doc = json.load(f)
    wl = make_workload(1)
    out = attnres_oracle(wl.values, wl.q, dy=wl.dy, key_offset=0, nthreads=2)
    np.testing.assert_allclose(out["alpha"], doc["alpha"], rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(out["rstd"], doc["rstd"], rtol=1e-14)
    np.testing.assert_allclose(out["logit"], doc["logit"], rtol=1e-12)
    np.testing.assert_allclose(out["y"][:, :16], doc["y_head"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(np.linalg.norm(out["y"]), doc["y_norm"], rtol=1e-12)
    np.testing.assert_allclose(out["dq"][:16], doc["dq_head"], rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(np.linalg.norm(out["dq"]), doc["dq_norm"], rtol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(out["dvalues"]), doc["dvalues_norm"], rtol=1e-12)
