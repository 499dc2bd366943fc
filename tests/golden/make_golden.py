"""Write tests/golden/quickstart_oracle.json from the FP64 oracle alone.

The input is the quickstart-shaped workload of "Fast Attention Residuals"
(section "Quickstart: standard AttnRes": values [8, 2, 1024], query [1024],
eps = 2^-23, scale = 1) drawn from the seeded generator.  The stored numbers
are the oracle's own; the file is a regression fixture that catches later
changes to the oracle's arithmetic.  Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

from attention_residuals_gb300.workloads import make_workload  # noqa: E402
from oracle import attnres_oracle  # noqa: E402


def main():
    wl = make_workload(1)
    out = attnres_oracle(wl.values, wl.q, dy=wl.dy, key_offset=0, nthreads=1)
    doc = {
        "source": "Fast Attention Residuals, Quickstart shape; values from the FP64 oracle",
        "workload": "make_workload(1): S=8 N=2 D=1024 R=1024 key_offset=0 eps=2^-23 scale=1",
        "alpha": out["alpha"].tolist(),
        "rstd": out["rstd"].tolist(),
        "logit": out["logit"].tolist(),
        "y_head": out["y"][:, :16].tolist(),
        "y_norm": float(np.linalg.norm(out["y"])),
        "dq_head": out["dq"][:16].tolist(),
        "dq_norm": float(np.linalg.norm(out["dq"])),
        "dvalues_norm": float(np.linalg.norm(out["dvalues"])),
        "dvalues_sum": float(out["dvalues"].sum()),
    }
    with open(os.path.join(HERE, "quickstart_oracle.json"), "w") as f:
        json.dump(doc, f, indent=1)


if __name__ == "__main__":
    main()
