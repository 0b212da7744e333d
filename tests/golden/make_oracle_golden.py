"""Writes tiny_oracle.json: the oracle's outputs on the tiny workload.

The pages print no worked example (their tables hold timings only), so no
stored value here comes from them.  This script calls only the oracle and the
seeded input generator; the values guard the oracle's own arithmetic against
unintended change.  Run from the repository root:

    python tests/golden/make_oracle_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from joint_attention_gb300.inputs import CONFIGS, make_config_inputs  # noqa: E402

ROWS = (0, 7, 8, 23)  # first and last caption row, first and last image row


def golden() -> dict:
    cfg = CONFIGS["tiny"]
    inp = make_config_inputs(cfg)
    ref = oracle.joint_attention_bwd(inp.q, inp.k, inp.v, inp.gq, inp.gk, inp.dout)
    out = {
        "workload": "tiny: B=1, H=2, N_img=16, N_txt=8, d=64, seed 0",
        "rows": list(ROWS),
        "LSE": ref["LSE"].tolist(),
        "dgq": ref["dgq"].tolist(),
        "dgk": ref["dgk"].tolist(),
        "norms": {key: float(np.linalg.norm(ref[key])) for key in ("O", "dq", "dk", "dv")},
    }
    for key in ("O", "dq", "dk", "dv"):
        out[key + "_rows"] = ref[key][:, :, list(ROWS), :].tolist()
    return out


if __name__ == "__main__":
    with open(os.path.join(HERE, "tiny_oracle.json"), "w") as f:
        json.dump(golden(), f, indent=None, separators=(",", ":"))
        f.write("\n")
