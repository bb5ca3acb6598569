"""Writes the stored oracle fixtures in this folder.

Calls only the float64 oracle (and the seeded input generators); no value here
ever comes from the CUDA library.  Run from the repository root:

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import muon_ref as R  # noqa: E402
from newton_schulz_gb300 import synth  # noqa: E402


def c1_summary():
    groups = synth.config_c1_numpy()
    outs = R.muon_step_groups_ref(groups, mu=0.95, nesterov=True, lr=0.02, wd=0.01)
    doc = {"source": "oracle.muon_step_ref on synth.config_c1_numpy(); mu=0.95 nesterov, "
                     "lr=0.02, wd=0.01, 5 steps (3.4445,-4.7750,2.0315), eps=1e-7, "
                     "scale sqrt(max(1,rows/cols))",
           "groups": []}
    for w2, m2, o in outs:
        doc["groups"].append({
            "shape": list(w2.shape),
            "O_fro": [float(np.linalg.norm(o[i])) for i in range(o.shape[0])],
            "W_fro": [float(np.linalg.norm(w2[i])) for i in range(w2.shape[0])],
            "O_head": [o[i].ravel()[:4].tolist() for i in range(o.shape[0])],
        })
    with open(os.path.join(HERE, "c1_oracle_summary.json"), "w") as f:
        json.dump(doc, f, indent=1)


if __name__ == "__main__":
    c1_summary()
