"""Writes tests/golden/c1.json from the seeded c1 input and the fp64 oracle.

Only synth/ (inputs) and oracle/ (expected values) are called; nothing here
comes from the CUDA library.  Run from the repository root:
    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402


def main():
    g = synth.c1().grads[0]
    O = oracle.newton_schulz(g.double().numpy(), 5)
    sv = np.linalg.svd(O, compute_uv=False)
    out = {
        "what": "c1: one 128x256 fp32 matrix N(0,1) from torch seed 0; quintic (3.4445,-4.7750,2.0315), 5 steps",
        "source": "fp64 oracle (oracle/ns_oracle.py), Muon update rule of the DMuon technical summary §1",
        "input_sha256": synth.sha256_of(g),
        "steps": 5,
        "O_fro": float(np.linalg.norm(O)),
        "O_first8": [float(v) for v in O.ravel()[:8]],
        "O_sigma_min": float(sv.min()),
        "O_sigma_max": float(sv.max()),
    }
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "c1.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
