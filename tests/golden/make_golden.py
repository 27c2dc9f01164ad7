"""Writes the stored expected values under tests/golden/ by calling only the
oracle (and the seeded input generator).  Re-run after a change to the oracle
that a cited passage justifies:  python tests/golden/make_golden.py"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synthetic as syn  # noqa: E402


def tiny_case():
    """B=2, T=12, d_h=8 rectangular batch and a 4-segment pack (N=12)."""
    w = syn.small_workload(B=2, T=12, d_in=4, d_h=8, seed=101)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    out = {
        "source": "oracle/nrnn_oracle.c via tests/golden/make_golden.py; cell of "
                  "ParaGRU(mix='diag'), Newton+scan per the pararnn-torch numerics contract",
        "P": P.tolist(),
        "params": {k: v.tolist() for k, v in prm.items()},
        "sequential": oracle.sequential(P, prm).tolist(),
        "newton": {},
    }
    for K in (0, 1, 2, 3):
        H, rho = oracle.newton(P, prm, K)
        out["newton"][str(K)] = {"H": H.tolist(), "rho": rho}
    cu = syn.cu_from_lengths([5, 0, 4, 3])
    Pp = P[:1]
    out["pack"] = {"cu_seqlens": cu.tolist(),
                   "sequential": oracle.sequential(Pp, prm, cu_seqlens=cu).tolist(),
                   "newton3": oracle.newton(Pp, prm, 3, cu_seqlens=cu)[0].tolist()}
    return out


if __name__ == "__main__":
    with open(os.path.join(HERE, "tiny_newton.json"), "w") as fh:
        json.dump(tiny_case(), fh, indent=1)
    print("wrote tiny_newton.json")
