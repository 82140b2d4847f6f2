"""Writes the stored expected values under tests/golden/ (calls only the oracle).

Run from the repository root:  python tests/golden/make_golden.py
The inputs are the seeded CPU draws of the tiny workload (T=256, H=256, E=8,
I=512, top-2 softmax router, all tensors ~N(0, 0.02), dY ~N(0, 1), seed 0).
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from mixture_experts_layer_table_gb300 import workloads as W  # noqa: E402  (seeded draws only)
from oracle import moe_oracle as O  # noqa: E402


def main():
    shp = W.TINY
    inp = W.make_inputs(shp, seed=0, device="cpu")
    f64 = {k: (v.double().numpy() if v is not None else None) for k, v in inp.items()}
    fwd = O.forward(f64["x"], f64["w_router"], f64["w13"], f64["w2"], kind=shp.router,
                    k=shp.k, renorm=shp.renorm)
    bwd = O.backward(fwd, f64["dy"], f64["x"], f64["w_router"], f64["w13"], f64["w2"],
                     kind=shp.router, k=shp.k, renorm=shp.renorm)
    rows = [0, 1, 77, 255]
    out = {
        "workload": shp.name,
        "seed": 0,
        "counts": fwd["counts"].tolist(),
        "topk_idx_rows": {str(t): fwd["topk_idx"][t].tolist() for t in rows},
        "y_rows_first8": {str(t): fwd["y"][t, :8].tolist() for t in rows},
        "y_fro": float(np.linalg.norm(fwd["y"])),
        "dx_fro": float(np.linalg.norm(bwd["dx"])),
        "dw13_fro": float(np.linalg.norm(bwd["dw13"])),
        "dw2_fro": float(np.linalg.norm(bwd["dw2"])),
        "dw_router_fro": float(np.linalg.norm(bwd["dw_router"])),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle_summary.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
