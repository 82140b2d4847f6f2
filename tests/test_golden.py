"""Stored expected values: the oracle against its committed summary, and host logic
against the numbers the pages print (CPU only)."""
import json
import os

import numpy as np

from mixture_experts_layer_table_gb300 import workloads as W
from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_tiny_oracle_summary_regression():
    with open(os.path.join(GOLDEN, "tiny_oracle_summary.json")) as f:
        ref = json.load(f)
    shp = W.TINY
    inp = W.make_inputs(shp, seed=0, device="cpu")
    f64 = {k: (v.double().numpy() if v is not None else None) for k, v in inp.items()}
    fwd = O.forward(f64["x"], f64["w_router"], f64["w13"], f64["w2"], kind=shp.router,
                    k=shp.k, renorm=shp.renorm)
    assert fwd["counts"].tolist() == ref["counts"]
    for t, idx in ref["topk_idx_rows"].items():
        assert fwd["topk_idx"][int(t)].tolist() == idx
    for t, vals in ref["y_rows_first8"].items():
        assert np.allclose(fwd["y"][int(t), :8], vals, rtol=1e-10, atol=0)
    assert np.isclose(np.linalg.norm(fwd["y"]), ref["y_fro"], rtol=1e-10)
    bwd = O.backward(fwd, f64["dy"], f64["x"], f64["w_router"], f64["w13"], f64["w2"],
                     kind=shp.router, k=shp.k, renorm=shp.renorm)
    for name in ("dx", "dw13", "dw2", "dw_router"):
        assert np.isclose(np.linalg.norm(bwd[name]), ref[name + "_fro"], rtol=1e-10), name
