"""The sampled-output checker of the full-size GPU tests, pinned on the CPU: it accepts the
oracle's own whole-layer output and rejects a row with one element moved or a wrong expert."""
import numpy as np
import pytest

from mixture_experts_layer_table_gb300 import workloads as W
from oracle import moe_oracle as O
from tests.parity import check_sampled_token_outputs, clear_margin_tokens


def _case():
    shp = W.MoEShape("helper_T64_H32_E8_I64_top2_sigmoid", T=64, H=32, E=8, I=64, k=2,
                     router=W.ROUTER_SIGMOID, renorm=True, x_std=1.0, w_std=0.2)
    rng = np.random.default_rng(3)
    x = rng.normal(0, 1, (shp.T, shp.H))
    w_r = rng.normal(0, 0.2, (shp.E, shp.H))
    w13 = rng.normal(0, 0.2, (shp.E, 2 * shp.I, shp.H))
    w2 = rng.normal(0, 0.2, (shp.E, shp.H, shp.I))
    f = O.forward(x, w_r, w13, w2, kind=shp.router, k=shp.k, renorm=shp.renorm)
    return shp, x, w_r, w13, w2, f


def test_checker_accepts_the_layer_output_and_rejects_errors():
    shp, x, w_r, w13, w2, f = _case()
    _, scores = O.router_scores(x, w_r, shp.router)
    toks = clear_margin_tokens(scores, shp.k, 6, seed=0)
    assert len(toks) == 6
    srt = -np.sort(-scores[toks], axis=1)
    assert np.all(srt[:, shp.k - 1] - srt[:, shp.k] > 1e-4)
    experts = lambda e: (w13[e], w2[e])
    args = (toks, x[toks], w_r, None, experts, shp)
    check_sampled_token_outputs(*args, f["y"][toks], f["topk_idx"][toks], "exact")
    bad = f["y"][toks].copy()
    bad[2, 5] += 0.5 * np.sqrt(np.mean(f["y"][toks] ** 2)) + 1.0
    with pytest.raises(AssertionError):
        check_sampled_token_outputs(*args, bad, f["topk_idx"][toks], "one element moved")
    idx = f["topk_idx"][toks].copy()
    idx[0] = idx[0][::-1]
    with pytest.raises(AssertionError):
        check_sampled_token_outputs(*args, f["y"][toks], idx, "experts swapped")
