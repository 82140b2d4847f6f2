"""The sampled-output checker of the full-size GPU tests, pinned on the CPU: it accepts the
oracle's own whole-layer output and rejects a row with one element moved or a wrong expert."""
import numpy as np
import pytest

from mixture_experts_layer_table_gb300 import workloads as W
from oracle import moe_oracle as O
from tests.parity import (check_sampled_expert_wgrads, check_sampled_token_backward, check_sampled_token_outputs,
                          clear_margin_tokens)


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


def _backward_case(quant=None):
    shp, x, w_r, w13, w2, _ = _case()
    rng = np.random.default_rng(4)
    dy = rng.normal(0, 1, (shp.T, shp.H))
    f = O.forward(x, w_r, w13, w2, kind=shp.router, k=shp.k, renorm=shp.renorm, quant=quant)
    b = O.backward(f, dy, x, w_r, w13, w2, kind=shp.router, k=shp.k, renorm=shp.renorm, quant=quant)
    return shp, x, w_r, w13, w2, dy, f, b


def test_token_backward_checker_accepts_the_layer_and_rejects_errors():
    shp, x, w_r, w13, w2, dy, f, b = _backward_case()
    _, scores = O.router_scores(x, w_r, shp.router)
    toks = clear_margin_tokens(scores, shp.k, 5, seed=1)
    experts = lambda e: (w13[e], w2[e])
    args = (toks, x[toks], dy[toks], w_r, None, experts, shp)
    dx, dg, idx = b["dx"][toks], b["dgates"][toks], f["topk_idx"][toks]
    check_sampled_token_backward(*args, dx, dg, idx, "exact")
    bad = dx.copy()
    bad[1, 3] = -bad[1, 3] + 0.5 * np.sqrt(np.mean(dx ** 2))          # a sign slip
    with pytest.raises(AssertionError):
        check_sampled_token_backward(*args, bad, dg, idx, "dx sign")
    bad = dg.copy()
    bad[0] = bad[0][::-1]                                                # gate gradients of the wrong expert
    with pytest.raises(AssertionError):
        check_sampled_token_backward(*args, dx, bad, idx, "dgates swapped")
    bad = dx.copy()
    bad[2] = b["dx"][(toks[2] + 1) % shp.T]                              # another token's row
    with pytest.raises(AssertionError):
        check_sampled_token_backward(*args, bad, dg, idx, "dx wrong token")


@pytest.mark.parametrize("quant", [False, True])
def test_expert_wgrad_checker_accepts_the_layer_and_rejects_errors(quant):
    qf = O.mx_quantize_dequantize if quant else None
    fro = 5e-2 if quant else None
    shp, x, w_r, w13, w2, dy, f, b = _backward_case(quant=qf)
    counts = f["counts"]
    e = int(np.argmax(counts))
    lo, hi = int(f["offsets"][e]), int(f["offsets"][e + 1])
    src = f["src_of"][lo:hi].astype(np.int64)
    toks = src // shp.k
    g_rows = f["gates"].reshape(-1)[src]
    r13 = np.array([0, 9, 100, 127])
    r2 = np.array([3, 31, 12])
    got13, got2, dg = b["dw13"][e][r13], b["dw2"][e][r2], b["dgates"].reshape(-1)[src]
    args = (x[toks], dy[toks], g_rows, w13[e], w2[e], r13, r2)
    check_sampled_expert_wgrads(*args, got13, got2, "exact", got_dg=dg, quant=qf, fro_tol=fro)
    with pytest.raises(AssertionError):                                  # rows off by one
        check_sampled_expert_wgrads(*args, b["dw13"][e][(r13 + 1) % (2 * shp.I)], got2, "dw13 shifted", quant=qf, fro_tol=fro)
    with pytest.raises(AssertionError):                                  # a sign slip
        check_sampled_expert_wgrads(*args, got13, -got2, "dw2 sign", quant=qf, fro_tol=fro)
    with pytest.raises(AssertionError):                                  # up and gate halves exchanged
        swapped = b["dw13"][e][(r13 + shp.I) % (2 * shp.I)]
        check_sampled_expert_wgrads(*args, swapped, got2, "dw13 halves", quant=qf, fro_tol=fro)
    with pytest.raises(AssertionError):                                  # gate gradients of other rows
        check_sampled_expert_wgrads(*args, got13, got2, "dg rolled", got_dg=np.roll(dg, 1), quant=qf, fro_tol=fro)
