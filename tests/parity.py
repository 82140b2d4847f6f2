"""Shared helpers of the GPU parity tests: tolerance checks and oracle runs on the inputs
handed to the CUDA path (the oracle only ever sees generator draws, never GPU output)."""
import numpy as np
import torch

from oracle import moe_oracle as O

# bf16 outputs and gradients: max|err| <= 2e-2 * RMS(reference), relative Frobenius <= 1e-2
BF16_MAX_REL_RMS = 2e-2
BF16_FRO = 1e-2


def to_f64(t):
    return t.detach().to("cpu").double().numpy()


def err_stats(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    diff = got - want
    rms = np.sqrt(np.mean(want ** 2)) if want.size else 0.0
    fro = np.linalg.norm(diff) / max(np.linalg.norm(want), 1e-300)
    return float(np.abs(diff).max() if diff.size else 0.0), float(rms), float(fro)


def assert_bf16_close(got, want, name, max_rel_rms=BF16_MAX_REL_RMS, fro_tol=BF16_FRO):
    mx, rms, fro = err_stats(got, want)
    assert mx <= max_rel_rms * rms and fro <= fro_tol, (
        f"{name}: max|err| {mx:.3e} vs {max_rel_rms}*rms {max_rel_rms * rms:.3e}, rel fro {fro:.3e}")


def assert_intermediate_close(got, want, name, rel=2.0 ** -7, fro_tol=BF16_FRO):
    """Intermediates (h | u in fp32, a and dh | du as bf16 hi + lo pairs, o and dX rows in fp32):
    each element within `rel` of the float64 value plus 1e-2 of the RMS, and the relative
    Frobenius error within 1e-2.  The elementwise form (rather than max error against the
    RMS) suits heavy-tailed products such as a = silu(h) * u."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    _, rms, fro = err_stats(got, want)
    bound = rel * np.abs(want) + 1e-2 * rms
    worst = np.max(np.abs(got - want) - bound)
    assert worst <= 0 and fro <= fro_tol, f"{name}: worst excess {worst:.3e}, rel fro {fro:.3e}"


def inputs_f64(inp):
    return {k: (to_f64(v) if v is not None else None) for k, v in inp.items()}


def oracle_layer(shape, f64, topk_idx=None, backward=True, route_scale=1.0):
    fwd = O.forward(f64["x"], f64["w_router"], f64["w13"], f64["w2"], kind=shape.router, k=shape.k,
                    renorm=shape.renorm, router_bias=f64.get("router_bias"), topk_idx=topk_idx,
                    route_scale=route_scale)
    bwd = None
    if backward:
        bwd = O.backward(fwd, f64["dy"], f64["x"], f64["w_router"], f64["w13"], f64["w2"], kind=shape.router,
                         k=shape.k, renorm=shape.renorm, route_scale=route_scale)
    return fwd, bwd


def selection_is_valid(sel_scores, gpu_idx, k, rel_margin=1e-5):
    """GPU top-k against the oracle's selection scores: every chosen expert must score at least
    as high as every unchosen one, up to a relative margin (near-ties may break either way).
    Returns the number of tokens whose chosen set differs from the oracle's exact top-k."""
    T, E = sel_scores.shape
    n_diff = 0
    exact = O.select_topk(sel_scores, k)
    for t in range(T):
        chosen = set(int(e) for e in gpu_idx[t])
        assert len(chosen) == k, f"token {t}: repeated experts {gpu_idx[t]}"
        if chosen != set(int(e) for e in exact[t]):
            n_diff += 1
            lo = min(sel_scores[t, e] for e in chosen)
            hi = max(sel_scores[t, e] for e in range(E) if e not in chosen)
            assert lo >= hi - rel_margin * max(abs(hi), 1.0), f"token {t}: {lo} < {hi}"
    return n_diff


def clear_margin_tokens(sel_scores, k, n, seed, margin=1e-4):
    """n tokens drawn (seeded) among those whose k-th and (k+1)-th selection scores differ by
    more than `margin`, so that the GPU's fp32 router and the oracle must pick the same experts."""
    srt = -np.sort(-sel_scores, axis=1)
    ok = np.nonzero(srt[:, k - 1] - srt[:, k] > margin)[0]
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(ok, size=min(n, ok.size), replace=False))


def check_sampled_token_outputs(tokens, x_rows, w_router, router_bias, expert_weights, shape, y_rows, idx_rows,
                                name):
    """Output rows of sampled tokens against the oracle computing each token on its own: the
    GPU's experts for each token must be the oracle's, and the rows must meet the bf16 bar.
    x_rows / y_rows / idx_rows hold the sampled tokens' rows (float64 / float64 / int)."""
    want = []
    for i, t in enumerate(tokens):
        y_t, idx, _, _, _ = O.token_forward(x_rows[i], w_router, router_bias, expert_weights, kind=shape.router,
                                            k=shape.k, renorm=shape.renorm)
        assert list(idx) == list(idx_rows[i]), f"{name}: token {t} experts {list(idx_rows[i])} vs {list(idx)}"
        want.append(y_t)
    assert_bf16_close(np.asarray(y_rows), np.array(want), name)


def check_sampled_token_backward(tokens, x_rows, dy_rows, w_router, router_bias, expert_weights, shape, dx_rows,
                                 dg_rows, idx_rows, name, quant=None, fro_tol=None):
    """Input-gradient and gate-gradient rows of sampled tokens against the oracle's per-token
    backward (oracle.token_backward, each token computed on its own): the GPU's experts for each
    token must be the oracle's; dx and dgates must meet the bf16 bar (or, with `fro_tol`, the
    relative Frobenius bar alone, as for MXFP8)."""
    want_dx, want_dg = [], []
    for i, t in enumerate(tokens):
        r = O.token_backward(x_rows[i], dy_rows[i], w_router, router_bias, expert_weights, kind=shape.router,
                             k=shape.k, renorm=shape.renorm, quant=quant)
        assert list(r["topk_idx"]) == list(idx_rows[i]), f"{name}: token {t} experts {list(idx_rows[i])}"
        want_dx.append(r["dx"])
        want_dg.append(r["dgates"])
    for what, got, want in (("dx", dx_rows, want_dx), ("dgates", dg_rows, want_dg)):
        if fro_tol is None:
            assert_bf16_close(np.asarray(got), np.array(want), f"{name} {what}")
        else:
            _, _, fro = err_stats(np.asarray(got), np.array(want))
            assert fro <= fro_tol, f"{name} {what}: rel fro {fro:.3e}"


def check_sampled_expert_wgrads(x_rows, dy_rows, g_rows, w13_e, w2_e, rows13, rows2, got13, got2, name,
                                got_dg=None, quant=None, fro_tol=None):
    """Sampled rows of one expert's weight gradients (and optionally the gate gradients of its
    rows) against oracle.expert_weight_grads on that expert's rows in schedule order."""
    r = O.expert_weight_grads(x_rows, dy_rows, g_rows, w13_e, w2_e, rows13=rows13, rows2=rows2, quant=quant)
    pairs = [("dw13", got13, r["dw13"]), ("dw2", got2, r["dw2"])]
    if got_dg is not None:
        pairs.append(("dgates", got_dg, r["dg"]))
    for what, got, want in pairs:
        if fro_tol is None:
            assert_bf16_close(np.asarray(got), want, f"{name} {what}")
        else:
            _, _, fro = err_stats(np.asarray(got), want)
            assert fro <= fro_tol, f"{name} {what}: rel fro {fro:.3e}"
