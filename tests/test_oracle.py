"""Pins of the CPU oracle against facts other than itself (CPU only).

Each check is chosen so that a plausible mistake in the oracle (a dropped term,
a wrong sign or index, a transposed operand, a wrong tie rule) fails one of them:
brute force on tiny inputs written with plain Python loops, a stable library
sort, closed-form special cases, invariants of the schedule table, central finite
differences and torch float64 autograd for the backward, and the E4M3 grid for
the MX quantiser.
"""
import itertools
import math

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand_layer(rng, T, H, E, I, scale=0.5):
    x = rng.normal(0, 1.0, (T, H))
    w_r = rng.normal(0, scale, (E, H))
    w13 = rng.normal(0, scale, (E, 2 * I, H))
    w2 = rng.normal(0, scale, (E, H, I))
    return x, w_r, w13, w2


# ---------------------------------------------------------------------------
# top-k
# ---------------------------------------------------------------------------

def _topk_brute(row, k):
    """Best-first experts by plain comparison: larger score first, then lower index."""
    chosen = []
    for _ in range(k):
        best = None
        for e, v in enumerate(row):
            if e in chosen:
                continue
            if best is None or v > row[best]:
                best = e
        chosen.append(best)
    return chosen


def test_topk_matches_brute_force_with_ties():
    rng = np.random.default_rng(3)
    sel = rng.integers(0, 5, size=(64, 12)).astype(np.float64)   # many exact ties
    for k in (1, 3, 8):
        got = O.select_topk(sel, k)
        for t in range(sel.shape[0]):
            assert list(got[t]) == _topk_brute(list(sel[t]), k)


def test_topk_all_equal_takes_lowest_indices():
    sel = np.zeros((2, 9))
    assert O.select_topk(sel, 4).tolist() == [[0, 1, 2, 3]] * 2


def test_gate_values_softmax_and_renorm():
    scores = np.array([[0.1, 0.5, 0.2, 0.2]])
    idx = np.array([[1, 2]], dtype=np.int32)
    assert np.allclose(O.gate_values(scores, idx, False), [[0.5, 0.2]])
    assert np.allclose(O.gate_values(scores, idx, True), [[0.5 / 0.7, 0.2 / 0.7]])
    assert np.allclose(O.gate_values(scores, idx, True, 2.5), [[2.5 * 0.5 / 0.7, 2.5 * 0.2 / 0.7]])


def test_router_scores_closed_forms():
    x = np.array([[1.0, -2.0]])
    w = np.array([[0.5, 0.25], [0.0, 1.0], [-1.0, 0.0]])
    logits, p = O.router_scores(x, w, O.SOFTMAX)
    assert np.allclose(logits, [[0.0, -2.0, -1.0]])
    ex = np.exp([0.0, -2.0, -1.0])
    assert np.allclose(p, ex / ex.sum())
    _, s = O.router_scores(x, w, O.SIGMOID)
    assert np.allclose(s, [[0.5, 1 / (1 + math.e ** 2), 1 / (1 + math.e)]])


def test_bias_moves_selection_not_gates():
    x = np.array([[1.0, 0.0]])
    w = np.array([[0.3, 0.0], [0.2, 0.0], [0.1, 0.0]])
    bias = np.array([0.0, 0.0, 1.0])
    r = O.route(x, w, bias, O.SIGMOID, 1, False)
    assert r["topk_idx"].tolist() == [[2]]
    assert np.isclose(r["gates"][0, 0], 1 / (1 + math.exp(-0.1)))


# ---------------------------------------------------------------------------
# schedule table
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,E,k,seed", [(1, 1, 1, 0), (7, 3, 2, 1), (100, 8, 2, 2), (513, 16, 4, 3)])
def test_schedule_equals_stable_argsort_and_invariants(T, E, k, seed):
    rng = np.random.default_rng(seed)
    # skewed draws, some experts empty
    p = rng.dirichlet(np.ones(E) * 0.3)
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p) if k <= E else None
                    for _ in range(T)]).astype(np.int32)
    s = O.schedule(idx, E)
    flat = idx.reshape(-1)
    R = flat.size
    # independent construction: numpy's stable sort of expert ids
    src_ref = np.argsort(flat, kind="stable")
    assert np.array_equal(s["src_of"], src_ref)
    row_ref = np.empty(R, dtype=np.int64)
    row_ref[src_ref] = np.arange(R)
    assert np.array_equal(s["row_of"], row_ref)
    assert np.array_equal(s["counts"], np.bincount(flat, minlength=E))
    assert s["offsets"][0] == 0 and s["offsets"][-1] == R
    assert np.array_equal(np.diff(s["offsets"]), s["counts"])
    assert sorted(s["row_of"].tolist()) == list(range(R))            # bijection
    assert np.array_equal(s["src_of"][s["row_of"]], np.arange(R))    # inverse
    for e in range(E):
        seg = s["src_of"][s["offsets"][e]:s["offsets"][e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)                               # ascending (stable)


# ---------------------------------------------------------------------------
# forward
# ---------------------------------------------------------------------------

def _forward_brute(x, w_r, w13, w2, kind, k, renorm, bias=None):
    """Each token runs its k experts directly, scalar Python loops, no schedule."""
    T, H = x.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    y = np.zeros((T, H))
    for t in range(T):
        logits = [sum(x[t, c] * w_r[e, c] for c in range(H)) for e in range(E)]
        if kind == O.SOFTMAX:
            m = max(logits)
            ex = [math.exp(v - m) for v in logits]
            sc = [v / sum(ex) for v in ex]
        else:
            sc = [1.0 / (1.0 + math.exp(-v)) for v in logits]
        sel = [sc[e] + (0.0 if bias is None else bias[e]) for e in range(E)]
        chosen = _topk_brute(sel, k)
        g = [sc[e] for e in chosen]
        if renorm:
            tot = sum(g)
            g = [v / tot for v in g]
        for j, e in enumerate(chosen):
            hh = [sum(w13[e, i, c] * x[t, c] for c in range(H)) for i in range(I)]
            uu = [sum(w13[e, I + i, c] * x[t, c] for c in range(H)) for i in range(I)]
            aa = [hh[i] / (1 + math.exp(-hh[i])) * uu[i] for i in range(I)]
            for c in range(H):
                y[t, c] += g[j] * sum(w2[e, c, i] * aa[i] for i in range(I))
    return y


@pytest.mark.parametrize("kind,renorm,use_bias", [(O.SOFTMAX, False, False), (O.SIGMOID, True, False),
                                                  (O.SIGMOID, True, True), (O.SOFTMAX, True, False)])
def test_forward_matches_per_token_brute_force(kind, renorm, use_bias):
    rng = np.random.default_rng(11)
    T, H, E, I, k = 9, 6, 5, 4, 2
    x, w_r, w13, w2 = _rand_layer(rng, T, H, E, I)
    bias = rng.normal(0, 0.3, E) if use_bias else None
    got = O.forward(x, w_r, w13, w2, kind=kind, k=k, renorm=renorm, router_bias=bias)["y"]
    ref = _forward_brute(x, w_r, w13, w2, kind, k, renorm, bias)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_single_expert_is_dense_swiglu_ffn():
    """E=1, k=1, softmax: the gate is 1 and the layer is a dense SwiGLU FFN."""
    rng = np.random.default_rng(5)
    T, H, I = 17, 12, 10
    x, w_r, w13, w2 = _rand_layer(rng, T, H, 1, I)
    got = O.forward(x, w_r, w13, w2, kind=O.SOFTMAX, k=1, renorm=False)["y"]
    xt = torch.tensor(x)
    wg, wu = torch.tensor(w13[0, :I]), torch.tensor(w13[0, I:])
    ref = (torch.nn.functional.silu(xt @ wg.T) * (xt @ wu.T)) @ torch.tensor(w2[0]).T
    assert np.allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_identity_experts_combine_returns_input():
    """With o = x_g, sigmoid+renorm gates sum to 1, so the merge returns x; with
    softmax (no renorm) it returns (sum of the k selected probabilities) * x."""
    rng = np.random.default_rng(6)
    T, H, E, k = 40, 8, 6, 3
    x = rng.normal(0, 1, (T, H))
    w_r = rng.normal(0, 1, (E, H))
    for kind, renorm in ((O.SIGMOID, True), (O.SOFTMAX, False)):
        r = O.route(x, w_r, None, kind, k, renorm)
        s = O.schedule(r["topk_idx"], E)
        x_g = O.dispatch(x, s["src_of"], k)
        y = O.combine(x_g, r["gates"], s["row_of"])
        expect = x * r["gates"].sum(axis=1, keepdims=True)
        assert np.allclose(y, expect, rtol=1e-13, atol=1e-13)
        if renorm:
            assert np.allclose(y, x, rtol=1e-13, atol=1e-13)


def test_dispatch_rows_are_expert_contiguous_tokens():
    idx = np.array([[2, 0], [0, 1], [2, 1]], dtype=np.int32)
    s = O.schedule(idx, 3)
    x = np.arange(3 * 2, dtype=np.float64).reshape(3, 2)
    x_g = O.dispatch(x, s["src_of"], 2)
    # expert 0: tokens 0,1; expert 1: tokens 1,2; expert 2: tokens 0,2
    assert np.array_equal(x_g, x[[0, 1, 1, 2, 0, 2]])
    assert s["counts"].tolist() == [2, 2, 2]
    assert s["row_of"].tolist() == [4, 0, 1, 2, 5, 3]


# ---------------------------------------------------------------------------
# backward
# ---------------------------------------------------------------------------

def _tiny_case(kind, renorm, seed=21, T=8, H=16, E=4, I=32, k=2):
    rng = np.random.default_rng(seed)
    x, w_r, w13, w2 = _rand_layer(rng, T, H, E, I, scale=0.3)
    dy = rng.normal(0, 1, (T, H))
    return x, w_r, w13, w2, dy, k


def _selection_margin(x, w_r, kind, k, bias=None):
    _, sc = O.router_scores(x, w_r, kind)
    sel = sc if bias is None else sc + bias
    srt = -np.sort(-sel, axis=1)
    return (srt[:, k - 1] - srt[:, k]).min()


@pytest.mark.parametrize("kind,renorm,scale,use_bias", [(O.SOFTMAX, False, 1.0, False), (O.SIGMOID, True, 1.0, False),
                                                        (O.SOFTMAX, True, 1.0, False), (O.SIGMOID, False, 1.0, False),
                                                        (O.SIGMOID, True, 2.5, True), (O.SOFTMAX, False, 0.7, False)])
def test_backward_matches_central_differences(kind, renorm, scale, use_bias):
    x, w_r, w13, w2, dy, k = _tiny_case(kind, renorm)
    E = w_r.shape[0]
    bias = np.linspace(-0.05, 0.05, E) if use_bias else None
    assert _selection_margin(x, w_r, kind, k, bias) > 1e-4
    fwd = O.forward(x, w_r, w13, w2, kind=kind, k=k, renorm=renorm, router_bias=bias, route_scale=scale)
    grads = O.backward(fwd, dy, x, w_r, w13, w2, kind=kind, k=k, renorm=renorm, route_scale=scale)
    idx = fwd["topk_idx"]

    def loss(x_, w_r_, w13_, w2_):
        f = O.forward(x_, w_r_, w13_, w2_, kind=kind, k=k, renorm=renorm, topk_idx=idx, route_scale=scale)
        return float((dy * f["y"]).sum())

    eps = 1e-6
    rng = np.random.default_rng(0)
    args = [x, w_r, w13, w2]
    names = ["dx", "dw_router", "dw13", "dw2"]
    for ai, name in enumerate(names):
        flat_n = args[ai].size
        for pos in rng.choice(flat_n, size=12, replace=False):
            ip = np.unravel_index(pos, args[ai].shape)
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[ai][ip] += eps
            minus[ai][ip] -= eps
            fd = (loss(*plus) - loss(*minus)) / (2 * eps)
            assert abs(fd - grads[name][ip]) <= 1e-6 * max(1.0, abs(fd)), (name, ip, fd, grads[name][ip])


@pytest.mark.parametrize("kind,renorm", [(O.SOFTMAX, False), (O.SIGMOID, True)])
def test_route_scale_is_linear(kind, renorm):
    """For a fixed selection y is linear in the gates, and the gates in the route scale s: y and
    every gradient at scale s are s times those at scale 1; the selection does not move."""
    x, w_r, w13, w2, dy, k = _tiny_case(kind, renorm, seed=6)
    f1 = O.forward(x, w_r, w13, w2, kind=kind, k=k, renorm=renorm)
    g1 = O.backward(f1, dy, x, w_r, w13, w2, kind=kind, k=k, renorm=renorm)
    s = 2.5
    fs = O.forward(x, w_r, w13, w2, kind=kind, k=k, renorm=renorm, route_scale=s)
    gs = O.backward(fs, dy, x, w_r, w13, w2, kind=kind, k=k, renorm=renorm, route_scale=s)
    assert np.array_equal(fs["topk_idx"], f1["topk_idx"])
    assert np.allclose(fs["gates"], s * f1["gates"], rtol=1e-14, atol=0)
    assert np.allclose(fs["y"], s * f1["y"], rtol=1e-12, atol=1e-15)
    for name in ("dx", "dw_router", "dw13", "dw2"):
        assert np.allclose(gs[name], s * g1[name], rtol=1e-12, atol=1e-15), name
    # d loss / d gate is <dY, o>, which does not depend on the gates
    assert np.allclose(gs["dgates"], g1["dgates"], rtol=1e-12, atol=1e-15)


def test_unselected_experts_have_zero_gradient_and_no_influence():
    """With a selection that never picks some experts: their dW13 / dW2 are exactly zero, and
    changing their weights changes neither y nor any other gradient (an expert-index slip in the
    grouped steps would move one of these)."""
    rng = np.random.default_rng(11)
    T, H, E, I, k = 9, 12, 6, 8, 2
    x, w_r, w13, w2 = _rand_layer(rng, T, H, E, I, scale=0.3)
    dy = rng.normal(0, 1, (T, H))
    idx = np.array([[(t % 3) * 2, (t % 3) * 2 + 2 if t % 3 < 2 else 0] for t in range(T)], dtype=np.int32)
    unused = sorted(set(range(E)) - set(idx.ravel().tolist()))
    assert unused == [1, 3, 5]
    kw = dict(kind=O.SIGMOID, k=k, renorm=True)
    f = O.forward(x, w_r, w13, w2, topk_idx=idx, **kw)
    g = O.backward(f, dy, x, w_r, w13, w2, **kw)
    assert not g["dw13"][unused].any() and not g["dw2"][unused].any()
    w13b, w2b = w13.copy(), w2.copy()
    w13b[unused] = rng.normal(0, 5.0, w13b[unused].shape)
    w2b[unused] = rng.normal(0, 5.0, w2b[unused].shape)
    fb = O.forward(x, w_r, w13b, w2b, topk_idx=idx, **kw)
    gb = O.backward(fb, dy, x, w_r, w13b, w2b, **kw)
    assert np.array_equal(fb["y"], f["y"])
    for name in ("dx", "dw_router", "dw13", "dw2", "dgates"):
        assert np.array_equal(gb[name], g[name]), name


def test_dgates_is_derivative_of_merge():
    x, w_r, w13, w2, dy, k = _tiny_case(O.SIGMOID, True, seed=4)
    fwd = O.forward(x, w_r, w13, w2, kind=O.SIGMOID, k=k, renorm=True)
    grads = O.backward(fwd, dy, x, w_r, w13, w2, kind=O.SIGMOID, k=k, renorm=True)
    eps = 1e-6
    for t, j in [(0, 0), (3, 1), (7, 0)]:
        gp = fwd["gates"].copy(); gp[t, j] += eps
        gm = fwd["gates"].copy(); gm[t, j] -= eps
        fd = ((dy * O.combine(fwd["o"], gp, fwd["row_of"])).sum()
              - (dy * O.combine(fwd["o"], gm, fwd["row_of"])).sum()) / (2 * eps)
        assert abs(fd - grads["dgates"][t, j]) < 1e-7 * max(1, abs(fd))


@pytest.mark.parametrize("kind,renorm", [(O.SOFTMAX, False), (O.SIGMOID, True)])
def test_backward_matches_torch_autograd(kind, renorm):
    """Independent forward in torch float64 (per token), gradients by autograd."""
    x, w_r, w13, w2, dy, k = _tiny_case(kind, renorm, seed=8, T=10, H=12, E=5, I=8, k=3)
    fwd = O.forward(x, w_r, w13, w2, kind=kind, k=k, renorm=renorm)
    grads = O.backward(fwd, dy, x, w_r, w13, w2, kind=kind, k=k, renorm=renorm)
    tx, tr, t13, t2 = (torch.tensor(a, requires_grad=True) for a in (x, w_r, w13, w2))
    I = w13.shape[1] // 2
    logits = tx @ tr.T
    sc = torch.softmax(logits, dim=1) if kind == O.SOFTMAX else torch.sigmoid(logits)
    idx = torch.tensor(fwd["topk_idx"], dtype=torch.long)
    ys = []
    for t in range(x.shape[0]):
        g = sc[t, idx[t]]
        if renorm:
            g = g / g.sum()
        yt = 0
        for j in range(k):
            e = int(idx[t, j])
            h = t13[e, :I] @ tx[t]
            u = t13[e, I:] @ tx[t]
            yt = yt + g[j] * (t2[e] @ (torch.nn.functional.silu(h) * u))
        ys.append(yt)
    y = torch.stack(ys)
    assert np.allclose(y.detach().numpy(), fwd["y"], rtol=1e-12, atol=1e-12)
    (y * torch.tensor(dy)).sum().backward()
    for name, tgt in (("dx", tx), ("dw_router", tr), ("dw13", t13), ("dw2", t2)):
        assert np.allclose(grads[name], tgt.grad.numpy(), rtol=1e-10, atol=1e-12), name


# ---------------------------------------------------------------------------
# MXFP8
# ---------------------------------------------------------------------------

def _all_e4m3_values():
    """Every finite E4M3 value, decoded from its 8-bit code (bias 7, no infinities)."""
    vals = []
    for code in range(256):
        s = -1.0 if code & 0x80 else 1.0
        ex = (code >> 3) & 0xF
        m = code & 0x7
        if ex == 0xF and m == 0x7:
            continue                      # NaN
        v = m / 8 * 2.0 ** -6 if ex == 0 else (1 + m / 8) * 2.0 ** (ex - 7)
        vals.append(s * v)
    return np.array(sorted(set(vals)))


def test_e4m3_grid_round_trips_and_nearest():
    grid = _all_e4m3_values()
    assert grid.max() == 448.0 and len(grid) == 253    # 126 positive, 126 negative, one zero
    assert np.array_equal(O.round_e4m3(grid), grid)
    rng = np.random.default_rng(1)
    v = rng.uniform(-460, 460, 20000)
    r = O.round_e4m3(v)
    dist = np.abs(grid[None, :] - v[:, None])
    best = dist.min(axis=1)
    assert np.all(np.abs(r - v) <= best + 0)          # nearest
    assert np.all(np.isin(r, grid))


def test_e4m3_matches_torch_float8_cast():
    rng = np.random.default_rng(2)
    v = np.concatenate([rng.normal(0, 30, 5000), rng.normal(0, 0.01, 5000), rng.uniform(-448, 448, 2000)])
    ref = torch.tensor(v, dtype=torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.round_e4m3(v.astype(np.float32).astype(np.float64))
    assert np.array_equal(got, ref)


def test_e4m3_ties_to_even():
    # 17 lies halfway between 16 and 18 (quantum 2 in [16, 32)); the even mantissa is 16.
    assert O.round_e4m3(np.array([17.0, 19.0, -17.0]))[0] == 16.0
    assert O.round_e4m3(np.array([19.0]))[0] == 20.0
    assert O.round_e4m3(np.array([1000.0]))[0] == 448.0


def test_mx_block_scale_and_error_bound():
    rng = np.random.default_rng(9)
    v = rng.normal(0, 1, (6, 96)) * np.exp(rng.normal(0, 3, (6, 1)))
    v[0, :32] = 0.0
    elems, X = O.mx_quantize(v, axis=1)
    assert X.shape == (6, 3)
    assert X[0, 0] == -127 and np.all(elems[0, :32] == 0)
    blocks = np.abs(v).reshape(6, 3, 32).max(axis=-1)
    nz = blocks > 0
    ratio = blocks[nz] / np.ldexp(1.0, X[nz])
    assert np.all((ratio >= 256) & (ratio < 512))     # amax lands in [2^8, 2^9) before rounding
    deq = O.mx_quantize_dequantize(v, axis=1)
    scale = np.repeat(np.ldexp(1.0, X), 32, axis=1)
    scaled = np.abs(v) / scale
    normal = (scaled >= 2.0 ** -6) & (scaled <= 448.0)
    rel = np.abs(deq - v)[normal] / np.abs(v)[normal]
    assert rel.max() <= 2.0 ** -4 + 1e-15             # half a unit in the last place of 3 bits
    # scaled magnitudes above 448 (possible up to 2^9 with this scale rule) saturate
    over = scaled > 464.0
    assert np.all(np.abs(deq[over]) == 448.0 * scale[over])
    # values already on the grid times a power of two survive exactly
    g = _all_e4m3_values()[::3][:32] * 2.0 ** -5
    assert np.array_equal(O.mx_quantize_dequantize(g[None, :], axis=1)[0], g)


def test_mx_ragged_axis_and_axis0():
    rng = np.random.default_rng(10)
    v = rng.normal(0, 1, (45, 7))
    d0 = O.mx_quantize_dequantize(v, axis=0)
    d1 = O.mx_quantize_dequantize(v.T, axis=1).T
    assert np.array_equal(d0, d1)
    _, X = O.mx_quantize(v, axis=0)
    scale = np.repeat(np.ldexp(1.0, X), 32, axis=0)[:45]
    err = np.abs(d0 - v)
    # within half a quantum, or clipped at 448 * scale
    ok = (err <= np.abs(v) * 2.0 ** -4 + 2.0 ** -10 * scale) | (np.abs(d0) == 448.0 * scale)
    assert np.all(ok)


def test_quantized_forward_close_to_exact():
    rng = np.random.default_rng(12)
    x, w_r, w13, w2 = _rand_layer(rng, 32, 64, 4, 64, scale=0.2)
    ref = O.forward(x, w_r, w13, w2, kind=O.SIGMOID, k=2, renorm=True)["y"]
    q = O.forward(x, w_r, w13, w2, kind=O.SIGMOID, k=2, renorm=True, quant=O.mx_quantize_dequantize)["y"]
    rel = np.linalg.norm(q - ref) / np.linalg.norm(ref)
    # four quantised operands of about 3% error each, through the SwiGLU
    assert 1e-3 < rel < 0.15


def test_token_forward_matches_layer():
    rng = np.random.default_rng(13)
    x, w_r, w13, w2 = _rand_layer(rng, 12, 16, 6, 8)
    bias = rng.normal(0, 0.1, 6)
    fwd = O.forward(x, w_r, w13, w2, kind=O.SIGMOID, k=3, renorm=True, router_bias=bias)
    for t in (0, 5, 11):
        y, idx, g, _, _ = O.token_forward(x[t], w_r, bias, lambda e: (w13[e], w2[e]),
                                          kind=O.SIGMOID, k=3, renorm=True)
        assert np.array_equal(idx, fwd["topk_idx"][t])
        assert np.allclose(y, fwd["y"][t], rtol=1e-13, atol=1e-13)


def test_token_forward_quantized_matches_layer():
    rng = np.random.default_rng(14)
    x, w_r, w13, w2 = _rand_layer(rng, 10, 64, 4, 64, scale=0.2)
    q = O.mx_quantize_dequantize
    fwd = O.forward(x, w_r, w13, w2, kind=O.SIGMOID, k=2, renorm=True, quant=q)
    for t in (0, 7):
        y, *_ = O.token_forward(x[t], w_r, None, lambda e: (w13[e], w2[e]), kind=O.SIGMOID, k=2, renorm=True,
                                quant=q)
        assert np.allclose(y, fwd["y"][t], rtol=1e-12, atol=1e-14)


def test_quantized_backward_quantises_each_operand_along_its_reduction():
    """MX emulation of the backward: every GEMM operand goes through q exactly once, along the
    reduction dimension of its GEMM: dY_g rows and W2[e] along H for dA' = dY_g W2[e]; dHU rows
    and W13[e] along 2I for dX_g = dHU W13[e]; the expert's rows for both weight gradients
    (dO and a for dW2, dHU and x_g for dW13).  With q the identity the result is unchanged."""
    rng = np.random.default_rng(15)
    T, H, E, I, k = 12, 96, 3, 32, 2   # H, I, 2I and every expert's row count all differ
    x, w_r, w13, w2 = _rand_layer(rng, T, H, E, I, scale=0.2)
    dy = rng.normal(0, 1, (T, H))
    fwd = O.forward(x, w_r, w13, w2, kind=O.SIGMOID, k=k, renorm=True)
    calls = []

    def rec(v, axis):
        calls.append((tuple(np.asarray(v).shape), axis))
        return v

    ref = O.backward(fwd, dy, x, w_r, w13, w2, kind=O.SIGMOID, k=k, renorm=True)
    got = O.backward(fwd, dy, x, w_r, w13, w2, kind=O.SIGMOID, k=k, renorm=True, quant=rec)
    for name in ("dx", "dw13", "dw2", "dgates", "dw_router"):
        assert np.allclose(got[name], ref[name], rtol=1e-12, atol=1e-12), name
    expected = []
    for e in range(E):
        n = int(fwd["offsets"][e + 1] - fwd["offsets"][e])
        if n == 0:
            continue
        assert n not in (H, I, 2 * I)
        expected += [((n, H), 1), ((H, I), 0),          # dA' = dY_g W2[e]
                     ((n, H), 0), ((n, I), 0),          # dW2 = dO^T a
                     ((n, 2 * I), 0), ((n, H), 0),      # dW13 = dHU^T x_g
                     ((n, 2 * I), 1), ((2 * I, H), 0)]  # dX_g = dHU W13[e]
    assert sorted(calls) == sorted(expected)


def test_quantized_backward_close_to_exact():
    rng = np.random.default_rng(16)
    x, w_r, w13, w2 = _rand_layer(rng, 32, 64, 4, 64, scale=0.2)
    dy = rng.normal(0, 1, (32, 64))
    q = O.mx_quantize_dequantize
    f_ref = O.forward(x, w_r, w13, w2, kind=O.SIGMOID, k=2, renorm=True)
    f_q = O.forward(x, w_r, w13, w2, kind=O.SIGMOID, k=2, renorm=True, quant=q)
    ref = O.backward(f_ref, dy, x, w_r, w13, w2, kind=O.SIGMOID, k=2, renorm=True)
    got = O.backward(f_q, dy, x, w_r, w13, w2, kind=O.SIGMOID, k=2, renorm=True, quant=q)
    for name in ("dx", "dw13", "dw2", "dgates"):
        rel = np.linalg.norm(got[name] - ref[name]) / np.linalg.norm(ref[name])
        assert 1e-3 < rel < 0.2, (name, rel)


# ---------------------------------------------------------------------------
# Sampled evaluators (the full-size GPU checks use them one token / one expert at a time)
# ---------------------------------------------------------------------------

def test_quantized_forward_quantises_each_operand_along_its_reduction():
    """MX emulation of the forward: x_g and W13[e] along H for h | u = x_g W13[e]^T, a and W2[e]
    along I for o = a W2[e]^T; each operand exactly once per expert.  token_forward quantises
    the same operands along the same axes.  With q the identity nothing changes."""
    rng = np.random.default_rng(21)
    T, H, E, I, k = 14, 96, 3, 40, 2      # H, I, 2I and the experts' row counts all differ
    x, w_r, w13, w2 = _rand_layer(rng, T, H, E, I, scale=0.2)
    calls = []

    def rec(v, axis):
        calls.append((tuple(np.asarray(v).shape), axis))
        return v

    ref = O.forward(x, w_r, w13, w2, kind=O.SIGMOID, k=k, renorm=True)
    got = O.forward(x, w_r, w13, w2, kind=O.SIGMOID, k=k, renorm=True, quant=rec)
    assert np.allclose(got["y"], ref["y"], rtol=1e-13, atol=1e-13)
    expected = []
    for e in range(E):
        n = int(ref["offsets"][e + 1] - ref["offsets"][e])
        if n == 0:
            continue
        assert n not in (H, I, 2 * I)
        expected += [((n, H), 1), ((2 * I, H), 1),     # h | u = x_g W13[e]^T, reduction over H
                     ((n, I), 1), ((H, I), 1)]         # o = a W2[e]^T, reduction over I
    assert sorted(calls) == sorted(expected)
    calls.clear()
    O.token_forward(x[3], w_r, None, lambda e: (w13[e], w2[e]), kind=O.SIGMOID, k=k, renorm=True, quant=rec)
    assert sorted(calls) == sorted([((1, H), 1)] + [((2 * I, H), 1), ((1, I), 1), ((H, I), 1)] * k)


def _layer_case(kind, renorm, use_bias, scale, seed):
    rng = np.random.default_rng(seed)
    T, H, E, I, k = 20, 64, 6, 32, 3
    x, w_r, w13, w2 = _rand_layer(rng, T, H, E, I, scale=0.3)
    dy = rng.normal(0, 1, (T, H))
    bias = rng.normal(0, 0.1, E) if use_bias else None
    return x, w_r, w13, w2, dy, bias, k


@pytest.mark.parametrize("kind,renorm,use_bias,scale,quant", [
    (O.SIGMOID, True, False, 1.0, False), (O.SIGMOID, True, True, 2.5, False),
    (O.SOFTMAX, False, False, 1.0, False), (O.SOFTMAX, True, True, 0.7, False),
    (O.SIGMOID, True, True, 1.0, True)])
def test_token_backward_matches_layer(kind, renorm, use_bias, scale, quant):
    """token_backward equals the whole-layer backward on every token, element by element: dx,
    the gate gradients, dl, and the token's k rows of dh | du and of the dX_g rows."""
    x, w_r, w13, w2, dy, bias, k = _layer_case(kind, renorm, use_bias, scale, seed=22)
    qf = O.mx_quantize_dequantize if quant else None
    if quant:   # H and I multiples of 32 so that the row blocks are whole
        assert x.shape[1] % 32 == 0 and w13.shape[1] % 64 == 0
    fwd = O.forward(x, w_r, w13, w2, kind=kind, k=k, renorm=renorm, router_bias=bias, route_scale=scale, quant=qf)
    bwd = O.backward(fwd, dy, x, w_r, w13, w2, kind=kind, k=k, renorm=renorm, route_scale=scale, quant=qf)
    rows = fwd["row_of"].reshape(-1, k)
    for t in range(x.shape[0]):
        got = O.token_backward(x[t], dy[t], w_r, bias, lambda e: (w13[e], w2[e]), kind=kind, k=k, renorm=renorm,
                               route_scale=scale, quant=qf)
        assert np.array_equal(got["topk_idx"], fwd["topk_idx"][t])
        close = dict(rtol=1e-12, atol=1e-12)
        assert np.allclose(got["y"], fwd["y"][t], **close)
        assert np.allclose(got["dx"], bwd["dx"][t], **close)
        assert np.allclose(got["dgates"], bwd["dgates"][t], **close)
        assert np.allclose(got["dl"], bwd["dl"][t], **close)
        assert np.allclose(got["dhu"], bwd["dhu"][rows[t]], **close)
        assert np.allclose(got["dx_g"], bwd["dx_g"][rows[t]], **close)


@pytest.mark.parametrize("quant", [False, True])
def test_expert_weight_grads_match_layer(quant):
    """expert_weight_grads on one expert's rows (schedule order) equals the whole-layer
    backward's dW13[e], dW2[e], the rows' gate gradients and dh | du; selected output rows equal
    the same rows of the full result."""
    x, w_r, w13, w2, dy, bias, k = _layer_case(O.SIGMOID, True, True, 1.0, seed=23)
    qf = O.mx_quantize_dequantize if quant else None
    fwd = O.forward(x, w_r, w13, w2, kind=O.SIGMOID, k=k, renorm=True, router_bias=bias, quant=qf)
    bwd = O.backward(fwd, dy, x, w_r, w13, w2, kind=O.SIGMOID, k=k, renorm=True, quant=qf)
    E = w13.shape[0]
    src = fwd["src_of"].astype(np.int64)
    seen = 0
    for e in range(E):
        lo, hi = int(fwd["offsets"][e]), int(fwd["offsets"][e + 1])
        if hi == lo:
            continue
        seen += 1
        toks = src[lo:hi] // k
        g_rows = fwd["gates"].reshape(-1)[src[lo:hi]]
        got = O.expert_weight_grads(x[toks], dy[toks], g_rows, w13[e], w2[e], quant=qf)
        close = dict(rtol=1e-12, atol=1e-12)
        assert np.allclose(got["dw13"], bwd["dw13"][e], **close)
        assert np.allclose(got["dw2"], bwd["dw2"][e], **close)
        assert np.allclose(got["dg"], bwd["dgates"].reshape(-1)[src[lo:hi]], **close)
        assert np.allclose(got["dhu"], bwd["dhu"][lo:hi], **close)
        r13 = np.array([5, 0, 63, 17])
        r2 = np.array([1, 40, 7])
        sel = O.expert_weight_grads(x[toks], dy[toks], g_rows, w13[e], w2[e], rows13=r13, rows2=r2, quant=qf)
        assert np.allclose(sel["dw13"], got["dw13"][r13], rtol=1e-13, atol=1e-13)
        assert np.allclose(sel["dw2"], got["dw2"][r2], rtol=1e-13, atol=1e-13)
    assert seen >= 3


def test_expert_weight_grads_quantises_each_operand_along_its_reduction():
    """The weight-gradient operands along the expert's rows (axis 0), the forward and dA'
    operands along their own reductions, each once."""
    x, w_r, w13, w2, dy, bias, k = _layer_case(O.SIGMOID, True, False, 1.0, seed=24)
    n, H = 7, x.shape[1]
    I = w13.shape[1] // 2
    calls = []

    def rec(v, axis):
        calls.append((tuple(np.asarray(v).shape), axis))
        return v

    O.expert_weight_grads(x[:n], dy[:n], np.full(n, 0.3), w13[0], w2[0], quant=rec)
    assert sorted(calls) == sorted([((n, H), 1), ((2 * I, H), 1),     # h | u
                                    ((n, H), 1), ((H, I), 0),         # dA' = dY W2[e]
                                    ((n, H), 0), ((n, I), 0),         # dW2 = dO^T a
                                    ((n, 2 * I), 0), ((n, H), 0)])    # dW13 = dHU^T x
