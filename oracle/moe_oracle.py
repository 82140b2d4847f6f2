"""CPU oracle of one mixture-of-experts layer, forward and backward, in float64.

TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the benchmark's
CPU-baseline / reference leg may import or run this module.  The library's CUDA
path never calls it, shares no code with it and is never replaced by it.

What the layer computes comes from three web pages about Mixture-of-Kittens
(MoK), cited by short names:

* [wiki]        "Mixture-of-Kittens (MoK)", sd114.wiki
* [aitrending]  "Cursor Open-Sources Mixture-of-Kittens (MoK): A Deterministic MoE
                Training Megakernel for GB300 NVL72 Racks", aitrending.vip
* [entropygate] "把 MoE 通信延迟从 103μs 压到 18μs：Cursor 开源 GPU 内核 MoK",
                aientropygate.com

The pages name the steps of one MoE layer ([entropygate] §02, §04): the router
picks a few experts per token, a schedule table counts the tokens of each
expert, places them and keeps each expert's tokens contiguous, the dispatch
moves the tokens to their experts, a grouped GEMM runs each expert, and the
combine ends in a weighted merge.  The expert is a SwiGLU FFN whose backward
carries the router-weight gradient ([wiki] benchmark section; [aitrending]
"Technical Details").  The pages print no formula for any of these; where they
are silent this module takes the plain DeepSeek-V3-style reading and says so
at the function.

Every floating-point step runs in float64 on float64 copies of the bf16
inputs (exact widening).  Library primitives used as single steps: numpy
matmul and a stable argsort.  No step is blocked, fused or reordered.

Pins (tests, CPU only): brute force per token for the forward, stable
argsort and invariants for the schedule, finite differences and torch
autograd for the backward, closed forms for special cases, the E4M3 grid and
torch's float8 cast for the MX quantiser.  No function here is unpinned.
"""
from __future__ import annotations

from typing import Dict, Optional, Tuple

import numpy as np

SOFTMAX = 0
SIGMOID = 1


# ---------------------------------------------------------------------------
# Router and top-k
# ---------------------------------------------------------------------------

def router_scores(x: np.ndarray, w_router: np.ndarray, kind: int) -> Tuple[np.ndarray, np.ndarray]:
    """Router logits l = x W_r^T and per-expert scores.

    The router picks a few experts per token and its choice changes every step
    ([entropygate] §02).  The pages do not give the scoring function; the plain
    readings are softmax over the E logits, or DeepSeek-V3's elementwise sigmoid.
    Returns (logits [T][E], scores [T][E]).
    """
    logits = x @ w_router.T
    if kind == SOFTMAX:
        shifted = logits - logits.max(axis=1, keepdims=True)
        ex = np.exp(shifted)
        scores = ex / ex.sum(axis=1, keepdims=True)
    elif kind == SIGMOID:
        scores = 1.0 / (1.0 + np.exp(-logits))
    else:
        raise ValueError(f"unknown router kind {kind}")
    return logits, scores


def select_topk(selection: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest selection scores per token, best first.

    Ties go to the lower expert index (a stable sort of the negated scores), so the
    choice is a function of the scores alone, as the layer's determinism needs
    ([wiki] introduction: the fused kernel is fully deterministic).
    Returns int32 [T][k].
    """
    order = np.argsort(-selection, axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def gate_values(scores: np.ndarray, topk_idx: np.ndarray, renorm: bool,
                route_scale: float = 1.0) -> np.ndarray:
    """Gate weight of each selected expert: its score, optionally renormalised.

    Reading (pages silent): g_j = score[e_j], divided by the sum over the k selected
    scores when ``renorm`` is set, times ``route_scale``.  Returns float64 [T][k].
    """
    g = np.take_along_axis(scores, topk_idx.astype(np.int64), axis=1)
    if renorm:
        g = g / g.sum(axis=1, keepdims=True)
    return g * route_scale


def route(x, w_router, router_bias, kind, k, renorm, route_scale=1.0):
    """Router step: logits, scores, top-k experts (on score + bias) and gates.

    The bias shifts only the selection, never the gate values, and gets no
    gradient (reading: DeepSeek-V3's load-balancing bias; the pages are silent).
    """
    logits, scores = router_scores(x, w_router, kind)
    selection = scores if router_bias is None else scores + router_bias[None, :]
    topk_idx = select_topk(selection, k)
    gates = gate_values(scores, topk_idx, renorm, route_scale)
    return {"logits": logits, "scores": scores, "topk_idx": topk_idx, "gates": gates}


# ---------------------------------------------------------------------------
# Schedule table
# ---------------------------------------------------------------------------

def schedule(topk_idx: np.ndarray, E: int) -> Dict[str, np.ndarray]:
    """Schedule table: tokens per expert, where each goes, same-expert rows contiguous.

    [entropygate] §02 lists the three jobs of this step: count how many tokens each
    expert receives, decide where each lands, and keep an expert's tokens together;
    [wiki] (pull section) and [aitrending] ("Technical Details") say one table
    serves dispatch, combine and both backward transfers.  The fields are not
    given; the reading here is a stable counting sort of the assignments
    a = t*k + j by expert:

    * counts[e]  = number of assignments to expert e
    * offsets    = exclusive prefix sum of counts, offsets[E] = T*k
    * row_of[a]  = offsets[e_a] + number of earlier assignments a' < a with e_a' = e_a
    * src_of[r]  = the assignment a with row_of[a] = r
    """
    flat = topk_idx.reshape(-1)
    R = flat.shape[0]
    counts = np.zeros(E, dtype=np.int64)
    for a in range(R):
        counts[flat[a]] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    seen = np.zeros(E, dtype=np.int64)
    row_of = np.zeros(R, dtype=np.int64)
    src_of = np.zeros(R, dtype=np.int64)
    for a in range(R):
        e = flat[a]
        r = offsets[e] + seen[e]
        seen[e] += 1
        row_of[a] = r
        src_of[r] = a
    return {"counts": counts.astype(np.int32), "offsets": offsets.astype(np.int32),
            "row_of": row_of.astype(np.int32), "src_of": src_of.astype(np.int32)}


# ---------------------------------------------------------------------------
# Dispatch, expert FFN, combine
# ---------------------------------------------------------------------------

def dispatch(x: np.ndarray, src_of: np.ndarray, k: int) -> np.ndarray:
    """Pull dispatch on one device: row r of the expert-sorted buffer is token src_of[r] // k.

    [entropygate] §03 ①: the side holding the expert reads the tokens it needs and
    lays them out per local expert itself.
    """
    return x[src_of.astype(np.int64) // k]


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def expert_ffn(x_g: np.ndarray, offsets: np.ndarray, w13: np.ndarray, w2: np.ndarray):
    """Grouped SwiGLU expert FFN over the expert-contiguous rows.

    One GEMM per expert over that expert's rows ([entropygate] §02: dispatch, then
    grouped GEMM, then combine); the activation is SwiGLU ([wiki] benchmark
    section).  Reading of SwiGLU: a = silu(h) * u with h the gate half (rows
    0..I-1 of W13[e]) and u the up half (rows I..2I-1); o = a W2[e]^T.
    Returns (h, u, a, o), each [R][.] float64, o unweighted.
    """
    R, H = x_g.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    h = np.zeros((R, I))
    u = np.zeros((R, I))
    o = np.zeros((R, H))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        h[lo:hi] = x_g[lo:hi] @ w13[e, :I].T
        u[lo:hi] = x_g[lo:hi] @ w13[e, I:].T
    a = silu(h) * u
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        o[lo:hi] = a[lo:hi] @ w2[e].T
    return h, u, a, o


def combine(o: np.ndarray, gates: np.ndarray, row_of: np.ndarray) -> np.ndarray:
    """Weighted merge: y[t] = sum over j = 0..k-1 of g[t][j] * o[row_of[t*k + j]].

    [entropygate] §04 counts the final weighted merge as part of the layer; the
    sum runs in the fixed order j = 0..k-1.
    """
    T, k = gates.shape
    rows = row_of.reshape(T, k).astype(np.int64)
    y = np.zeros((T, o.shape[1]))
    for j in range(k):
        y += gates[:, j:j + 1] * o[rows[:, j]]
    return y


def forward(x, w_router, w13, w2, *, kind, k, renorm, router_bias=None,
            route_scale=1.0, topk_idx=None, quant=None) -> Dict[str, np.ndarray]:
    """The whole layer forward: route -> schedule -> dispatch -> expert FFN -> combine.

    ``topk_idx`` (optional) fixes the selected experts instead of taking them from
    the router; gates are still the router's scores at those experts.
    ``quant`` (optional) is a function q(v, axis) applied to each GEMM operand
    along that GEMM's reduction axis before the GEMM (MXFP8 emulation, see
    ``mx_quantize_dequantize``).
    """
    E = w13.shape[0]
    r = route(x, w_router, router_bias, kind, k, renorm, route_scale)
    if topk_idx is not None:
        r["topk_idx"] = np.asarray(topk_idx, dtype=np.int32)
        r["gates"] = gate_values(r["scores"], r["topk_idx"], renorm, route_scale)
    s = schedule(r["topk_idx"], E)
    x_g = dispatch(x, s["src_of"], k)
    if quant is None:
        h, u, a, o = expert_ffn(x_g, s["offsets"], w13, w2)
    else:
        h, u, a, o = _expert_ffn_quant(x_g, s["offsets"], w13, w2, quant)
    y = combine(o, r["gates"], s["row_of"])
    out = dict(r)
    out.update(s)
    out.update({"x_g": x_g, "h": h, "u": u, "a": a, "o": o, "y": y})
    return out


# ---------------------------------------------------------------------------
# Backward
# ---------------------------------------------------------------------------

def dsilu(z: np.ndarray) -> np.ndarray:
    """d silu(z) / dz = sigma(z) * (1 + z * (1 - sigma(z)))."""
    sg = 1.0 / (1.0 + np.exp(-z))
    return sg * (1.0 + z * (1.0 - sg))


def router_backward(dgates, scores, topk_idx, kind, renorm, route_scale=1.0):
    """Gradient of the loss w.r.t. the router logits, selection held fixed.

    Chain rule through gate_values and router_scores, written per token with the
    explicit Jacobian of the k gates w.r.t. the E logits.  Returns dl [T][E].
    """
    T, k = topk_idx.shape
    E = scores.shape[1]
    dl = np.zeros((T, E))
    for t in range(T):
        idx = topk_idx[t].astype(np.int64)
        sel = scores[t, idx]
        # dg_j / d score_m for the k selected experts (other scores do not enter g)
        if renorm:
            S = sel.sum()
            jac_g_s = (np.eye(k) / S - sel[:, None] / S ** 2) * route_scale
        else:
            jac_g_s = np.eye(k) * route_scale
        dsel = jac_g_s.T @ dgates[t]          # d loss / d score at the selected experts
        dscore = np.zeros(E)
        dscore[idx] = dsel
        if kind == SOFTMAX:
            p = scores[t]
            jac_s_l = np.diag(p) - np.outer(p, p)   # d p_i / d l_m
        else:
            s = scores[t]
            jac_s_l = np.diag(s * (1.0 - s))
        dl[t] = jac_s_l.T @ dscore
    return dl


def backward(fwd: Dict[str, np.ndarray], dy, x, w_router, w13, w2, *, kind, k, renorm,
             route_scale=1.0, quant=None) -> Dict[str, np.ndarray]:
    """Layer backward: dX, dW_r, dW13, dW2 and d(gates), selection held fixed.

    The pages give the transfers of the backward (reverse combine pulls dY rows,
    reverse dispatch returns dX rows; [entropygate] §03 ①) and say the router-weight
    gradient is computed inside the SwiGLU backward ([wiki] benchmark section;
    [aitrending] "Technical Details").  The arithmetic is the calculus of
    ``forward``:

    * dg[t][j]  = <dA'_row, a_row>, dA' = dY[t] W2[e]   (= <dY[t], o[row]>)
    * dO_row    = g[t][j] * dY[t]
    * dW2[e]    = sum over the expert's rows of dO_row (x) a_row
    * dA_row    = dO_row W2[e]
    * dh, du    = dA * u * silu'(h), dA * silu(h)
    * dW13[e]   = sum over rows of [dh | du]_row (x) x_g[row]
    * dX[t]     = sum over j of [dh | du]_row W13[e]  +  dl[t] W_r
    * dW_r      = dl^T x, with dl from ``router_backward``.
    """
    gates, row_of, src_of, offsets = fwd["gates"], fwd["row_of"], fwd["src_of"], fwd["offsets"]
    T, H = x.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    R = T * k
    tok = src_of.astype(np.int64) // k                   # token of each sorted row
    g_row = gates.reshape(-1)[src_of.astype(np.int64)]   # gate of each sorted row
    h, u, a, o, x_g = fwd["h"], fwd["u"], fwd["a"], fwd["o"], fwd["x_g"]
    dy_g = dy[tok]

    q = quant if quant is not None else (lambda v, axis: v)
    # d(gate) of each row, computed where the pages put it, inside the SwiGLU backward:
    # <dA'_row, a_row> with dA' = dY_g W2[e] (the product the SwiGLU backward receives).  It
    # equals <dY[t], o[row]>; under MX emulation dA' is the quantised product.
    dg_row = np.zeros(R)
    dA = np.zeros((R, I))
    dw2 = np.zeros((E, H, I))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        dA_prime = q(dy_g[lo:hi], 1) @ q(w2[e], 0)               # [n][I], reduction over H
        dg_row[lo:hi] = np.einsum("ri,ri->r", dA_prime, a[lo:hi])
        dA[lo:hi] = g_row[lo:hi, None] * dA_prime
        dO = g_row[lo:hi, None] * dy_g[lo:hi]
        dw2[e] = q(dO, 0).T @ q(a[lo:hi], 0)                      # reduction over rows
    dh = dA * u * dsilu(h)
    du = dA * silu(h)
    dhu = np.concatenate([dh, du], axis=1)                       # [R][2I]
    dw13 = np.zeros((E, twoI, H))
    dx_g = np.zeros((R, H))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        dw13[e] = q(dhu[lo:hi], 0).T @ q(x_g[lo:hi], 0)          # reduction over rows
        dx_g[lo:hi] = q(dhu[lo:hi], 1) @ q(w13[e], 0)            # reduction over 2I
    dgates = np.zeros(R)
    dgates[src_of.astype(np.int64)] = dg_row
    dgates = dgates.reshape(T, k)
    dl = router_backward(dgates, fwd["scores"], fwd["topk_idx"], kind, renorm, route_scale)
    dx = np.zeros((T, H))
    rows = row_of.reshape(T, k).astype(np.int64)
    for j in range(k):
        dx += dx_g[rows[:, j]]
    dx += dl @ w_router
    dw_router = dl.T @ x
    return {"dx": dx, "dw_router": dw_router, "dw13": dw13, "dw2": dw2, "dgates": dgates,
            "dl": dl, "dhu": dhu, "dx_g": dx_g}


# ---------------------------------------------------------------------------
# MXFP8 (E4M3 elements, E8M0 scale per 32-element block)
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0
E4M3_EMAX = 8          # exponent of the largest normal, 448 = 1.75 * 2^8
E4M3_EMIN = -6         # smallest normal exponent
E4M3_MANT = 3
MX_BLOCK = 32


def round_e4m3(v: np.ndarray) -> np.ndarray:
    """Round to the nearest E4M3 value (ties to even), saturating at +-448.

    E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; normals 2^-6 .. 448,
    subnormals are multiples of 2^-9.  The quantum of a value with exponent e is
    2^(e-3) (2^-9 below 2^-6); np.rint rounds halves to even.
    """
    v = np.asarray(v, dtype=np.float64)
    mag = np.abs(v)
    _, ex = np.frexp(mag)                      # mag = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, E4M3_EMIN)          # floor(log2 mag), clamped to the subnormal range
    quantum = np.ldexp(1.0, e - E4M3_MANT)
    r = np.rint(mag / quantum) * quantum
    r = np.minimum(r, E4M3_MAX)
    return np.sign(v) * r


def mx_block_scale_exponent(amax: np.ndarray) -> np.ndarray:
    """Shared E8M0 exponent of one block: clamp(floor(log2 amax) - 8, -127, 127); amax 0 -> -127.

    OCP Microscaling v1.0 rule for E4M3 elements (emax 8); the pages only say "MXFP8".
    """
    amax = np.asarray(amax, dtype=np.float64)
    _, ex = np.frexp(amax)
    X = np.where(amax > 0, (ex - 1) - E4M3_EMAX, -127)
    return np.clip(X, -127, 127).astype(np.int64)


def mx_quantize(v: np.ndarray, axis: int) -> Tuple[np.ndarray, np.ndarray]:
    """MXFP8 quantisation of ``v`` in blocks of 32 along ``axis``.

    Returns (elements as float64 on the E4M3 grid, exponent X per block), with the
    block's value element * 2^X.  A ragged last block is padded with zeros.
    """
    v = np.moveaxis(np.asarray(v, dtype=np.float64), axis, -1)
    n = v.shape[-1]
    nb = (n + MX_BLOCK - 1) // MX_BLOCK
    pad = nb * MX_BLOCK - n
    vp = np.concatenate([v, np.zeros(v.shape[:-1] + (pad,))], axis=-1) if pad else v
    blocks = vp.reshape(v.shape[:-1] + (nb, MX_BLOCK))
    X = mx_block_scale_exponent(np.abs(blocks).max(axis=-1))
    elems = round_e4m3(blocks / np.ldexp(1.0, X)[..., None])
    elems = elems.reshape(v.shape[:-1] + (nb * MX_BLOCK,))[..., :n]
    return np.moveaxis(elems, -1, axis), np.moveaxis(X, -1, axis)


def mx_quantize_dequantize(v: np.ndarray, axis: int) -> np.ndarray:
    """Value seen by an MXFP8 GEMM: quantise in 32-blocks along ``axis``, then scale back."""
    elems, X = mx_quantize(v, axis)
    scale = np.repeat(np.ldexp(1.0, X), MX_BLOCK, axis=axis)
    n = np.asarray(v).shape[axis]
    scale = np.take(scale, np.arange(n), axis=axis)
    return elems * scale


def _expert_ffn_quant(x_g, offsets, w13, w2, q):
    """``expert_ffn`` with each GEMM operand passed through q along its reduction axis.

    [entropygate] §03 ③: MXFP8 activation quantisation sits on the dispatch, grouped
    GEMM and SwiGLU data paths.  x_g and W13 are blocked along H, a and W2 along I.
    """
    R, H = x_g.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    h = np.zeros((R, I))
    u = np.zeros((R, I))
    o = np.zeros((R, H))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        hu = q(x_g[lo:hi], 1) @ q(w13[e], 1).T
        h[lo:hi], u[lo:hi] = hu[:, :I], hu[:, I:]
    a = silu(h) * u
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        o[lo:hi] = q(a[lo:hi], 1) @ q(w2[e], 1).T
    return h, u, a, o


# ---------------------------------------------------------------------------
# Sampled evaluation for large shapes
# ---------------------------------------------------------------------------

def token_forward(x_t, w_router, router_bias, expert_weights, *, kind, k, renorm,
                  route_scale=1.0, topk_idx=None, quant=None):
    """Output of one token, computed on its own (for sampled checks at full size).

    ``expert_weights(e)`` returns (W13[e], W2[e]) as float64, so a caller can fetch
    only the experts this token uses.  ``quant`` as in ``forward`` (each GEMM operand
    quantised along that GEMM's reduction axis).  Returns (y_t, topk_idx_t, gates_t,
    o rows, scores_t).
    """
    r = route(x_t[None, :], w_router, router_bias, kind, k, renorm, route_scale)
    idx = r["topk_idx"][0] if topk_idx is None else np.asarray(topk_idx, dtype=np.int32)
    g = gate_values(r["scores"], idx[None, :], renorm, route_scale)[0]
    q = quant if quant is not None else (lambda v, axis: v)
    xq = q(x_t[None, :], 1)[0]
    y = np.zeros_like(x_t)
    outs = []
    for j in range(k):
        w13_e, w2_e = expert_weights(int(idx[j]))
        I = w13_e.shape[0] // 2
        w13_q = q(w13_e, 1)
        h = w13_q[:I] @ xq
        u = w13_q[I:] @ xq
        a = q((silu(h) * u)[None, :], 1)[0]
        o = q(w2_e, 1) @ a
        outs.append(o)
        y += g[j] * o
    return y, idx, g, outs, r["scores"][0]


def token_backward(x_t, dy_t, w_router, router_bias, expert_weights, *, kind, k, renorm,
                   route_scale=1.0, topk_idx=None, quant=None):
    """Input gradient and gate gradients of one token, computed on its own.

    The per-token part of ``backward`` (for sampled checks at full size): each step
    below is the step of ``backward`` restricted to the k rows of token t, in the same
    order and with the same operands.  For the expert j = 0..k-1 of the token:

    * h, u       = the forward's gate and up projections (``token_forward``)
    * dA'_j      = dY[t] W2[e_j]                (reduction over H)
    * dg_j       = <dA'_j, a_j>                 (the gate gradient, formed in the
                                                 SwiGLU backward: [wiki] benchmark section)
    * dA_j       = g_j dA'_j
    * dh, du     = dA_j * u * silu'(h), dA_j * silu(h)
    * dX_g row   = [dh | du] W13[e_j]           (reduction over 2I)

    then dl = ``router_backward`` of the k gate gradients and
    dX[t] = sum over j of the dX_g rows (j in order) + dl W_r.  ``quant`` as in
    ``backward``: every operand of these row GEMMs is quantised along its reduction
    axis (dY and W2[e] along H, [dh | du] and W13[e] along 2I; the forward's as in
    ``token_forward``).  ``topk_idx`` fixes the token's experts.
    Returns a dict: dx [H], dgates [k], dl [E], dhu [k][2I], dx_g [k][H], topk_idx,
    gates, y.
    """
    r = route(x_t[None, :], w_router, router_bias, kind, k, renorm, route_scale)
    idx = r["topk_idx"][0] if topk_idx is None else np.asarray(topk_idx, dtype=np.int32)
    scores = r["scores"]
    g = gate_values(scores, idx[None, :], renorm, route_scale)[0]
    q = quant if quant is not None else (lambda v, axis: v)
    xq = q(x_t[None, :], 1)[0]
    dyq = q(dy_t[None, :], 1)[0]
    y = np.zeros_like(x_t)
    dgates = np.zeros(k)
    dhu = []
    dx_g = []
    for j in range(k):
        w13_e, w2_e = expert_weights(int(idx[j]))
        I = w13_e.shape[0] // 2
        w13_f = q(w13_e, 1)
        h = w13_f[:I] @ xq
        u = w13_f[I:] @ xq
        a = silu(h) * u
        y += g[j] * (q(w2_e, 1) @ q(a[None, :], 1)[0])
        dA_prime = q(w2_e, 0).T @ dyq
        dgates[j] = dA_prime @ a
        dA = g[j] * dA_prime
        dhu_j = np.concatenate([dA * u * dsilu(h), dA * silu(h)])
        dhu.append(dhu_j)
        dx_g.append(q(dhu_j[None, :], 1)[0] @ q(w13_e, 0))
    dl = router_backward(dgates[None, :], scores, idx[None, :], kind, renorm, route_scale)[0]
    dx = np.zeros_like(x_t)
    for j in range(k):
        dx += dx_g[j]
    dx += dl @ w_router
    return {"dx": dx, "dgates": dgates, "dl": dl, "dhu": np.array(dhu), "dx_g": np.array(dx_g),
            "topk_idx": idx, "gates": g, "y": y}


def expert_weight_grads(x_rows, dy_rows, g_rows, w13_e, w2_e, *, rows13=None, rows2=None, quant=None):
    """Weight gradients of one expert from that expert's rows alone (sampled checks at full size).

    ``x_rows`` [n][H] and ``dy_rows`` [n][H] are the expert's dispatched input and
    upstream-gradient rows in schedule order (ascending assignment), ``g_rows`` [n] their
    gates.  The steps are those of ``backward`` for one expert segment:

    * h | u      = x W13[e]^T,  a = silu(h) * u
    * dA'        = dY W2[e],  dg = <dA', a> per row,  dA = g * dA'
    * dO         = g * dY,    dW2[e] = dO^T a       (reduction over the expert's rows)
    * dh | du    = dA * u * silu'(h) | dA * silu(h)
    * dW13[e]    = [dh | du]^T x                    (reduction over the expert's rows)

    ``rows13`` / ``rows2`` (optional) select output rows of dW13[e] [2I][H] and dW2[e] [H][I];
    a selected row is the same whether it is computed alone or with the rest (each output
    row reduces over the expert's rows only, and ``quant`` along the rows treats every
    column on its own).  ``quant`` as in ``backward`` (the weight-gradient operands in
    32-row blocks from the expert's first row).
    Returns a dict: dw13, dw2 (all rows or the selected ones), dg [n], dhu [n][2I].
    """
    q = quant if quant is not None else (lambda v, axis: v)
    I = w13_e.shape[0] // 2
    hu = q(x_rows, 1) @ q(w13_e, 1).T
    h, u = hu[:, :I], hu[:, I:]
    a = silu(h) * u
    dA_prime = q(dy_rows, 1) @ q(w2_e, 0)
    dg = np.einsum("ri,ri->r", dA_prime, a)
    dA = g_rows[:, None] * dA_prime
    dO = g_rows[:, None] * dy_rows
    dhu = np.concatenate([dA * u * dsilu(h), dA * silu(h)], axis=1)
    sel2 = slice(None) if rows2 is None else np.asarray(rows2, dtype=np.int64)
    sel13 = slice(None) if rows13 is None else np.asarray(rows13, dtype=np.int64)
    dw2 = q(dO[:, sel2], 0).T @ q(a, 0)
    dw13 = q(dhu[:, sel13], 0).T @ q(x_rows, 0)
    return {"dw13": dw13, "dw2": dw2, "dg": dg, "dhu": dhu}
