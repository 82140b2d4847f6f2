"""GPU parity of the layer through the C ABI against the float64 CPU oracle.

Sizes here finish in seconds on the oracle and still span several 128 x 256 tiles with
ragged expert segments (and empty experts).  Bars: the schedule table and the dispatched
rows are bit-exact; bf16 outputs and gradients meet max|err| <= 2e-2 * RMS and relative
Frobenius <= 1e-2; runs are bitwise reproducible.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_table_gb300 as mok
from mixture_experts_layer_table_gb300 import workloads as W
from oracle import moe_oracle as O
from tests.parity import assert_bf16_close, assert_intermediate_close, inputs_f64, oracle_layer, selection_is_valid, to_f64

pytestmark = pytest.mark.gpu

MID = W.MoEShape("mid_T600_H512_E16_I768_top4_sigmoid", T=600, H=512, E=16, I=768, k=4,
                 router=W.ROUTER_SIGMOID, renorm=True, x_std=1.0, w_std=0.03)
MID_SKEW = MID.scaled(name="mid_skew", skew=True)
TINY = W.TINY
ONE = W.MoEShape("T1_H256_E1_I256_top1_softmax", T=1, H=256, E=1, I=256, k=1, router=W.ROUTER_SOFTMAX,
                 renorm=False, x_std=1.0, w_std=0.05)
DENSE = W.MoEShape("dense_T300_H256_E1_I512_top1", T=300, H=256, E=1, I=512, k=1, router=W.ROUTER_SOFTMAX,
                   renorm=False, x_std=1.0, w_std=0.05)
# the largest expert count and top-k the ABI accepts: 1024 experts (most with 0-8 rows), top-16
MAXES = W.MoEShape("max_T200_H256_E1024_I256_top16_sigmoid", T=200, H=256, E=1024, I=256, k=16,
                   router=W.ROUTER_SIGMOID, renorm=True, x_std=1.0, w_std=0.05)


def _skewed_topk(T, E, k, seed, empty=(3, 9)):
    """Given selections with a hot expert and some experts never chosen."""
    rng = np.random.default_rng(seed)
    p = np.array([0.0 if e in empty else (8.0 if e == 0 else 1.0) for e in range(E)])
    p /= p.sum()
    return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)


def _gpu_inputs(inp):
    return {k: (v.cuda() if v is not None else None) for k, v in inp.items()}


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_ok):
    from mixture_experts_layer_table_gb300 import build
    build.build()
    mok.load()


def _run(shape, inp, given=None, flags=0, route_scale=1.0):
    dev = _gpu_inputs(inp)
    layer = mok.MoELayer(mok.desc_from_shape(shape, flags=flags, route_scale=route_scale))
    given_t = torch.tensor(given, dtype=torch.int32, device="cuda") if given is not None else None
    y = layer.forward(dev["x"], dev["w_router"], dev["w13"], dev["w2"], router_bias=dev["router_bias"],
                      given_topk=given_t)
    grads = layer.backward(dev["dy"], dev["x"], dev["w_router"], dev["w13"], dev["w2"])
    torch.cuda.synchronize()
    code, site = layer.status()
    assert code == 0, f"device status {code} at site {site}"
    return layer, y, grads


# ----------------------------------------------------------------------------- schedule

@pytest.mark.parametrize("T,E,k,seed", [(1, 4, 2, 0), (600, 16, 4, 1), (4096, 256, 8, 2), (777, 64, 6, 3)])
def test_schedule_bit_exact_on_given_selection(T, E, k, seed):
    idx = _skewed_topk(T, E, k, seed, empty=(1, 3) if E > 4 else ())
    ref = O.schedule(idx, E)
    desc = mok.make_desc(T, 256, 256, E, k, W.ROUTER_SIGMOID, True)
    lay = mok.get_layout(desc)
    ws = torch.zeros(lay["ws_bytes"], dtype=torch.uint8, device="cuda")
    given = torch.tensor(idx, device="cuda")
    out = {n: torch.full(s, -7, dtype=torch.int32, device="cuda") for n, s in
           (("topk_idx", (T, k)), ("counts", (E,)), ("offsets", (E + 1,)), ("row_of", (T * k,)), ("src_of", (T * k,)))}
    mok.schedule(desc, None, None, None, given, out["topk_idx"], None, out["counts"], out["offsets"], out["row_of"],
                 out["src_of"], ws)
    assert mok.read_status(ws) == (0, 0)
    assert np.array_equal(out["topk_idx"].cpu().numpy(), idx)
    for name in ("counts", "offsets", "row_of", "src_of"):
        assert np.array_equal(out[name].cpu().numpy(), ref[name]), name


def test_schedule_reports_invalid_routing():
    T, E, k = 8, 4, 2
    idx = np.array([[0, 1]] * T, dtype=np.int32)
    idx[5, 1] = E          # out of range
    idx[6] = [2, 2]        # repeated
    desc = mok.make_desc(T, 256, 256, E, k, W.ROUTER_SIGMOID, True)
    ws = torch.zeros(mok.get_layout(desc)["ws_bytes"], dtype=torch.uint8, device="cuda")
    outs = [torch.empty(s, dtype=torch.int32, device="cuda") for s in ((T, k), (E,), (E + 1,), (T * k,), (T * k,))]
    mok.schedule(desc, None, None, None, torch.tensor(idx, device="cuda"), outs[0], None, *outs[1:], ws)
    code, _ = mok.read_status(ws)
    assert code == 6
    # the table stays a valid permutation (bad entries clamped), so nothing downstream leaves its buffers
    row_of = outs[3].cpu().numpy()
    assert sorted(row_of.tolist()) == list(range(T * k))


# ----------------------------------------------------------------------------- router

@pytest.mark.parametrize("shape", [TINY, MID, MID_SKEW], ids=lambda s: s.name)
def test_router_topk_and_gates(shape):
    inp = W.make_inputs(shape, seed=0, device="cpu")
    f64 = inputs_f64(inp)
    logits, scores = O.router_scores(f64["x"], f64["w_router"], shape.router)
    sel = scores + (f64["router_bias"][None, :] if f64["router_bias"] is not None else 0.0)
    layer, _, _ = _run(shape, inp)
    gidx = layer.view("topk_idx").cpu().numpy()
    n_diff = selection_is_valid(sel, gidx, shape.k)
    assert n_diff == 0          # the seeded cases have a clear margin at the k-th score
    ref_g = O.gate_values(scores, gidx, shape.renorm)
    assert np.allclose(layer.view("gates").cpu().numpy(), ref_g, rtol=2e-5, atol=1e-7)
    assert np.allclose(layer.view("logits").cpu().numpy(), logits, rtol=1e-4, atol=1e-5)
    assert np.allclose(layer.view("scores").cpu().numpy(), scores, rtol=2e-5, atol=1e-7)


# expert counts that take the top-k kernel's other per-lane widths (2, 4 and 16 experts per lane)
ROUTER_WIDTHS = [
    W.MoEShape("router_T200_H256_E48_I256_top6_softmax", T=200, H=256, E=48, I=256, k=6,
               router=W.ROUTER_SOFTMAX, renorm=False, x_std=1.0, w_std=0.05),
    W.MoEShape("router_T200_H256_E96_I256_top8_sigmoid", T=200, H=256, E=96, I=256, k=8,
               router=W.ROUTER_SIGMOID, renorm=True, x_std=1.0, w_std=0.05),
    W.MoEShape("router_T200_H256_E300_I256_top8_sigmoid", T=200, H=256, E=300, I=256, k=8,
               router=W.ROUTER_SIGMOID, renorm=True, x_std=1.0, w_std=0.05),
]


@pytest.mark.parametrize("shape", ROUTER_WIDTHS, ids=lambda s: s.name)
def test_router_topk_at_other_expert_counts(shape):
    """The selection is a valid top-k of the oracle's scores (near-ties within the margin may
    break either way), and the gates, scores and logits match the oracle on it."""
    inp = W.make_inputs(shape, seed=0, device="cpu")
    f64 = inputs_f64(inp)
    logits, scores = O.router_scores(f64["x"], f64["w_router"], shape.router)
    layer, _, _ = _run(shape, inp)
    gidx = layer.view("topk_idx").cpu().numpy()
    selection_is_valid(scores, gidx, shape.k)
    ref_g = O.gate_values(scores, gidx, shape.renorm)
    assert np.allclose(layer.view("gates").cpu().numpy(), ref_g, rtol=2e-5, atol=1e-7)
    assert np.allclose(layer.view("logits").cpu().numpy(), logits, rtol=1e-4, atol=1e-5)
    assert np.allclose(layer.view("scores").cpu().numpy(), scores, rtol=2e-5, atol=1e-7)


# ----------------------------------------------------------------------------- forward / backward

LONG = W.MoEShape("long_T1500_H512_E8_I768_top4_sigmoid", T=1500, H=512, E=8, I=768, k=4,
                  router=W.ROUTER_SIGMOID, renorm=True, x_std=1.0, w_std=0.03)
# skewed long segments: hot experts with several full 256-row blocks, cold ones with only a tail
LONG_SKEW = LONG.scaled(name="long_skew", skew=True)
# LONG: 750 rows per expert, the expert GEMMs' 256-row chunks and GEMM1's paired form
# H and I odd multiples of 128: the last 256-row weight tile of GEMM2, dA' and dX_g reaches past the
# end (zeros loaded, nothing stored); ODD_LONG has 1500 rows per expert, where GEMM1 keeps its
# unpaired form (the paired one takes whole 256-index tiles); ODD_SHORT takes the paired GEMM2 /
# dX_g form with one 512-row tile over H = 384; EDGE128 has one CTA of each pair past the end
ODD = W.MoEShape("odd_T600_H384_E8_I640_top4_sigmoid", T=600, H=384, E=8, I=640, k=4,
                 router=W.ROUTER_SIGMOID, renorm=True, x_std=1.0, w_std=0.03)
ODD_LONG = W.MoEShape("odd_long_T1500_H384_E4_I640_top4", T=1500, H=384, E=4, I=640, k=4,
                      router=W.ROUTER_SIGMOID, renorm=True, x_std=1.0, w_std=0.03)
ODD_SHORT = W.MoEShape("odd_short_T256_H384_E16_I640_top4", T=256, H=384, E=16, I=640, k=4,
                       router=W.ROUTER_SIGMOID, renorm=True, x_std=1.0, w_std=0.03, skew=True)
EDGE128 = W.MoEShape("edge_T100_H128_E4_I128_top2_softmax", T=100, H=128, E=4, I=128, k=2,
                     router=W.ROUTER_SOFTMAX, renorm=False, x_std=1.0, w_std=0.05)
CASES = [(TINY, None), (MID, None), (MID_SKEW, None), (MID, "skewed_given"), (ONE, None), (DENSE, None),
         (MAXES, None), (LONG, None), (LONG_SKEW, None), (ODD, None), (ODD_LONG, None), (ODD_SHORT, None),
         (EDGE128, None)]


@pytest.mark.parametrize("shape,mode", CASES, ids=lambda c: getattr(c, "name", str(c)))
def test_forward_backward_parity(shape, mode):
    inp = W.make_inputs(shape, seed=0, device="cpu")
    f64 = inputs_f64(inp)
    if mode == "skewed_given":
        given = _skewed_topk(shape.T, shape.E, shape.k, seed=5)
    else:
        given = O.route(f64["x"], f64["w_router"], f64["router_bias"], shape.router, shape.k, shape.renorm)["topk_idx"]
    fwd, bwd = oracle_layer(shape, f64, topk_idx=given)
    layer, y, g = _run(shape, inp, given=given)
    # schedule and dispatch: exact
    for name in ("counts", "offsets", "row_of", "src_of"):
        assert np.array_equal(layer.view(name).cpu().numpy(), fwd[name]), name
    assert np.array_equal(to_f64(layer.view("x_g")), fwd["x_g"])
    # forward intermediates (fp32, or bf16 hi + lo pairs) and output
    hu = to_f64(layer.view("hu"))
    assert_intermediate_close(hu[:, :shape.I], fwd["h"], "h", rel=1e-4)
    assert_intermediate_close(hu[:, shape.I:], fwd["u"], "u", rel=1e-4)
    assert_intermediate_close(to_f64(layer.view_split("act")), fwd["a"], "a", rel=1e-3)
    assert_intermediate_close(to_f64(layer.view("expert_out")), fwd["o"], "o", rel=1e-3)
    assert_bf16_close(to_f64(y), fwd["y"], "y")
    # backward
    assert_intermediate_close(to_f64(layer.view_split("dhu")), bwd["dhu"], "dhu", rel=1e-3)
    assert_intermediate_close(to_f64(layer.view("dx_g")), bwd["dx_g"], "dx_g", rel=1e-3)
    assert_bf16_close(to_f64(g["dgates"]), bwd["dgates"], "dgates")
    assert_bf16_close(to_f64(g["dw2"]), bwd["dw2"], "dw2")
    assert_bf16_close(to_f64(g["dw13"]), bwd["dw13"], "dw13")
    assert_bf16_close(to_f64(g["dw_router"]), bwd["dw_router"], "dw_router")
    assert_bf16_close(to_f64(g["dx"]), bwd["dx"], "dx")


@pytest.mark.parametrize("shape,scale", [(MID_SKEW, 2.5), (TINY, 0.7)], ids=lambda c: getattr(c, "name", str(c)))
def test_route_scale(shape, scale):
    """A route scale other than 1 (the gates times a constant after any renormalisation): gates,
    y and every gradient against the oracle with the same scale."""
    inp = W.make_inputs(shape, seed=0, device="cpu")
    f64 = inputs_f64(inp)
    fwd, bwd = oracle_layer(shape, f64, route_scale=scale)
    layer, y, g = _run(shape, inp, route_scale=scale)
    assert np.array_equal(layer.view("topk_idx").cpu().numpy(), fwd["topk_idx"])
    assert np.allclose(layer.view("gates").cpu().numpy(), fwd["gates"], rtol=2e-5, atol=1e-7)
    assert_bf16_close(to_f64(y), fwd["y"], "y")
    for name in ("dgates", "dw_router", "dw2", "dw13", "dx"):
        assert_bf16_close(to_f64(g[name]), bwd[name], name)


@pytest.mark.parametrize("shape,mode", [(MID, None), (MID, "skewed_given"), (TINY, None), (ODD, None),
                                        (EDGE128, None)],
                         ids=lambda c: getattr(c, "name", str(c)))
def test_row_tile_gemms_forward_backward(shape, mode):
    """MOK_FLAG_GEMM_SINGLE: the expert GEMMs on the 128-row-tile single-CTA kernels and the weight
    gradients on single CTAs (128 x 128 tiles) instead of the CTA-pair kernels; o, y, dX_g, dX,
    dW2 and dW13 against the oracle."""
    from mixture_experts_layer_table_gb300 import _native as N
    inp = W.make_inputs(shape, seed=0, device="cpu")
    f64 = inputs_f64(inp)
    if mode == "skewed_given":
        given = _skewed_topk(shape.T, shape.E, shape.k, seed=5)
    else:
        given = O.route(f64["x"], f64["w_router"], f64["router_bias"], shape.router, shape.k, shape.renorm)["topk_idx"]
    fwd, bwd = oracle_layer(shape, f64, topk_idx=given)
    layer, y, g = _run(shape, inp, given=given, flags=N.FLAG_GEMM_SINGLE)
    assert_intermediate_close(to_f64(layer.view("expert_out")), fwd["o"], "o", rel=1e-3)
    assert_bf16_close(to_f64(y), fwd["y"], "y")
    assert_intermediate_close(to_f64(layer.view("dx_g")), bwd["dx_g"], "dx_g", rel=1e-3)
    assert_bf16_close(to_f64(g["dx"]), bwd["dx"], "dx")
    assert_bf16_close(to_f64(g["dw2"]), bwd["dw2"], "dw2")
    assert_bf16_close(to_f64(g["dw13"]), bwd["dw13"], "dw13")


@pytest.mark.parametrize("shape", [MID, MID_SKEW], ids=lambda s: s.name)
def test_bf16_weight_gradients_are_rounded_fp32_ones(shape):
    """MOK_FLAG_WGRAD_BF16 stores dW13 / dW2 in bf16.  The kernels and reduction order are the
    same as the default fp32 output, so the result must be that fp32 result rounded to nearest
    even, bit for bit (the fp32 result itself meets the bar against the oracle above).  Pure
    bf16 rounding of an exact gradient alone moves its largest elements by up to 2^-8 of
    their size, about 2% of the RMS at 5 sigma, so the max-error bar is not asked of bf16."""
    inp = W.make_inputs(shape, seed=0, device="cpu")
    f64 = inputs_f64(inp)
    given = O.route(f64["x"], f64["w_router"], f64["router_bias"], shape.router, shape.k, shape.renorm)["topk_idx"]
    _, g32 = _run(shape, inp, given=given)[1:]
    dev = _gpu_inputs(inp)
    layer = mok.MoELayer(mok.desc_from_shape(shape, flags=1))
    layer.forward(dev["x"], dev["w_router"], dev["w13"], dev["w2"], router_bias=dev["router_bias"],
                  given_topk=torch.tensor(given, device="cuda"))
    g = layer.backward(dev["dy"], dev["x"], dev["w_router"], dev["w13"], dev["w2"])
    torch.cuda.synchronize()
    assert g["dw13"].dtype == torch.bfloat16 and layer.status() == (0, 0)
    for name in ("dw13", "dw2"):
        assert torch.equal(g[name], g32[name].to(torch.bfloat16)), name
    for name in ("dx", "dw_router", "dgates"):
        assert torch.equal(g[name], g32[name]), name


def test_weight_gradients_pair_and_single_bitwise_with_a_hot_expert():
    """The pair kernel deals its strips back and forth over the pairs, the single-CTA kernel from a
    counter: with a hot expert and an empty one the weight gradients are bitwise the same."""
    from mixture_experts_layer_table_gb300 import _native as N
    shape = MID_SKEW
    inp = W.make_inputs(shape, seed=2, device="cpu")
    given = _skewed_topk(shape.T, shape.E, shape.k, seed=11, empty=(5,))
    _, _, g = _run(shape, inp, given=given)
    _, _, g1 = _run(shape, inp, given=given, flags=N.FLAG_GEMM_SINGLE)
    for name in ("dw13", "dw2"):
        assert torch.equal(g[name], g1[name]), name


@pytest.mark.parametrize("T", [1200, 1199])
def test_weight_gradients_of_long_experts_on_odd_strips(T):
    """Every token takes all four experts, so each expert has T rows: far more than the pair
    kernel's three stationary K blocks, so its tiles are dealt two at a time.  With H = 768 a dW13
    strip has three tiles (its last item one tile); T = 1200 has no K block ending inside an MMA
    K step, T = 1199 has one per expert.  The pair kernel is bitwise the single-CTA kernel and
    both meet the bar against the oracle."""
    from mixture_experts_layer_table_gb300 import _native as N
    shape = W.MoEShape(f"odd_strip_T{T}_H768_E4_I512_top4", T=T, H=768, E=4, I=512, k=4,
                       router=W.ROUTER_SIGMOID, renorm=True, x_std=1.0, w_std=0.03)
    inp = W.make_inputs(shape, seed=6, device="cpu")
    f64 = inputs_f64(inp)
    given = np.tile(np.arange(4, dtype=np.int32), (T, 1))
    _, bwd = oracle_layer(shape, f64, topk_idx=given)
    _, _, g = _run(shape, inp, given=given)
    _, _, g1 = _run(shape, inp, given=given, flags=N.FLAG_GEMM_SINGLE)
    for name in ("dw13", "dw2"):
        assert torch.equal(g[name], g1[name]), name
        assert_bf16_close(to_f64(g[name]), bwd[name], name)


def test_empty_experts_get_zero_weight_gradient():
    shape = MID
    inp = W.make_inputs(shape, seed=1, device="cpu")
    given = _skewed_topk(shape.T, shape.E, shape.k, seed=7, empty=(3, 9))
    _, _, g = _run(shape, inp, given=given)
    for e in (3, 9):
        assert torch.count_nonzero(g["dw13"][e]) == 0 and torch.count_nonzero(g["dw2"][e]) == 0
        assert torch.count_nonzero(g["dw_router"][e]) == 0


def test_bitwise_deterministic():
    shape = MID_SKEW
    inp = W.make_inputs(shape, seed=3, device="cpu")
    outs = []
    for _ in range(2):
        layer, y, g = _run(shape, inp)
        outs.append([y.clone()] + [g[n].clone() for n in ("dx", "dw_router", "dw13", "dw2", "dgates")] +
                    [layer.view(n).clone() for n in ("topk_idx", "row_of", "hu")])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_repeated_backward_on_one_layer_single_cta_kernels():
    """The single-CTA weight-gradient kernels deal their strips from counters in the workspace;
    each backward call clears them, so repeated backward calls on one layer object (same
    workspace) give the same gradients bit for bit, and the forward's status word survives."""
    from mixture_experts_layer_table_gb300 import _native as N
    shape = MID_SKEW
    inp = W.make_inputs(shape, seed=4, device="cpu")
    dev = _gpu_inputs(inp)
    layer = mok.MoELayer(mok.desc_from_shape(shape, flags=N.FLAG_GEMM_SINGLE))
    layer.forward(dev["x"], dev["w_router"], dev["w13"], dev["w2"], router_bias=dev["router_bias"])
    grads = []
    for _ in range(3):
        g = layer.backward(dev["dy"], dev["x"], dev["w_router"], dev["w13"], dev["w2"])
        grads.append({n: g[n].clone() for n in ("dx", "dw13", "dw2")})
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    for g in grads[1:]:
        for n in ("dx", "dw13", "dw2"):
            assert torch.equal(g[n], grads[0][n]), n


# ----------------------------------------------------------------------------- CTA-pair GEMMs

# long expert segments (~750 rows: several 256-row pair tiles and a ragged one per expert)
PAIR_CASES = [(LONG, None), (LONG_SKEW, None), (LONG, "skewed_given"), (MID, None), (MID, "skewed_given"),
              (TINY, None), (ONE, None), (ODD_LONG, None), (EDGE128, None)]


@pytest.mark.parametrize("shape,mode", PAIR_CASES, ids=lambda c: getattr(c, "name", str(c)))
def test_pair_gemm_forward(shape, mode):
    """Forward expert GEMMs on CTA pairs (tcgen05 cta_group::2, 256-row tiles split over two
    SMs): h|u, a, o and y against the oracle, and bitwise equal to the single-CTA GEMMs."""
    from mixture_experts_layer_table_gb300 import _native as N
    inp = W.make_inputs(shape, seed=0, device="cpu")
    f64 = inputs_f64(inp)
    if mode == "skewed_given":
        given = _skewed_topk(shape.T, shape.E, shape.k, seed=5)
    else:
        given = O.route(f64["x"], f64["w_router"], f64["router_bias"], shape.router, shape.k, shape.renorm)["topk_idx"]
    fwd, _ = oracle_layer(shape, f64, topk_idx=given)
    dev = _gpu_inputs(inp)
    given_t = torch.tensor(given, dtype=torch.int32, device="cuda")
    outs = {}
    # default flags: GEMM2 on the narrow-segment pair kernel (expert rows as the MMA's N)
    for name, flag in (("pair", N.FLAG_GEMM_PAIR), ("single", N.FLAG_GEMM_SINGLE), ("narrow", 0)):
        layer = mok.MoELayer(mok.desc_from_shape(shape, flags=flag))
        y = layer.forward(dev["x"], dev["w_router"], dev["w13"], dev["w2"], router_bias=dev["router_bias"],
                          given_topk=given_t)
        torch.cuda.synchronize()
        assert layer.status() == (0, 0)
        outs[name] = {"y": y.clone(), "hu": layer.view("hu").clone(), "act": layer.view_split("act").clone(),
                      "o": layer.view("expert_out").clone()}
    p = outs["pair"]
    hu = to_f64(p["hu"])
    assert_intermediate_close(hu[:, :shape.I], fwd["h"], "h", rel=1e-4)
    assert_intermediate_close(hu[:, shape.I:], fwd["u"], "u", rel=1e-4)
    assert_intermediate_close(to_f64(p["act"]), fwd["a"], "a", rel=1e-3)
    assert_intermediate_close(to_f64(p["o"]), fwd["o"], "o", rel=1e-3)
    assert_bf16_close(to_f64(p["y"]), fwd["y"], "y")
    for name in ("hu", "act", "o", "y"):
        assert torch.equal(p[name], outs["single"][name]), name
    nw = outs["narrow"]
    assert_intermediate_close(to_f64(nw["o"]), fwd["o"], "o (narrow)", rel=1e-3)
    assert_bf16_close(to_f64(nw["y"]), fwd["y"], "y (narrow)")
    for name in ("hu", "act"):
        assert torch.equal(nw[name], outs["single"][name]), name


# ----------------------------------------------------------------------------- bounded waits

def test_stuck_wait_times_out_and_context_survives():
    desc = mok.desc_from_shape(TINY)
    ws = torch.zeros(mok.get_layout(desc)["ws_bytes"], dtype=torch.uint8, device="cuda")
    from mixture_experts_layer_table_gb300 import _native as N
    N.test_bounded_wait(ws, 50)
    code, site = mok.read_status(ws)
    assert code == 5 and site == 30
    # the context is still usable afterwards
    inp = W.make_inputs(TINY, seed=0, device="cpu")
    _run(TINY, inp)


# ----------------------------------------------------------------------------- ring forward

@pytest.mark.parametrize("shape,minibatch,slots,comm,flags", [
    (MID, 300, 2, 4, 0),        # ragged minibatches (not a multiple of 128), the ring wraps 4 times
    (MID, 1024, 1, 8, 0),       # one slot: gathering and GEMM1 alternate
    (MID_SKEW, 700, 3, 2, 0),   # skewed experts cut at minibatch edges
    (TINY, 96, 2, 2, 0),        # tiny layer, softmax router
    (LONG, 3000, 2, 6, 0),      # 750 rows per expert: chunks of up to 256 rows cut at minibatch edges
    (LONG, 700, 3, 4, 0),       # the paired SwiGLU GEMM1 (>= 384 rows per expert) on ragged cuts
    (LONG_SKEW, 1000, 2, 2, 0),  # paired GEMM1, hot and cold experts cut at minibatch edges
    (MID, 300, 2, 3, "single"),  # the row-tile ring kernel (one CTA per 128-row tile), odd comm count
    (MID_SKEW, 700, 2, 4, "pair"),  # the row-tile ring kernel under the CTA-pair flag
    (ODD, 500, 2, 4, 0),        # H and I odd multiples of 128
    # GEMM2 and the merge in the persistent launch too (every GEMM1 / GEMM2 form pairing)
    (MID, 300, 2, 4, "persistent"),        # unpaired GEMM1, paired GEMM2 (short rows)
    (MID_SKEW, 700, 3, 2, "persistent"),   # skewed experts cut at minibatch edges
    (LONG, 700, 3, 4, "persistent"),       # paired SwiGLU GEMM1, unpaired GEMM2
    (LONG_SKEW, 1000, 2, 6, "persistent"),
    (TINY, 96, 2, 2, "persistent"),        # tiny layer, softmax router, top-2
    (ODD, 500, 2, 4, "persistent"),        # ragged last weight tiles
], ids=lambda v: getattr(v, "name", str(v)))
def test_ring_forward_is_bitwise_the_plain_forward(shape, minibatch, slots, comm, flags):
    """The ring forward (persistent launch: gathering CTAs fill ring slots while GEMM CTAs run
    GEMM1 on earlier minibatches; GEMM1 on the narrow-segment CTA-pair kernel by default, on the
    row-tile kernel under the row-tile flags) computes every row exactly as the plain forward does,
    so y, h|u and a must be bitwise equal; the backward after a ring forward must match too."""
    flags = {0: 0, "single": mok.FLAG_GEMM_SINGLE, "pair": mok.FLAG_GEMM_PAIR,
             "persistent": mok.FLAG_RING_PERSISTENT}[flags]
    inp = W.make_inputs(shape, seed=0, device="cpu")
    dev = _gpu_inputs(inp)
    plain = mok.MoELayer(mok.desc_from_shape(shape, flags=flags))
    y0 = plain.forward(dev["x"], dev["w_router"], dev["w13"], dev["w2"], router_bias=dev["router_bias"])
    g0 = plain.backward(dev["dy"], dev["x"], dev["w_router"], dev["w13"], dev["w2"])
    ring_bytes = slots * minibatch * shape.H * 2
    ring = mok.MoELayer(mok.desc_from_shape(shape, minibatch=minibatch, ring_bytes=ring_bytes, comm_sms=comm,
                                            flags=flags))
    assert ring.layout["ring"] >= 0
    for _ in range(2):  # the second call reuses the ring and the counters
        y1 = ring.forward(dev["x"], dev["w_router"], dev["w13"], dev["w2"], router_bias=dev["router_bias"])
        torch.cuda.synchronize()
        assert ring.status() == (0, 0)
        assert torch.equal(y1, y0)
        assert torch.equal(ring.view("hu"), plain.view("hu"))
        assert torch.equal(ring.view("act"), plain.view("act"))
        assert torch.equal(ring.view("expert_out"), plain.view("expert_out"))
    g1 = ring.backward(dev["dy"], dev["x"], dev["w_router"], dev["w13"], dev["w2"])
    torch.cuda.synchronize()
    assert ring.status() == (0, 0)
    for name in ("dx", "dw_router", "dw13", "dw2", "dgates"):
        assert torch.equal(g1[name], g0[name]), name


def test_ring_backward_reuses_the_resident_minibatches():
    """The ring-based backward: after a ring forward the ring still holds its last minibatches at
    their own rows of the dispatched-row region, and the backward gathers again only the rows in
    front of them.  Shown by handing the backward another x: the replayed rows come from it, the
    resident ones are still the forward's.  With a fresh workspace (stamp mismatch) every row is
    replayed.  The stamp in ws names the forward's ctx and its count of ring forwards."""
    shape, minibatch, slots = MID, 300, 2
    inp = W.make_inputs(shape, seed=0, device="cpu")
    dev = _gpu_inputs(inp)
    desc = mok.desc_from_shape(shape, minibatch=minibatch, ring_bytes=slots * minibatch * shape.H * 2, comm_sms=4)
    ring = mok.MoELayer(desc)
    ring.forward(dev["x"], dev["w_router"], dev["w13"], dev["w2"])
    torch.cuda.synchronize()
    assert ring.status() == (0, 0)
    R = shape.R
    n_mb = -(-R // minibatch)
    head = (n_mb - slots) * minibatch
    stamp_ws = ring.ws[ring.layout["mb_counters"]:].view(torch.int32)
    off = (((2 * n_mb + 1) * 4 + 15) // 16) * 4  # the u64 stamp after the counters, in int32 units
    stamp = stamp_ws[off:off + 4].view(torch.int64).cpu().tolist()
    assert stamp == [ring.ctx.data_ptr(), int(ring.view("ring_stamp")[0])]
    src = ring.view("src_of").cpu().numpy().astype(np.int64) // shape.k
    x2 = dev["x"] + 1.0                                            # another x for the backward
    ring.backward(dev["dy"], x2, dev["w_router"], dev["w13"], dev["w2"])
    torch.cuda.synchronize()
    rows = ring.view("ring")[:R].float().cpu()
    x_cpu, x2_cpu = dev["x"].float().cpu(), x2.float().cpu()
    assert torch.equal(rows[:head], x2_cpu[src[:head]])          # replayed from the backward's x
    assert torch.equal(rows[head:], x_cpu[src[head:]])           # still the forward's rows
    fresh = mok.MoELayer(desc)
    fresh.ctx.copy_(ring.ctx)                                      # the forward's ctx, another ws
    fresh_ctx_stamp = fresh.view("ring_stamp").clone()
    fresh.backward(dev["dy"], x2, dev["w_router"], dev["w13"], dev["w2"])
    torch.cuda.synchronize()
    assert torch.equal(fresh.view("ring")[:R].float().cpu(), x2_cpu[src])
    assert torch.equal(fresh.view("ring_stamp"), fresh_ctx_stamp)  # the backward does not touch ctx


def test_ring_rejects_a_ring_smaller_than_one_minibatch():
    shape = MID
    desc = mok.desc_from_shape(shape, minibatch=512, ring_bytes=511 * shape.H * 2)
    with pytest.raises(mok.MokError) as info:
        mok.get_layout(desc)
    assert info.value.code == 2


def test_ring_rejects_an_odd_comm_count_on_the_pair_kernel():
    """The narrow-segment ring kernel launches its gathering CTAs in clusters of two: an odd
    comm_sms is an invalid argument there (and fine on the row-tile kernel, covered above)."""
    shape = MID
    inp = _gpu_inputs(W.make_inputs(shape, seed=0, device="cpu", with_dy=False))
    layer = mok.MoELayer(mok.desc_from_shape(shape, minibatch=300, ring_bytes=600 * shape.H * 2, comm_sms=3))
    with pytest.raises(mok.MokError) as info:
        layer.forward(inp["x"], inp["w_router"], inp["w13"], inp["w2"])
    assert info.value.code == 1


# ----------------------------------------------------------------------------- fp16 W2 (MOK_FLAG_W2_F16)

@pytest.mark.parametrize("shape", [MID, MID_SKEW, LONG, LONG_SKEW, ODD, ODD_SHORT], ids=lambda c: c.name)
def test_forward_with_fp16_w2(shape):
    """The forward on an fp16 copy of W2 with a kept as one fp16 value (GEMM1's SwiGLU epilogue in
    both forms: LONG has 750 rows per expert, the paired form): a is the fp16 rounding of the GPU's
    own silu(h) u, the expert outputs and y meet the bars against the float64 oracle on the bf16
    weights, and the backward (bf16 W2) is unchanged."""
    inp = W.make_inputs(shape, seed=0, device="cpu")
    f64 = inputs_f64(inp)
    given = O.route(f64["x"], f64["w_router"], f64["router_bias"], shape.router, shape.k, shape.renorm)["topk_idx"]
    fwd, bwd = oracle_layer(shape, f64, topk_idx=given)
    dev = _gpu_inputs(inp)
    w2_f16 = mok.convert_f16(dev["w2"])
    w32, h32 = dev["w2"].float(), w2_f16.float()
    big = w32.abs() >= 2.0 ** -14                                      # fp16 normals: exact
    assert torch.equal(h32[big], w32[big])
    assert float((h32 - w32).abs().max()) <= 2.0 ** -25                # subnormals: half a step
    layer = mok.MoELayer(mok.desc_from_shape(shape, flags=mok.FLAG_W2_F16))
    given_t = torch.tensor(given, dtype=torch.int32, device="cuda")
    y = layer.forward(dev["x"], dev["w_router"], dev["w13"], w2_f16, router_bias=dev["router_bias"], given_topk=given_t)
    grads = layer.backward(dev["dy"], dev["x"], dev["w_router"], dev["w13"], dev["w2"])
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    hu = layer.view("hu").double()
    a_gpu = (hu[:, :shape.I] / (1 + torch.exp(-hu[:, :shape.I])) * hu[:, shape.I:]).float()
    a16 = layer.view("act").view(torch.float16)
    assert torch.allclose(a16.float(), a_gpu.half().float(), rtol=2.0 ** -10, atol=1e-30)
    assert_intermediate_close(to_f64(a16), fwd["a"], "a (fp16)", rel=2.0 ** -10)
    assert_intermediate_close(to_f64(layer.view("expert_out")), fwd["o"], "o", rel=1e-3)
    assert_bf16_close(to_f64(y), fwd["y"], "y")
    for name in ("dx", "dw13", "dw2", "dgates", "dw_router"):
        assert_bf16_close(to_f64(grads[name]), bwd[name], name)


def test_fp16_w2_refused_with_ring_and_row_tiles():
    d_ring = mok.desc_from_shape(MID, flags=mok.FLAG_W2_F16, minibatch=256, ring_bytes=8 << 20)
    d_rows = mok.desc_from_shape(MID, flags=mok.FLAG_W2_F16 | mok.FLAG_GEMM_SINGLE)
    inp = _gpu_inputs(W.make_inputs(MID, seed=0, device="cpu", with_dy=False))
    w2_f16 = mok.convert_f16(inp["w2"])
    for d in (d_ring, d_rows):
        layer = mok.MoELayer(d)
        with pytest.raises(mok.MokError) as err:
            layer.forward(inp["x"], inp["w_router"], inp["w13"], w2_f16)
        assert err.value.code == 2
