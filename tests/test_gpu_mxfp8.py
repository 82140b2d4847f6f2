"""MXFP8 forward and backward on the GPU against the oracle's MX emulation (quantise every GEMM operand in
32-element blocks along that GEMM's reduction axis, then multiply in float64).

Bars: the quantised weights (E4M3 bytes and E8M0 scales) and the quantised dispatched rows are
bit-exact against the oracle's quantiser; the layer output is within relative Frobenius 5e-2 of
the MX-emulating oracle (in practice far closer: only the quantisation of a, whose input the
GPU computes in fp32, can fall on the other side of a rounding boundary).
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_table_gb300 as mok
from mixture_experts_layer_table_gb300 import workloads as W
from oracle import moe_oracle as O
from tests.parity import (check_sampled_expert_wgrads, check_sampled_token_backward, clear_margin_tokens,
                          err_stats, inputs_f64, to_f64)

pytestmark = pytest.mark.gpu

MX_FRO = 5e-2
MID = W.MoEShape("mid_mx_T600_H512_E16_I768_top4", T=600, H=512, E=16, I=768, k=4, router=W.ROUTER_SIGMOID,
                 renorm=True, x_std=1.0, w_std=0.03, mxfp8=True)
# H and I odd multiples of 128: the last 256-row pair tile of GEMM2, dA' and dX_g reaches past the
# end, the row quantisers see half-width chunks
ODD = W.MoEShape("odd_mx_T600_H384_E8_I640_top4", T=600, H=384, E=8, I=640, k=4, router=W.ROUTER_SIGMOID,
                 renorm=True, x_std=1.0, w_std=0.03, mxfp8=True)
q = O.mx_quantize_dequantize


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_ok):
    from mixture_experts_layer_table_gb300 import build
    build.build()
    mok.load()


def _sf_byte(r, kb):
    """Byte of (row r, 32-element block kb) in a 512-byte scale block: 128 rows x 4 blocks, row
    32 j + l and block b at byte 16 l + 4 j + b (the order the tensor cores read from TMEM)."""
    return (r % 32) * 16 + ((r // 32) % 4) * 4 + kb % 4


def _decode_w(qb, sb, N, K, gate_up_I=0):
    """E4M3 bytes [E, N, K] and scale blocks [E, N/128, K/128, 512] -> (float64 values [E, N, K],
    exponents [E, N, K/32]).  gate_up_I > 0 (W13, N = 2I): block t holds the gate rows 64 t .. +63
    (block rows 0..63) and the up rows I + 64 t .. +63 (block rows 64..127)."""
    vals = qb.view(torch.float8_e4m3fn).double().cpu().numpy()
    blocks = sb.cpu().numpy().astype(np.int64).reshape(qb.shape[0], N // 128, K // 128, 512)
    n = np.arange(N)[:, None]
    kb = np.arange(K // 32)[None, :]
    if gate_up_I:
        tile, local = (n % gate_up_I) // 64, (n // gate_up_I) * 64 + n % 64
    else:
        tile, local = n // 128, n % 128
    X = blocks[:, tile, kb // 4, _sf_byte(local, kb)] - 127               # [E, N, K/32]
    return np.ldexp(vals, np.repeat(X, 32, axis=-1)), X


def _decode_rows(layer, xq_name, sf_name, K, prows):
    """Rows `prows` of an E4M3 row operand of the MXFP8 forward (padded row space) and their scales:
    (float64 values [n, K], exponents [n, K/32]).  Every row's scales are stored in four blocks (row
    groups p/32 - 3 .. p/32); all four copies must agree."""
    vals = layer.view(xq_name)[torch.as_tensor(prows, device="cuda")].view(torch.float8_e4m3fn).double().cpu().numpy()
    blocks = layer.view(sf_name).cpu().numpy().astype(np.int64)            # [G, K/128, 512]
    p = np.asarray(prows)[:, None]
    kb = np.arange(K // 32)[None, :]
    X = blocks[p // 32, kb // 4, (p % 32) * 16 + kb % 4] - 127
    for jj in (1, 2, 3):
        ok = p // 32 - jj >= 0
        Xj = blocks[np.maximum(p // 32 - jj, 0), kb // 4, (p % 32) * 16 + jj * 4 + kb % 4] - 127
        assert np.all((Xj == X) | ~ok), f"scale copy {jj} disagrees"
    return np.ldexp(vals, np.repeat(X, 32, axis=-1)), X


def _padded_rows(layer, shape):
    """Padded row of each schedule-order row, and the padding rows (expert rows padded to 32)."""
    off = layer.view("offsets").cpu().numpy().astype(np.int64)
    blk = layer.view("mx_blk_off").cpu().numpy().astype(np.int64)
    assert np.array_equal(blk[1:] - blk[:-1], (off[1:] - off[:-1] + 31) // 32)
    rows, pads = [], []
    for e in range(shape.E):
        n = off[e + 1] - off[e]
        rows.append(32 * blk[e] + np.arange(n))
        pads.append(32 * blk[e] + np.arange(n, 32 * (blk[e + 1] - blk[e])))
    return np.concatenate(rows), np.concatenate(pads)


def _run_mx(shape, inp, given=None):
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    desc = mok.desc_from_shape(shape)
    wq = mok.quantize_weights(desc, dev["w13"], dev["w2"])
    layer = mok.MoELayer(desc)
    y = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
    g = torch.tensor(given, dtype=torch.int32, device="cuda") if given is not None else None
    mok.moe_forward_mxfp8(desc, dev["x"], dev["w_router"], dev["router_bias"], g, wq, y, layer.ctx, layer.ws)
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    return layer, y, wq


@pytest.mark.parametrize("shape", [MID, ODD], ids=lambda s: s.name)
def test_quantized_weights_bit_exact(shape):
    inp = W.make_inputs(shape, seed=0, device="cpu")
    f64 = inputs_f64(inp)
    _, _, wq = _run_mx(shape, inp)
    for name, w, N, K, gu in (("w13", f64["w13"], 2 * shape.I, shape.H, shape.I),
                              ("w2", f64["w2"], shape.H, shape.I, 0)):
        got, X_got = _decode_w(wq[name + "_q"], wq[name + "_scale"], N, K, gu)
        for e in range(shape.E):
            want = q(w[e], 1)
            bad = np.argwhere(got[e] != want)
            assert bad.size == 0, (name, e, len(bad), [(tuple(b), got[e][tuple(b)], want[tuple(b)], w[e][tuple(b)])
                                                       for b in bad[:4]])
            _, X = O.mx_quantize(w[e], 1)
            assert np.array_equal(X_got[e], X), (name, e)


@pytest.mark.parametrize("shape", [MID, MID.scaled(name="mid_mx_skew", skew=True), ODD], ids=lambda s: s.name)
def test_mx_forward_matches_mx_oracle(shape):
    inp = W.make_inputs(shape, seed=0, device="cpu")
    f64 = inputs_f64(inp)
    given = O.route(f64["x"], f64["w_router"], f64["router_bias"], shape.router, shape.k, shape.renorm)["topk_idx"]
    fwd = O.forward(f64["x"], f64["w_router"], f64["w13"], f64["w2"], kind=shape.router, k=shape.k,
                    renorm=shape.renorm, router_bias=f64["router_bias"], topk_idx=given, quant=q)
    layer, y, _ = _run_mx(shape, inp, given)
    # the dispatched rows are quantised in the gather into E4M3 bytes and scale blocks at their
    # padded rows: bit-exact against the oracle's quantiser (elements and exponents); the padding
    # rows are zero
    prows, pads = _padded_rows(layer, shape)
    xg, Xg = _decode_rows(layer, "mx_xq", "mx_xsf", shape.H, prows)
    assert np.array_equal(xg, q(fwd["x_g"], 1))
    assert np.array_equal(Xg, O.mx_quantize(fwd["x_g"], 1)[1])
    if len(pads):
        zp, _ = _decode_rows(layer, "mx_xq", "mx_xsf", shape.H, pads)
        assert not np.any(zp)
    # a = silu(h) u quantised along I by the GEMM1 epilogue: against the oracle's quantiser applied
    # to a computed from the GPU's own h | u (only a value on a rounding boundary can differ)
    hu_gpu = to_f64(layer.view("hu"))
    a_gpu = O.silu(hu_gpu[:, :shape.I]) * hu_gpu[:, shape.I:]
    ag, _ = _decode_rows(layer, "mx_aq", "mx_asf", shape.I, prows)
    _, _, fro_a = err_stats(ag, q(a_gpu, 1))
    assert fro_a <= 1e-3, fro_a
    if len(pads):
        zp, _ = _decode_rows(layer, "mx_aq", "mx_asf", shape.I, pads)
        assert not np.any(zp)
    _, _, fro = err_stats(to_f64(y), fwd["y"])
    assert fro <= MX_FRO, fro
    # h | u come from exact products of MX-grid operands: close to the oracle's
    hu = to_f64(layer.view("hu"))
    _, _, fro_h = err_stats(hu[:, :shape.I], fwd["h"])
    assert fro_h <= 1e-5, fro_h
    # against the unquantised layer (reported, not a bar): the MX quantisation error itself
    ref = O.forward(f64["x"], f64["w_router"], f64["w13"], f64["w2"], kind=shape.router, k=shape.k,
                    renorm=shape.renorm, router_bias=f64["router_bias"], topk_idx=given)
    print("MXFP8 vs unquantised: rel fro %.3e" % err_stats(to_f64(y), ref["y"])[2])


@pytest.mark.slow
def test_mx_forward_full_size_sampled_and_deterministic():
    shape = W.DSV3_MXFP8
    inp = W.make_inputs(shape, seed=0, device="cuda", with_dy=False)
    layer, y, wq = _run_mx(shape, inp)
    _, y2, _ = _run_mx(shape, inp)
    assert torch.equal(y, y2)
    w_r = to_f64(inp["w_router"])
    gpu_idx = layer.view("topk_idx").cpu().numpy()
    cache = {}

    def experts(e):
        if e not in cache:
            if len(cache) > 8:
                cache.pop(next(iter(cache)))
            cache[e] = (to_f64(inp["w13"][e]), to_f64(inp["w2"][e]))
        return cache[e]

    rng = np.random.default_rng(1)
    got, want = [], []
    for t in rng.choice(shape.T, size=4, replace=False):
        y_t, idx, *_ = O.token_forward(to_f64(inp["x"][t]), w_r, None, experts, kind=shape.router, k=shape.k,
                                       renorm=shape.renorm, quant=q)
        assert list(idx) == list(gpu_idx[t])
        got.append(to_f64(y[t]))
        want.append(y_t)
    _, _, fro = err_stats(np.array(got), np.array(want))
    assert fro <= MX_FRO, fro


# ----------------------------------------------------------------------------- backward

@pytest.mark.parametrize("shape", [MID, ODD], ids=lambda s: s.name)
def test_backward_weights_bit_exact(shape):
    """W2 quantised along H and W13 along 2I (32-row blocks of each expert's matrix), stored transposed
    ([E][I][H] and [E][H][2I]) as E4M3 bytes and scale blocks."""
    inp = W.make_inputs(shape, seed=0, device="cpu")
    f64 = inputs_f64(inp)
    desc = mok.desc_from_shape(shape)
    wb = mok.quantize_weights_backward(desc, inp["w13"].cuda(), inp["w2"].cuda())
    torch.cuda.synchronize()
    for name, w, N, K in (("w13", f64["w13"], shape.H, 2 * shape.I), ("w2", f64["w2"], shape.I, shape.H)):
        got, X_got = _decode_w(wb[name + "t_q"], wb[name + "t_scale"], N, K)
        for e in range(shape.E):
            want = q(w[e], 0).T
            assert np.array_equal(got[e], want), (name, e, int((got[e] != want).sum()))
            _, X = O.mx_quantize(w[e], 0)
            assert np.array_equal(X_got[e], X.T), (name, e)


def _mx_fwd_bwd(shape, seed=0, given=None, flags=0):
    inp = W.make_inputs(shape, seed=seed, device="cpu")
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    desc = mok.desc_from_shape(shape, flags=flags)
    wq = mok.quantize_weights(desc, dev["w13"], dev["w2"])
    wb = mok.quantize_weights_backward(desc, dev["w13"], dev["w2"])
    layer = mok.MoELayer(desc)
    y = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
    g = torch.tensor(given, dtype=torch.int32, device="cuda") if given is not None else None
    mok.moe_forward_mxfp8(desc, dev["x"], dev["w_router"], dev["router_bias"], g, wq, y, layer.ctx, layer.ws)
    grads = layer.backward_mxfp8(dev["dy"], dev["x"], dev["w_router"], wb)
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    return inp, layer, y, grads


@pytest.mark.parametrize("shape", [MID, MID.scaled(name="mid_mx_skew", skew=True), ODD], ids=lambda s: s.name)
def test_mx_backward_matches_mx_oracle(shape):
    """Every gradient within relative Frobenius 5e-2 of the oracle's MX-emulating backward (each
    backward GEMM operand quantised along its reduction axis, float64 products)."""
    inp0 = W.make_inputs(shape, seed=0, device="cpu")
    f64 = inputs_f64(inp0)
    given = O.route(f64["x"], f64["w_router"], f64["router_bias"], shape.router, shape.k, shape.renorm)["topk_idx"]
    inp, layer, y, g = _mx_fwd_bwd(shape, given=given)
    fwd = O.forward(f64["x"], f64["w_router"], f64["w13"], f64["w2"], kind=shape.router, k=shape.k,
                    renorm=shape.renorm, router_bias=f64["router_bias"], topk_idx=given, quant=q)
    bwd = O.backward(fwd, f64["dy"], f64["x"], f64["w_router"], f64["w13"], f64["w2"], kind=shape.router,
                     k=shape.k, renorm=shape.renorm, quant=q)
    ref_fwd = O.forward(f64["x"], f64["w_router"], f64["w13"], f64["w2"], kind=shape.router, k=shape.k,
                        renorm=shape.renorm, router_bias=f64["router_bias"], topk_idx=given)
    ref = O.backward(ref_fwd, f64["dy"], f64["x"], f64["w_router"], f64["w13"], f64["w2"], kind=shape.router,
                     k=shape.k, renorm=shape.renorm)
    for name in ("dx", "dw13", "dw2", "dgates", "dw_router"):
        _, _, fro = err_stats(to_f64(g[name]), bwd[name])
        _, _, fro_ref = err_stats(to_f64(g[name]), ref[name])
        print("%s: vs MX oracle %.3e, vs unquantised %.3e" % (name, fro, fro_ref))
        assert fro <= MX_FRO, (name, fro)


def test_mx_backward_bf16_weight_gradients_are_rounded_fp32_ones():
    """With bf16 weight gradients the MXFP8 backward gives the fp32 ones rounded to nearest even
    (the same kernels, one rounding at the store); the other gradients do not change."""
    from mixture_experts_layer_table_gb300 import _native as N
    shape = MID.scaled(name="mid_mx_skew", skew=True)
    _, _, _, g32 = _mx_fwd_bwd(shape, seed=5)
    _, _, _, g16 = _mx_fwd_bwd(shape, seed=5, flags=N.FLAG_WGRAD_BF16)
    for name in ("dw13", "dw2"):
        assert g16[name].dtype == torch.bfloat16
        assert torch.equal(g16[name], g32[name].to(torch.bfloat16)), name
    for name in ("dx", "dw_router", "dgates"):
        assert torch.equal(g16[name], g32[name]), name


def test_mx_backward_deterministic():
    shape = MID.scaled(skew=True)
    runs = [_mx_fwd_bwd(shape, seed=4) for _ in range(2)]
    for name in ("dx", "dw13", "dw2", "dgates", "dw_router"):
        assert torch.equal(runs[0][3][name], runs[1][3][name]), name


@pytest.mark.slow
def test_mx_backward_full_size_sampled_experts():
    """DSV3 layer in MXFP8, forward + backward as the benchmark runs it.  For the coldest and the
    hottest expert the oracle recomputes that expert's rows on their own (oracle.expert_weight_grads
    on the rows in schedule order, so that the 32-row quantisation blocks match): sampled rows of
    dW2 and dW13 and the gate gradients of the expert's rows.  For sampled tokens the oracle's
    per-token backward (oracle.token_backward): dx and the gate gradients.  Plus bitwise
    determinism of every gradient."""
    shape = W.DSV3_MXFP8
    inp = W.make_inputs(shape, seed=0, device="cuda")
    desc = mok.desc_from_shape(shape)
    wq = mok.quantize_weights(desc, inp["w13"], inp["w2"])
    wb = mok.quantize_weights_backward(desc, inp["w13"], inp["w2"])
    outs = []
    for _ in range(2):
        layer = mok.MoELayer(desc)
        y = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
        mok.moe_forward_mxfp8(desc, inp["x"], inp["w_router"], None, None, wq, y, layer.ctx, layer.ws)
        g = layer.backward_mxfp8(inp["dy"], inp["x"], inp["w_router"], wb)
        torch.cuda.synchronize()
        assert layer.status() == (0, 0)
        outs.append(g)
    for name in ("dx", "dw_router", "dw13", "dw2", "dgates"):
        assert torch.equal(outs[0][name], outs[1][name]), name
    g = outs[0]
    w_r = to_f64(inp["w_router"])
    r = O.route(to_f64(inp["x"]), w_r, None, shape.router, shape.k, shape.renorm)
    gpu_idx = layer.view("topk_idx").cpu().numpy()
    assert np.array_equal(gpu_idx, r["topk_idx"])
    sched = O.schedule(gpu_idx, shape.E)
    counts = sched["counts"]
    dgates = g["dgates"].cpu().double().numpy().reshape(-1)
    for e in (int(np.argmin(counts)), int(np.argmax(counts))):
        lo, hi = int(sched["offsets"][e]), int(sched["offsets"][e + 1])
        src = sched["src_of"][lo:hi].astype(np.int64)
        sel = torch.as_tensor(src // shape.k, device="cuda")
        rng = np.random.default_rng(e)
        rows2 = rng.choice(shape.H, size=32, replace=False)
        rows13 = rng.choice(2 * shape.I, size=32, replace=False)
        got2 = to_f64(g["dw2"][e][torch.as_tensor(rows2, device="cuda")])
        got13 = to_f64(g["dw13"][e][torch.as_tensor(rows13, device="cuda")])
        check_sampled_expert_wgrads(to_f64(inp["x"][sel]), to_f64(inp["dy"][sel]), r["gates"].reshape(-1)[src],
                                    to_f64(inp["w13"][e]), to_f64(inp["w2"][e]), rows13, rows2, got13, got2,
                                    f"MXFP8 expert {e} ({hi - lo} rows)", got_dg=dgates[src], quant=q,
                                    fro_tol=MX_FRO)
    toks = clear_margin_tokens(r["scores"], shape.k, 4, seed=3)
    sel = torch.as_tensor(toks, device="cuda")
    cache = {}

    def experts(e):
        if e not in cache:
            if len(cache) > 8:
                cache.pop(next(iter(cache)))
            cache[e] = (to_f64(inp["w13"][e]), to_f64(inp["w2"][e]))
        return cache[e]

    check_sampled_token_backward(toks, to_f64(inp["x"][sel]), to_f64(inp["dy"][sel]), w_r, None, experts, shape,
                                 to_f64(g["dx"][sel]), to_f64(g["dgates"][sel]), gpu_idx[toks],
                                 "MXFP8 (sampled tokens)", quant=q, fro_tol=MX_FRO)
