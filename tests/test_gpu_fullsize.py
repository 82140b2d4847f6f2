"""Full-size parity at the DeepSeek-V3 layer shape (T=4096, hidden 7168, 256 experts of
intermediate 2048, top-8 sigmoid router with renormalised gates), with near-uniform routing and
with the Zipf-Mandelbrot skewed routing (hottest expert about 10x the mean load, the coldest a
handful of rows), run in the same launch configuration the benchmark times (router on the GPU,
default fp32 weight gradients).

The oracle cannot run the whole layer at this size in a test's time, so it checks sampled
outputs it can compute one at a time (oracle.token_forward / token_backward /
expert_weight_grads): the output rows, input-gradient rows and gate gradients of sampled tokens
(each needs only that token's k experts), and sampled rows of the weight gradients and the gate
gradients of the coldest and the hottest expert (each needs only that expert and its rows).
The schedule table is compared in full.  The router-weight gradient needs every token of an
expert together with all of their experts; it is checked in full at the mid sizes of
test_gpu_layer.py instead.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_table_gb300 as mok
from mixture_experts_layer_table_gb300 import workloads as W
from oracle import moe_oracle as O
from tests.parity import (check_sampled_expert_wgrads, check_sampled_token_backward, check_sampled_token_outputs,
                          clear_margin_tokens, selection_is_valid, to_f64)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

N_TOKENS = 6
N_WROWS = 48


class ExpertCache:
    def __init__(self, inp):
        self.inp = inp
        self.cache = {}

    def __call__(self, e):
        if e not in self.cache:
            if len(self.cache) > 8:
                self.cache.pop(next(iter(self.cache)))
            self.cache[e] = (to_f64(self.inp["w13"][e]), to_f64(self.inp["w2"][e]))
        return self.cache[e]


@pytest.fixture(scope="module", params=[W.DSV3, W.DSV3_SKEW], ids=["uniform", "skew"])
def run(request, cuda_ok):
    from mixture_experts_layer_table_gb300 import build
    build.build()
    mok.load()
    shape = request.param
    inp = W.make_inputs(shape, seed=0, device="cuda")
    layer = mok.MoELayer(mok.desc_from_shape(shape))
    y = layer.forward(inp["x"], inp["w_router"], inp["w13"], inp["w2"], router_bias=inp["router_bias"])
    g = layer.backward(inp["dy"], inp["x"], inp["w_router"], inp["w13"], inp["w2"])
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    # the oracle's router over all tokens (float64), from the generator's inputs
    x = to_f64(inp["x"])
    bias = to_f64(inp["router_bias"]) if inp["router_bias"] is not None else None
    r = O.route(x, to_f64(inp["w_router"]), bias, shape.router, shape.k, shape.renorm)
    r["bias"] = bias
    r["selection"] = r["scores"] + (bias[None, :] if bias is not None else 0.0)
    yield shape, inp, layer, y, g, r
    del layer, y, g, inp
    torch.cuda.empty_cache()


def test_selection_matches_oracle(run):
    """Every GPU choice is a valid top-k of the oracle's float64 selection scores (a near-tie
    within 1e-5 relative may break either way); with this seed no token sits that close, so the
    choices are identical."""
    shape, inp, layer, y, g, r = run
    gpu = layer.view("topk_idx").cpu().numpy()
    n_diff = selection_is_valid(r["selection"], gpu, shape.k)
    assert n_diff == 0 and np.array_equal(gpu, r["topk_idx"])


def test_schedule_full_size(run):
    """The whole schedule table, bit-exact against the oracle's stable counting sort of the GPU's
    selection, and the dispatched rows bit-exact."""
    shape, inp, layer, y, g, r = run
    idx = layer.view("topk_idx").cpu().numpy()
    ref = O.schedule(idx, shape.E)
    for name in ("counts", "offsets", "row_of", "src_of"):
        assert np.array_equal(layer.view(name).cpu().numpy(), ref[name]), name
    src_of = ref["src_of"].astype(np.int64)
    assert np.array_equal(to_f64(layer.view("x_g")), to_f64(inp["x"])[src_of // shape.k])
    counts = ref["counts"]
    load = counts.max() / counts.mean()
    print(f"{shape.name}: rows per expert min {counts.min()} max {counts.max()}, max/mean {load:.2f}")
    if shape.skew:
        # the skewed workload: hottest expert ~10x the mean, every expert still served
        assert 8.0 <= load <= 12.0 and counts.min() >= 1
    else:
        assert load < 1.5


def test_sampled_tokens_output_and_input_gradient(run):
    shape, inp, layer, y, g, r = run
    toks = clear_margin_tokens(r["selection"], shape.k, N_TOKENS, seed=0)
    assert len(toks) == N_TOKENS
    sel = torch.as_tensor(toks, device="cuda")
    w_r = to_f64(inp["w_router"])
    experts = ExpertCache(inp)
    gpu_idx = layer.view("topk_idx").cpu().numpy()[toks]
    x_rows, dy_rows = to_f64(inp["x"][sel]), to_f64(inp["dy"][sel])
    check_sampled_token_outputs(toks, x_rows, w_r, r["bias"], experts, shape, to_f64(y[sel]), gpu_idx,
                                f"{shape.name} y (sampled tokens)")
    check_sampled_token_backward(toks, x_rows, dy_rows, w_r, r["bias"], experts, shape, to_f64(g["dx"][sel]),
                                 to_f64(g["dgates"][sel]), gpu_idx, f"{shape.name} (sampled tokens)")


def test_sampled_expert_weight_gradients(run):
    """The coldest and the hottest expert: sampled rows of dW13 and dW2 and the gate gradients of
    all the expert's rows, against the oracle on that expert's rows in schedule order."""
    shape, inp, layer, y, g, r = run
    idx = layer.view("topk_idx").cpu().numpy()
    sched = O.schedule(idx, shape.E)
    counts = sched["counts"]
    gates = O.gate_values(r["scores"], idx, shape.renorm)
    dgates = g["dgates"].cpu().double().numpy().reshape(-1)
    for e in (int(np.argmin(counts)), int(np.argmax(counts))):
        lo, hi = int(sched["offsets"][e]), int(sched["offsets"][e + 1])
        src = sched["src_of"][lo:hi].astype(np.int64)
        toks = torch.as_tensor(src // shape.k, device="cuda")
        rng = np.random.default_rng(e)
        rows13 = rng.choice(2 * shape.I, size=N_WROWS, replace=False)
        rows2 = rng.choice(shape.H, size=N_WROWS, replace=False)
        got13 = to_f64(g["dw13"][e][torch.as_tensor(rows13, device="cuda")])
        got2 = to_f64(g["dw2"][e][torch.as_tensor(rows2, device="cuda")])
        check_sampled_expert_wgrads(to_f64(inp["x"][toks]), to_f64(inp["dy"][toks]), gates.reshape(-1)[src],
                                    to_f64(inp["w13"][e]), to_f64(inp["w2"][e]), rows13, rows2, got13, got2,
                                    f"{shape.name} expert {e} ({hi - lo} rows)", got_dg=dgates[src])


def test_full_size_bitwise_deterministic(run):
    shape, inp, layer, y, g, r = run
    layer2 = mok.MoELayer(mok.desc_from_shape(shape))
    y2 = layer2.forward(inp["x"], inp["w_router"], inp["w13"], inp["w2"], router_bias=inp["router_bias"])
    g2 = layer2.backward(inp["dy"], inp["x"], inp["w_router"], inp["w13"], inp["w2"])
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    for name in ("dx", "dw_router", "dw13", "dw2", "dgates"):
        assert torch.equal(g[name], g2[name]), name
    del layer2, y2, g2
    torch.cuda.empty_cache()
