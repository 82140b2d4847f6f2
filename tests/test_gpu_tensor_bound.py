"""Full-size parity at the tensor-bound shape the benchmark times: T=16384 tokens of the DSV3
layer (hidden 7168, 256 experts of intermediate 2048, top-8 sigmoid router with renormalised
gates), 512 rows per expert, where GEMM1 takes its paired form and the expert GEMMs cut each
expert into 256-row chunks; plain, and through the 512 MiB token ring at the minibatch of two
GEMM1 waves (2368 rows).

The oracle computes sampled tokens on their own (each needs only its k experts) and the ring
forward must be bitwise the plain one.  Tokens are drawn among those whose k-th and (k+1)-th
router scores differ clearly, so that the GPU's fp32 router and the float64 oracle pick the
same experts.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_table_gb300 as mok
from mixture_experts_layer_table_gb300 import workloads as W
from oracle import moe_oracle as O
from tests.parity import check_sampled_token_outputs, clear_margin_tokens, to_f64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SHAPE = W.RING
MINIBATCH = 2368
N_TOKENS = 6
N_CANDIDATES = 64


@pytest.fixture(scope="module")
def run(cuda_ok):
    from mixture_experts_layer_table_gb300 import build
    build.build()
    mok.load()
    inp = W.make_inputs(SHAPE, seed=0, device="cuda", with_dy=False)
    plain = mok.MoELayer(mok.desc_from_shape(SHAPE))
    y_plain = plain.forward(inp["x"], inp["w_router"], inp["w13"], inp["w2"])
    torch.cuda.synchronize()
    assert plain.status() == (0, 0)
    idx = plain.view("topk_idx").cpu().numpy()
    table = {name: plain.view(name).cpu().numpy() for name in ("counts", "offsets", "row_of", "src_of")}
    del plain
    torch.cuda.empty_cache()
    ring = mok.MoELayer(mok.desc_from_shape(SHAPE, minibatch=MINIBATCH, ring_bytes=W.RING_BYTES))
    assert ring.layout["ring"] >= 0
    y_ring = ring.forward(inp["x"], inp["w_router"], inp["w13"], inp["w2"])
    torch.cuda.synchronize()
    assert ring.status() == (0, 0)
    idx_ring = ring.view("topk_idx").cpu().numpy()
    del ring
    torch.cuda.empty_cache()
    # GEMM2 and the weighted merge in the persistent launch too
    one = mok.MoELayer(mok.desc_from_shape(SHAPE, minibatch=MINIBATCH, ring_bytes=W.RING_BYTES,
                                           flags=mok.FLAG_RING_PERSISTENT))
    y_one = one.forward(inp["x"], inp["w_router"], inp["w13"], inp["w2"])
    torch.cuda.synchronize()
    assert one.status() == (0, 0)
    del one
    torch.cuda.empty_cache()
    return inp, idx, y_plain, idx_ring, y_ring, table, y_one


def test_ring_forward_is_bitwise_the_plain_forward(run):
    _, idx, y_plain, idx_ring, y_ring, _, _ = run
    assert np.array_equal(idx, idx_ring)
    assert torch.equal(y_plain, y_ring)


def test_persistent_ring_forward_is_bitwise_the_plain_forward(run):
    """GEMM2 and the weighted merge in the ring's persistent launch as well."""
    y_plain, y_persistent = run[2], run[6]
    assert torch.equal(y_plain, y_persistent)


def test_sampled_tokens_against_the_oracle(run):
    inp, idx, y_plain, _, _, _, _ = run
    rng = np.random.default_rng(1)
    cand = np.sort(rng.choice(SHAPE.T, size=N_CANDIDATES, replace=False))
    w_r = to_f64(inp["w_router"])
    x_c = to_f64(inp["x"][torch.as_tensor(cand, device=inp["x"].device)])
    _, scores = O.router_scores(x_c, w_r, SHAPE.router)
    pick = clear_margin_tokens(scores, SHAPE.k, N_TOKENS, seed=2)
    assert len(pick) == N_TOKENS
    toks = cand[pick]
    cache = {}

    def experts(e):
        if e not in cache:
            if len(cache) > 8:
                cache.pop(next(iter(cache)))
            cache[e] = (to_f64(inp["w13"][e]), to_f64(inp["w2"][e]))
        return cache[e]

    y_rows = to_f64(y_plain[torch.as_tensor(toks, device=y_plain.device)])
    check_sampled_token_outputs(toks, x_c[pick], w_r, None, experts, SHAPE, y_rows, idx[toks],
                                "y (T=16384, sampled tokens)")


def test_schedule_table_bit_exact(run):
    """The whole schedule table at T=16384 (131,072 assignments), bit-exact against the oracle's
    stable counting sort of the same selection."""
    _, idx, _, _, _, table, _ = run
    ref = O.schedule(idx, SHAPE.E)
    for name in ("counts", "offsets", "row_of", "src_of"):
        assert np.array_equal(table[name], ref[name]), name


def test_fp16_w2_forward_sampled_tokens(run):
    """The same T=16384 forward with MOK_FLAG_W2_F16 (fp16 copy of W2, a as one fp16 value, one GEMM2
    MMA per K step): the same selection, and the sampled tokens against the oracle on the bf16
    weights at the bf16 bar."""
    inp, idx, y_plain, _, _, _, _ = run
    w2_f16 = mok.convert_f16(inp["w2"])
    layer = mok.MoELayer(mok.desc_from_shape(SHAPE, flags=mok.FLAG_W2_F16))
    y = layer.forward(inp["x"], inp["w_router"], inp["w13"], w2_f16)
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    assert np.array_equal(layer.view("topk_idx").cpu().numpy(), idx)
    del layer, w2_f16
    torch.cuda.empty_cache()
    rng = np.random.default_rng(3)
    cand = np.sort(rng.choice(SHAPE.T, size=N_CANDIDATES, replace=False))
    w_r = to_f64(inp["w_router"])
    x_c = to_f64(inp["x"][torch.as_tensor(cand, device=inp["x"].device)])
    _, scores = O.router_scores(x_c, w_r, SHAPE.router)
    pick = clear_margin_tokens(scores, SHAPE.k, N_TOKENS, seed=4)
    toks = cand[pick]
    cache = {}

    def experts(e):
        if e not in cache:
            if len(cache) > 8:
                cache.pop(next(iter(cache)))
            cache[e] = (to_f64(inp["w13"][e]), to_f64(inp["w2"][e]))
        return cache[e]

    y_rows = to_f64(y[torch.as_tensor(toks, device=y.device)])
    check_sampled_token_outputs(toks, x_c[pick], w_r, None, experts, SHAPE, y_rows, idx[toks],
                                "y (T=16384, fp16 W2, sampled tokens)")


def test_ring_backward_full_size_bitwise(run):
    """Forward + backward at T=16384 through the 512 MiB ring (minibatch 2368): the ring-based
    backward reuses the minibatches the ring still holds and gathers the rest again; every
    gradient is bitwise the plain layer's."""
    inp = run[0]
    g = torch.Generator(device="cuda").manual_seed(4)
    dy = torch.empty((SHAPE.T, SHAPE.H), dtype=torch.float32, device="cuda").normal_(0.0, 1.0, generator=g)
    dy = dy.to(torch.bfloat16)
    args = (inp["x"], inp["w_router"], inp["w13"], inp["w2"])
    plain = mok.MoELayer(mok.desc_from_shape(SHAPE))
    plain.forward(*args)
    g0 = plain.backward(dy, *args)
    torch.cuda.synchronize()
    assert plain.status() == (0, 0)
    del plain
    torch.cuda.empty_cache()
    ring = mok.MoELayer(mok.desc_from_shape(SHAPE, minibatch=MINIBATCH, ring_bytes=W.RING_BYTES))
    ring.forward(*args)
    g1 = ring.backward(dy, *args)
    torch.cuda.synchronize()
    assert ring.status() == (0, 0)
    for name in ("dx", "dw_router", "dw13", "dw2", "dgates"):
        assert torch.equal(g1[name], g0[name]), name
    del ring, g0, g1
    torch.cuda.empty_cache()
