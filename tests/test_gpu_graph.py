"""CUDA-graph capture of the layer step.

The forward and backward entry points put only stream-ordered work on the caller's stream
(kernel launches and memsets, no host synchronisation, no allocation once the caller's
buffers exist), so a forward + backward captured once replays as the eager step did: the
outputs and gradients of each replay are bitwise those of the eager step.  A launch-bound
layer (the tiny one) gains the most from replaying its launches as one graph.
"""
import pytest
import torch

import mixture_experts_layer_table_gb300 as mok
from mixture_experts_layer_table_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MID = W.MoEShape("mid_T600_H512_E16_I768_top4_sigmoid", T=600, H=512, E=16, I=768, k=4,
                 router=W.ROUTER_SIGMOID, renorm=True, x_std=1.0, w_std=0.03)


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_ok):
    from mixture_experts_layer_table_gb300 import build
    build.build()
    mok.load()


@pytest.mark.parametrize("shape,ring", [(W.TINY, None), (MID.scaled(name="mid_skew", skew=True), None),
                                        (MID, "ring"), (MID, "persistent")],
                         ids=lambda v: getattr(v, "name", str(v)))
def test_graph_replay_is_bitwise_the_eager_step(shape, ring):
    inp = W.make_inputs(shape, seed=0, device="cuda")
    flags = mok.FLAG_RING_PERSISTENT if ring == "persistent" else 0
    desc = mok.desc_from_shape(shape, minibatch=300, ring_bytes=2 * 300 * shape.H * 2, comm_sms=4, flags=flags) \
        if ring else mok.desc_from_shape(shape)
    layer = mok.MoELayer(desc)
    T, H, E, I, k = shape.T, shape.H, shape.E, shape.I, shape.k
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    grads = {"dx": torch.empty((T, H), dtype=torch.bfloat16, device="cuda"),
             "dw_router": torch.empty((E, H), dtype=torch.float32, device="cuda"),
             "dw13": torch.empty((E, 2 * I, H), dtype=torch.float32, device="cuda"),
             "dw2": torch.empty((E, H, I), dtype=torch.float32, device="cuda"),
             "dgates": torch.empty((T, k), dtype=torch.float32, device="cuda")}

    def step():
        layer.forward(inp["x"], inp["w_router"], inp["w13"], inp["w2"], router_bias=inp["router_bias"], y=y)
        layer.backward(inp["dy"], inp["x"], inp["w_router"], inp["w13"], inp["w2"], out=grads)

    step()
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    y0 = y.clone()
    g0 = {n: t.clone() for n, t in grads.items()}

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(2):
        y.fill_(float("nan"))
        for t in grads.values():
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert layer.status() == (0, 0)
        assert torch.equal(y, y0)
        for n in grads:
            assert torch.equal(grads[n], g0[n]), n
