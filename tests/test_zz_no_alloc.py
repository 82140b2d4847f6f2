"""mok_schedule_noalloc: routing and the schedule table for callers that cannot allocate.

Callers such as code under an allocator that forbids new allocations, or a runtime that hands
out only its own pre-sized buffers, cannot give mok_schedule a workspace.  This entry point
keeps its scratch in a fixed array inside the library instead.  Its results must be the same
as mok_schedule's on the same inputs (the same kernels run, so bit for bit), on two calls in a
row (the second sees the scratch the first left behind), and it must refuse a problem whose
router logits do not fit the fixed scratch.

This file is collected last on purpose; it also passes when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_table_gb300 as mok
from mixture_experts_layer_table_gb300 import _native as N
from mixture_experts_layer_table_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_LOGITS = 1 << 20  # MOK_NOALLOC_MAX_LOGITS in include/mok.h


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_ok):
    from mixture_experts_layer_table_gb300 import build
    build.build()
    mok.load()


def _outputs(T, E, k, with_gates=True):
    R = T * k
    o = {"topk_idx": torch.full((T, k), -1, dtype=torch.int32, device="cuda"),
         "gates": torch.full((T, k), -1.0, dtype=torch.float32, device="cuda") if with_gates else None,
         "counts": torch.full((E,), -1, dtype=torch.int32, device="cuda"),
         "offsets": torch.full((E + 1,), -1, dtype=torch.int32, device="cuda"),
         "row_of": torch.full((R,), -1, dtype=torch.int32, device="cuda"),
         "src_of": torch.full((R,), -1, dtype=torch.int32, device="cuda")}
    return o


def _args(o):
    return (o["topk_idx"], o["gates"], o["counts"], o["offsets"], o["row_of"], o["src_of"])


def _with_workspace(desc, x, w_r, bias, given):
    o = _outputs(desc.T, desc.E, desc.k, with_gates=x is not None)
    ws = torch.zeros(mok.get_layout(desc)["ws_bytes"], dtype=torch.uint8, device="cuda")
    mok.schedule(desc, x, w_r, bias, given, *_args(o), ws)
    assert mok.read_status(ws) == (0, 0)
    return o


@pytest.mark.parametrize("shape", [W.DSV3.scaled(name="dsv3_router_max", H=1024, I=256),
                                   W.DSV3_SKEW.scaled(name="dsv3_skew_router", H=512, I=256, T=1000),
                                   W.TINY], ids=lambda s: s.name)
def test_router_path_matches_workspace_entry_point_twice(shape):
    assert shape.T * shape.E <= MAX_LOGITS
    inp = W.make_inputs(shape, seed=2, device="cuda", with_dy=False)
    desc = mok.desc_from_shape(shape)
    ref = _with_workspace(desc, inp["x"], inp["w_router"], inp["router_bias"], None)
    for _ in range(2):
        o = _outputs(shape.T, shape.E, shape.k)
        status = torch.full((2,), -1, dtype=torch.int32, device="cuda")
        N.schedule_noalloc(desc, inp["x"], inp["w_router"], inp["router_bias"], None, *_args(o),
                           device_status=status)
        torch.cuda.synchronize()
        assert status.tolist() == [0, 0]
        for name in ("topk_idx", "counts", "offsets", "row_of", "src_of"):
            assert torch.equal(o[name], ref[name]), name
        # gates: the same kernel on the same logits (well inside the bf16 parity bar)
        assert torch.equal(o["gates"], ref["gates"])


def test_given_selection_path_twice_and_error_report():
    T, E, k = 777, 64, 6
    rng = np.random.default_rng(4)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    desc = mok.make_desc(T, 256, 256, E, k, W.ROUTER_SIGMOID, True)
    given = torch.tensor(idx, device="cuda")
    ref = _with_workspace(desc, None, None, None, given)
    for _ in range(2):
        o = _outputs(T, E, k, with_gates=False)
        status = torch.full((2,), -1, dtype=torch.int32, device="cuda")
        N.schedule_noalloc(desc, None, None, None, given, *_args(o), device_status=status)
        torch.cuda.synchronize()
        assert status.tolist() == [0, 0]
        for name in ("topk_idx", "counts", "offsets", "row_of", "src_of"):
            assert torch.equal(o[name], ref[name]), name
    # a bad expert index is reported through device_status, and the next clean call is clean
    bad = given.clone()
    bad[3, 1] = E
    status = torch.zeros((2,), dtype=torch.int32, device="cuda")
    N.schedule_noalloc(desc, None, None, None, bad, *_args(_outputs(T, E, k, with_gates=False)),
                       device_status=status)
    torch.cuda.synchronize()
    assert int(status[0]) == 6
    N.schedule_noalloc(desc, None, None, None, given, *_args(_outputs(T, E, k, with_gates=False)),
                       device_status=status)
    torch.cuda.synchronize()
    assert status.tolist() == [0, 0]


def test_refuses_logits_beyond_the_fixed_scratch():
    T, E, H = MAX_LOGITS // 256 + 1, 256, 256
    desc = mok.make_desc(T, H, 256, E, 8, W.ROUTER_SIGMOID, True)
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    w_r = torch.zeros((E, H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(N.MokError) as info:
        N.schedule_noalloc(desc, x, w_r, None, None, *_args(_outputs(T, E, 8)))
    assert info.value.code == 3          # MOK_ERR_WORKSPACE_TOO_SMALL
