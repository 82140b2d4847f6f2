"""The C ABI library: loads, exports every declared entry point, host-side checks (CPU only)."""
import ctypes
import json
import os
import re

import pytest

import mixture_experts_layer_table_gb300 as mok
from mixture_experts_layer_table_gb300 import _native as N
from mixture_experts_layer_table_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_layer_table_gb300 import build
    build.build()
    return N.load()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names.update(re.findall(r"\b(mok_\w+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert {"mok_schedule", "mok_moe_forward", "mok_moe_backward"} <= declared
    for name in declared:
        assert hasattr(lib, name), name


def test_layout_sizes_and_alignment(lib):
    lay = mok.get_layout(mok.desc_from_shape(W.DSV3))
    R, H, I = W.DSV3.R, W.DSV3.H, W.DSV3.I
    for name, off in lay.items():
        assert off % 256 == 0 or (off == -1 and (name in ("ring", "mb_tables", "mb_counters", "ring_stamp") or
                                                 name.startswith("mx_"))), name
    assert lay["ctx_bytes"] >= lay["hu"] + R * 2 * I * 2
    assert lay["ws_bytes"] >= lay["dlogits"] + W.DSV3.T * W.DSV3.E * 4
    assert lay["status"] == 0
    assert lay["x_g"] < lay["hu"] and lay["hu"] - lay["x_g"] >= R * H * 2


@pytest.mark.parametrize("field,value,code", [("H", 300, 2), ("I", 100, 2), ("k", 9, 1), ("E", 2000, 2),
                                              ("T", 0, 1), ("router", 3, 1), ("k", 17, 1),
                                              ("flags", N.FLAG_GEMM_PAIR | N.FLAG_GEMM_SINGLE, 1)])
def test_desc_validation(lib, field, value, code):
    d = mok.desc_from_shape(W.TINY)
    setattr(d, field, value)
    if field == "k" and value == 17:
        d.E = 32
        code = 2
    lay = N.Layout()
    assert lib.mok_get_layout(ctypes.byref(d), ctypes.byref(lay)) == code


def test_mxfp8_layout_has_the_backward_operands(lib):
    bf = mok.get_layout(mok.desc_from_shape(W.DSV3))
    mx = mok.get_layout(mok.desc_from_shape(W.DSV3_MXFP8))
    R, H, I, E = W.DSV3.T * W.DSV3.k, W.DSV3.H, W.DSV3.I, W.DSV3.E
    RP = 32 * (-(-R // 32) + E)
    G = RP // 32 + 4
    sizes = {"mx_dhu_r": R * 2 * I * 2, "mx_xg_r": R * H * 2, "mx_do_r": R * H * 2,
             "mx_a_r": R * I * 2, "mx_blk_off": (E + 1) * 4, "mx_dyq": RP * H, "mx_dysf": G * (H // 128) * 512,
             "mx_dhuq": RP * 2 * I, "mx_dhusf": G * (2 * I // 128) * 512}
    ends = []
    for name, nbytes in sizes.items():
        assert bf[name] == -1, name
        assert mx[name] >= bf["dlogits"] and mx[name] % 256 == 0, name
        ends.append((mx[name], mx[name] + nbytes))
    ends.sort()
    assert all(a[1] <= b[0] for a, b in zip(ends, ends[1:]))  # disjoint
    assert ends[-1][1] <= mx["ws_bytes"]


def test_ring_layout(lib):
    """Ring forward: the ring holds whole minibatches (at most as many as there are)."""
    shp = W.RING
    m = 2368
    d = mok.desc_from_shape(shp, minibatch=m, ring_bytes=W.RING_BYTES)
    lay = mok.get_layout(d)
    slots = W.RING_BYTES // (m * shp.H * 2)
    n_mb = -(-shp.R // m)
    # the dispatched rows of every minibatch (the ring is their last `slots` minibatches)
    assert lay["mb_tables"] - lay["ring"] >= n_mb * m * shp.H * 2 and slots < n_mb
    assert lay["ring_stamp"] >= 0 and lay["ring_stamp"] + 16 <= lay["ctx_bytes"]
    assert lay["mb_counters"] - lay["mb_tables"] >= (2 * n_mb * (shp.E + 1) + 2 * n_mb + 1) * 4
    # a ring below one minibatch is refused
    d.ring_bytes = m * shp.H * 2 - 1
    lay_ = N.Layout()
    assert lib.mok_get_layout(ctypes.byref(d), ctypes.byref(lay_)) == 2


def test_min_minibatch_reproduces_page_number(lib):
    with open(os.path.join(ROOT, "tests", "golden", "pages_numbers.json")) as f:
        g = json.load(f)["min_minibatch_tokens"]
    assert mok.min_minibatch(148, g["intermediate"]) == g["value"]
    assert mok.min_minibatch(160, 2048) == 2560      # the other minibatch the pages time


def test_status_strings(lib):
    assert mok.status_string(0) == "ok"
    assert "timed out" in mok.status_string(5)


def _region_sizes(shp, ring_slots=0, minibatch=0):
    """Bytes of each tensor, as the comments of mok_layout in include/mok.h state them."""
    T, H, I, E, k = shp.T, shp.H, shp.I, shp.E, shp.k
    R = T * k
    ctx = {"topk_idx": R * 4, "gates": R * 4, "scores": T * E * 4, "counts": E * 4, "offsets": (E + 1) * 4,
           "row_of": R * 4, "src_of": R * 4, "tile_off": (E + 1) * 4, "gate_row": R * 4, "x_g": R * H * 2,
           "hu": R * 2 * I * 4}
    if minibatch:
        ctx["ring_stamp"] = 16
    ws = {"status": 64 * 4, "logits": T * E * 4, "sched": -(-R // 1024) * E * 4, "act": R * I * 2, "act_lo": R * I * 2, "expert_out": R * H * 4,
          "dy_g": R * H * 2, "dhu": R * 2 * I * 2, "dhu_lo": R * 2 * I * 2, "gact": R * I * 2,
          "gact_lo": R * I * 2, "dx_g": R * H * 4, "dg_part": R * (I // 128) * 4, "dlogits": T * E * 4}
    if minibatch:
        n_mb = -(-R // minibatch)
        ws.update({"ring": n_mb * minibatch * H * 2,
                   "mb_tables": (2 * n_mb * (E + 1) + n_mb + (n_mb + 1)) * 4,
                   "mb_counters": (((2 * n_mb + 1) * 4 + 15) // 16) * 16 + 16})
    if shp.mxfp8:
        ws.update({"mx_dhu_r": R * 2 * I * 2, "mx_xg_r": R * H * 2,
                   "mx_do_r": R * H * 2, "mx_a_r": R * I * 2, "mx_blk_off": (E + 1) * 4})
        RP = 32 * (-(-R // 32) + E)       # padded rows: every expert's rows rounded up to 32
        G = RP // 32 + 4                  # row groups of the scale blocks
        ws.update({"mx_xq": RP * H, "mx_xsf": G * (H // 128) * 512, "mx_aq": RP * I,
                   "mx_asf": G * (I // 128) * 512, "mx_dyq": RP * H, "mx_dysf": G * (H // 128) * 512,
                   "mx_dhuq": RP * 2 * I, "mx_dhusf": G * (2 * I // 128) * 512})
    return ctx, ws


@pytest.mark.parametrize("case", ["tiny", "dsv3", "skew", "mxfp8", "ring"])
def test_every_region_sized_aligned_and_disjoint(lib, case):
    """Each tensor of ctx and ws gets at least the bytes the header states, on a 256-byte boundary,
    without overlapping another; tensors a descriptor does not use are -1."""
    shp = {"tiny": W.TINY, "dsv3": W.DSV3, "skew": W.DSV3_SKEW, "mxfp8": W.DSV3_MXFP8, "ring": W.RING}[case]
    kw, slots, m = {}, 0, 0
    if case == "ring":
        m = 2368
        kw = dict(minibatch=m, ring_bytes=W.RING_BYTES)
        slots = W.RING_BYTES // (m * shp.H * 2)
    lay = mok.get_layout(mok.desc_from_shape(shp, **kw))
    ctx, ws = _region_sizes(shp, slots, m)
    assert set(ctx) | {"ring_stamp"} == set(N.CTX_FIELDS)   # ring_stamp: ring forward only
    for fields, sizes, total in ((N.CTX_FIELDS, ctx, lay["ctx_bytes"]), (N.WS_FIELDS, ws, lay["ws_bytes"])):
        spans = []
        for name in fields:
            if name not in sizes:
                assert lay[name] == -1, name
                continue
            off = lay[name]
            assert off >= 0 and off % 256 == 0, name
            spans.append((off, off + sizes[name], name))
        spans.sort()
        for a, b in zip(spans, spans[1:]):
            assert a[1] <= b[0], (a[2], b[2])
        assert spans[-1][1] <= total


def test_missing_library_fails_loudly(tmp_path):
    """No fallback: without libmok.so the binding raises instead of computing anything."""
    import subprocess
    import sys
    code = ("from mixture_experts_layer_table_gb300 import _native as N\n"
            f"N.load({str(tmp_path / 'libmok.so')!r})\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0 and "OSError" in r.stderr and "not found" in r.stderr


def test_host_tensors_are_refused(lib):
    """Every tensor the library reads or writes must be device memory: host tensors are refused
    by the binding before any library call (there is no CPU path)."""
    import torch
    shp = W.TINY
    d = mok.desc_from_shape(shp)
    layer = mok.MoELayer(d, device="cpu")
    inp = W.make_inputs(shp, seed=0, device="cpu")
    with pytest.raises(ValueError, match="CUDA"):
        layer.forward(inp["x"], inp["w_router"], inp["w13"], inp["w2"])
    with pytest.raises(ValueError, match="CUDA"):
        N.read_status(layer.ws)
    with pytest.raises(ValueError, match="CUDA"):
        N.test_bounded_wait(layer.ws, 10)
    y = torch.empty((shp.T, shp.H), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        N.moe_forward(d, inp["x"], inp["w_router"], None, None, inp["w13"], inp["w2"], y, layer.ctx, layer.ws)


def test_entry_points_reject_bad_arguments_before_any_device_work(lib):
    """The argument checks of the C ABI return their error codes before the library touches the
    GPU, so they are exercised here with placeholder (never dereferenced) addresses: a null or
    misaligned tensor is an invalid argument, a ctx / ws one byte short is too small, and a
    descriptor of the other precision is unsupported.  Host-only: with a GPU present a regression
    in the order of the checks could hand the placeholders to a kernel."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("placeholder addresses are for hosts without a GPU")
    P, SZ = ctypes.c_void_p, ctypes.c_size_t
    D = ctypes.POINTER(N.LayerDesc)
    fwd_mx = lib.mok_moe_forward_mxfp8
    fwd_mx.argtypes = [D] + [P] * 9 + [P, SZ, P, SZ, P]
    bwd_mx = lib.mok_moe_backward_mxfp8
    bwd_mx.argtypes = [D] + [P] * 8 + [SZ] + [P] * 6 + [SZ, P]
    for f in (fwd_mx, bwd_mx):
        f.restype = ctypes.c_int32
    bf = mok.desc_from_shape(W.TINY)
    mx = mok.desc_from_shape(W.TINY.scaled(mxfp8=True))
    lay = mok.get_layout(bf)
    lay_mx = mok.get_layout(mx)
    a = [P(0x100000 * (i + 1)) for i in range(16)]   # 16-byte aligned placeholders
    ctx_n, ws_n = lay["ctx_bytes"], lay["ws_bytes"]

    def fwd(desc, x=a[0], ctx_n=ctx_n, ws_n=ws_n):
        return lib.mok_moe_forward(ctypes.byref(desc), x, a[1], None, None, a[2], a[3], a[4], a[5], ctx_n, a[6],
                                   ws_n, None)

    def bwd(desc, dy=a[0], ctx_n=ctx_n, ws_n=ws_n):
        return lib.mok_moe_backward(ctypes.byref(desc), dy, a[1], a[2], a[3], a[4], a[5], ctx_n, a[6], a[7],
                                    a[8], a[9], None, a[10], ws_n, None)

    for call in (fwd, bwd):
        assert call(bf, ctx_n=ctx_n - 1) == 3
        assert call(bf, ws_n=ws_n - 1) == 3
        assert call(bf, P(0x100008), ctx_n=ctx_n - 1) == 1      # misaligned: checked first
        assert call(bf, None, ctx_n=ctx_n - 1) == 1
        assert call(mx) == 2                                    # MXFP8 has its own entry points
    m_ctx, m_ws = lay_mx["ctx_bytes"], lay_mx["ws_bytes"]
    assert fwd_mx(ctypes.byref(bf), *a[:9], a[9], m_ctx, a[10], m_ws, None) == 2
    assert fwd_mx(ctypes.byref(mx), *a[:9], a[9], m_ctx, a[10], m_ws - 1, None) == 3
    assert fwd_mx(ctypes.byref(mx), None, *a[1:9], a[9], m_ctx, a[10], m_ws - 1, None) == 1
    assert bwd_mx(ctypes.byref(bf), *a[:8], m_ctx, *a[8:14], m_ws, None) == 2
    assert bwd_mx(ctypes.byref(mx), *a[:8], m_ctx - 1, *a[8:14], m_ws, None) == 3
    assert bwd_mx(ctypes.byref(mx), *a[:7], P(0x100004), m_ctx - 1, *a[8:14], m_ws, None) == 1
    # schedule: ws one byte short, and a missing output
    sch = lambda topk, ws_n: lib.mok_schedule(ctypes.byref(bf), a[0], a[1], None, None, topk, a[2], a[3], a[4], a[5],
                                              a[6], a[7], ws_n, None)
    assert sch(a[8], ws_n - 1) == 3
    assert sch(None, ws_n) == 1


@pytest.mark.parametrize("case", ["tiny", "dsv3", "mxfp8", "ring"])
def test_workspace_size_matches_layout(lib, case):
    shp = {"tiny": W.TINY, "dsv3": W.DSV3, "mxfp8": W.DSV3_MXFP8, "ring": W.RING}[case]
    kw = dict(minibatch=2368, ring_bytes=W.RING_BYTES) if case == "ring" else {}
    d = mok.desc_from_shape(shp, **kw)
    lay = mok.get_layout(d)
    assert mok.workspace_size(d) == (lay["ws_bytes"], lay["ctx_bytes"])
    ws, ctx = ctypes.c_size_t(7), ctypes.c_size_t(7)
    assert lib.mok_workspace_size(ctypes.byref(d), None, ctypes.byref(ctx)) == 1
    d.k = d.E + 1                       # invalid descriptor: its status, outputs untouched
    assert lib.mok_workspace_size(ctypes.byref(d), ctypes.byref(ws), ctypes.byref(ctx)) == 1
    assert ws.value == 7 and ctx.value == 7


def test_trace_argument_checks(lib):
    """mok_trace_start takes 1 .. 2^20 launches and refuses a second start; mok_trace_stop without
    a trace running is an invalid argument (no device needed for these answers)."""
    n = ctypes.c_int32(-1)
    assert lib.mok_trace_start(0) == 1
    assert lib.mok_trace_start((1 << 20) + 1) == 1
    assert lib.mok_trace_stop(None, 0, ctypes.byref(n)) == 1
    code = lib.mok_trace_start(4)
    assert code in (0, 4)                  # 4 (a CUDA error) on a host without a GPU
    if code == 0:
        assert lib.mok_trace_start(4) == 1
        assert lib.mok_trace_stop(None, 0, ctypes.byref(n)) == 0 and n.value == 0


@pytest.mark.parametrize("H,I,ok", [(384, 640, True), (7168, 1408, True), (128, 128, True), (320, 512, False),
                                    (512, 448, False), (256, 64, False)])
def test_widths_are_multiples_of_128(lib, H, I, ok):
    """H and I: any multiple of 128 (odd multiples included: the last 256-row pair tile reads zeros
    past the end), anything else is unsupported (MOK_ERR_UNSUPPORTED = 2)."""
    desc = N.make_desc(64, H, I, 8, 2, W.ROUTER_SIGMOID, True)
    if ok:
        assert N.get_layout(desc)["ws_bytes"] > 0
    else:
        with pytest.raises(mok.MokError) as info:
            N.get_layout(desc)
        assert info.value.code == 2
