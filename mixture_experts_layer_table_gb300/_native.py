"""ctypes binding of libmok.so (include/mok.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Device memory comes from PyTorch (caller tensors, or torch.empty for
ctx / ws in MoELayer); the stream is PyTorch's current stream unless given.
There is no fallback: if libmok.so is missing or fails to load, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmok.so")

MOK_OK = 0
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "workspace too small", 4: "CUDA error",
                5: "timeout", 6: "invalid routing"}


class MokError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(code, code)} ({code})")
        self.code = code


class LayerDesc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("router", ctypes.c_int32), ("renorm", ctypes.c_int32),
                ("route_scale", ctypes.c_float), ("precision", ctypes.c_int32), ("minibatch", ctypes.c_int32),
                ("ring_bytes", ctypes.c_int64), ("flags", ctypes.c_int32), ("comm_sms", ctypes.c_int32)]


LAYOUT_FIELDS = ["topk_idx", "gates", "scores", "counts", "offsets", "row_of", "src_of", "tile_off", "gate_row",
                 "x_g", "hu", "ring_stamp", "ctx_bytes", "status", "logits", "sched", "act", "act_lo", "expert_out", "dy_g", "dhu", "dhu_lo",
                 "gact", "gact_lo", "dx_g", "dg_part", "dlogits", "ring", "mb_tables", "mb_counters",
                 "mx_dhu_r", "mx_xg_r", "mx_do_r", "mx_a_r", "mx_blk_off", "mx_xq", "mx_xsf", "mx_aq",
                 "mx_asf", "mx_dyq", "mx_dysf", "mx_dhuq", "mx_dhusf", "ws_bytes"]
FLAG_WGRAD_BF16 = 1
FLAG_GEMM_PAIR = 2     # GEMM1 / GEMM2 on CTA pairs with 256-row tiles (dX_g: single CTAs)
FLAG_GEMM_SINGLE = 4   # GEMM1 / GEMM2 / dX_g on single CTAs with 128-row tiles
FLAG_W2_F16 = 8        # forward: w2 is fp16 (convert_f16), a kept as fp16, GEMM2 on fp16 operands
FLAG_RING_PERSISTENT = 16  # ring forward: gather, GEMM1, GEMM2 and the merge in one persistent launch
# neither: GEMM1, GEMM2 and dX_g on the narrow-segment pair kernel (expert rows as the MMA's N)
CTX_FIELDS = LAYOUT_FIELDS[:LAYOUT_FIELDS.index("ctx_bytes")]
WS_FIELDS = LAYOUT_FIELDS[LAYOUT_FIELDS.index("ctx_bytes") + 1:LAYOUT_FIELDS.index("ws_bytes")]


class Layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in LAYOUT_FIELDS]


class TraceEntry(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int32), ("total_ms", ctypes.c_float)]


EXPORTS = ["mok_get_layout", "mok_workspace_size", "mok_schedule", "mok_moe_forward", "mok_moe_backward", "mok_read_status",
           "mok_test_bounded_wait", "mok_status_string", "mok_min_minibatch", "mok_trace_start", "mok_trace_stop"]

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libmok.so once (raises OSError when it is missing: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise OSError(f"{path} not found: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    D = ctypes.POINTER(LayerDesc)
    lib.mok_get_layout.argtypes = [D, ctypes.POINTER(Layout)]
    lib.mok_workspace_size.argtypes = [D, ctypes.POINTER(SZ), ctypes.POINTER(SZ)]
    lib.mok_schedule.argtypes = [D, P, P, P, P, P, P, P, P, P, P, P, SZ, P]
    lib.mok_moe_forward.argtypes = [D, P, P, P, P, P, P, P, P, SZ, P, SZ, P]
    lib.mok_moe_backward.argtypes = [D, P, P, P, P, P, P, SZ, P, P, P, P, P, P, SZ, P]
    lib.mok_read_status.argtypes = [P, SZ, P, ctypes.POINTER(I32)]
    lib.mok_test_bounded_wait.argtypes = [P, SZ, I32, P]
    lib.mok_status_string.argtypes = [I32]
    lib.mok_status_string.restype = ctypes.c_char_p
    lib.mok_min_minibatch.argtypes = [I32, I32]
    lib.mok_min_minibatch.restype = I32
    lib.mok_trace_start.argtypes = [I32]
    lib.mok_trace_stop.argtypes = [ctypes.POINTER(TraceEntry), I32, ctypes.POINTER(I32)]
    for name in EXPORTS:
        if name != "mok_status_string" and name != "mok_min_minibatch":
            getattr(lib, name).restype = I32
    _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libmok must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _buf(t: torch.Tensor, name: str):
    """Pointer and byte size of a ctx / ws buffer: device memory, contiguous (the library checks
    the size against the layout)."""
    if t is None or t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    return _ptr(t), t.numel() * t.element_size()


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(fn: str, code: int):
    if code != MOK_OK:
        raise MokError(fn, code)


def make_desc(T, H, I, E, k, router, renorm, route_scale=1.0, precision=0, minibatch=0, ring_bytes=0,
              flags=0, comm_sms=0) -> LayerDesc:
    return LayerDesc(T, H, I, E, k, router, int(bool(renorm)), route_scale, precision, minibatch, ring_bytes,
                     flags, comm_sms)


def desc_from_shape(shape, **kw) -> LayerDesc:
    return make_desc(shape.T, shape.H, shape.I, shape.E, shape.k, shape.router, shape.renorm,
                     precision=1 if shape.mxfp8 else 0, **kw)


def get_layout(desc: LayerDesc) -> Dict[str, int]:
    lay = Layout()
    _check("mok_get_layout", load().mok_get_layout(ctypes.byref(desc), ctypes.byref(lay)))
    return {n: getattr(lay, n) for n in LAYOUT_FIELDS}


def workspace_size(desc: LayerDesc) -> Tuple[int, int]:
    """(ws_bytes, ctx_bytes) for a descriptor (mok_workspace_size)."""
    ws, ctx = ctypes.c_size_t(), ctypes.c_size_t()
    _check("mok_workspace_size", load().mok_workspace_size(ctypes.byref(desc), ctypes.byref(ws), ctypes.byref(ctx)))
    return int(ws.value), int(ctx.value)


def min_minibatch(n_sm: int, I: int) -> int:
    return int(load().mok_min_minibatch(n_sm, I))


def status_string(code: int) -> str:
    return load().mok_status_string(code).decode()


def _expect(t, shape, dtype, name, nullable=False):
    """The C ABI takes bare pointers, so buffer sizes and dtypes are checked here, on the host."""
    if t is None:
        if nullable:
            return
        raise ValueError(f"{name} is required")
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype:
        raise ValueError(f"{name}: expected {tuple(shape)} {dtype}, got {tuple(t.shape)} {t.dtype}")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")


def _check_layer_inputs(desc, x, w_router, router_bias, w13, w2, w2_f16=False):
    bf = torch.bfloat16
    _expect(x, (desc.T, desc.H), bf, "x")
    _expect(w_router, (desc.E, desc.H), bf, "w_router")
    _expect(router_bias, (desc.E,), torch.float32, "router_bias", nullable=True)
    _expect(w13, (desc.E, 2 * desc.I, desc.H), bf, "w13")
    _expect(w2, (desc.E, desc.H, desc.I), torch.float16 if w2_f16 else bf, "w2")


def schedule(desc, x, w_router, router_bias, given_topk, topk_idx, gates, counts, offsets, row_of, src_of, ws,
             stream=None):
    R = desc.T * desc.k
    if x is not None:
        _expect(x, (desc.T, desc.H), torch.bfloat16, "x")
        _expect(w_router, (desc.E, desc.H), torch.bfloat16, "w_router")
    _expect(router_bias, (desc.E,), torch.float32, "router_bias", nullable=True)
    _expect(given_topk, (desc.T, desc.k), torch.int32, "given_topk", nullable=True)
    _expect(topk_idx, (desc.T, desc.k), torch.int32, "topk_idx")
    _expect(gates, (desc.T, desc.k), torch.float32, "gates", nullable=True)
    _expect(counts, (desc.E,), torch.int32, "counts")
    _expect(offsets, (desc.E + 1,), torch.int32, "offsets")
    _expect(row_of, (R,), torch.int32, "row_of")
    _expect(src_of, (R,), torch.int32, "src_of")
    _check("mok_schedule", load().mok_schedule(
        ctypes.byref(desc), _ptr(x), _ptr(w_router), _ptr(router_bias), _ptr(given_topk), _ptr(topk_idx),
        _ptr(gates), _ptr(counts), _ptr(offsets), _ptr(row_of), _ptr(src_of), *_buf(ws, "ws"),
        _stream(stream)))


def moe_forward(desc, x, w_router, router_bias, given_topk, w13, w2, y, ctx, ws, stream=None):
    _check_layer_inputs(desc, x, w_router, router_bias, w13, w2, w2_f16=bool(desc.flags & FLAG_W2_F16))
    _expect(given_topk, (desc.T, desc.k), torch.int32, "given_topk", nullable=True)
    _expect(y, (desc.T, desc.H), torch.bfloat16, "y")
    _check("mok_moe_forward", load().mok_moe_forward(
        ctypes.byref(desc), _ptr(x), _ptr(w_router), _ptr(router_bias), _ptr(given_topk), _ptr(w13), _ptr(w2),
        _ptr(y), *_buf(ctx, "ctx"), *_buf(ws, "ws"), _stream(stream)))


def moe_backward(desc, dy, x, w_router, w13, w2, ctx, dx, dw_router, dw13, dw2, dgates, ws, stream=None):
    _check_layer_inputs(desc, x, w_router, None, w13, w2)
    wdt = torch.bfloat16 if (desc.flags & FLAG_WGRAD_BF16) else torch.float32
    _expect(dy, (desc.T, desc.H), torch.bfloat16, "dy")
    _expect(dx, (desc.T, desc.H), torch.bfloat16, "dx")
    _expect(dw_router, (desc.E, desc.H), torch.float32, "dw_router")
    _expect(dw13, (desc.E, 2 * desc.I, desc.H), wdt, "dw13")
    _expect(dw2, (desc.E, desc.H, desc.I), wdt, "dw2")
    _expect(dgates, (desc.T, desc.k), torch.float32, "dgates", nullable=True)
    _check("mok_moe_backward", load().mok_moe_backward(
        ctypes.byref(desc), _ptr(dy), _ptr(x), _ptr(w_router), _ptr(w13), _ptr(w2), *_buf(ctx, "ctx"),
        _ptr(dx), _ptr(dw_router), _ptr(dw13), _ptr(dw2), _ptr(dgates), *_buf(ws, "ws"), _stream(stream)))


def read_status(ws, stream=None):
    """Synchronises the stream and returns (code, site) of the first device-side error, then clears it."""
    out = (ctypes.c_int32 * 2)()
    _check("mok_read_status", load().mok_read_status(*_buf(ws, "ws"), _stream(stream), out))
    return int(out[0]), int(out[1])


def trace_start(max_launches: int = 4096):
    """Starts per-kernel CUDA-event timing of every launch the library makes."""
    _check("mok_trace_start", load().mok_trace_start(max_launches))


def trace_stop() -> Dict[str, Dict[str, float]]:
    """Stops timing; returns {kernel: {"launches": n, "total_ms": t}} in first-launch order."""
    cap = 64
    arr = (TraceEntry * cap)()
    n = ctypes.c_int32(0)
    _check("mok_trace_stop", load().mok_trace_stop(arr, cap, ctypes.byref(n)))
    return {arr[i].name.decode(): {"launches": int(arr[i].launches), "total_ms": float(arr[i].total_ms)}
            for i in range(n.value)}


def test_bounded_wait(ws, limit_ms: int, stream=None):
    _check("mok_test_bounded_wait",
           load().mok_test_bounded_wait(*_buf(ws, "ws"), limit_ms, _stream(stream)))


_CTX_DTYPES = {"topk_idx": torch.int32, "gates": torch.float32, "scores": torch.float32, "counts": torch.int32,
               "offsets": torch.int32, "row_of": torch.int32, "src_of": torch.int32, "tile_off": torch.int32,
               "gate_row": torch.float32, "x_g": torch.bfloat16, "hu": torch.float32, "ring_stamp": torch.int64, "ring": torch.bfloat16, "status": torch.int32,
               "logits": torch.float32, "sched": torch.int32, "act": torch.bfloat16, "act_lo": torch.bfloat16,
               "expert_out": torch.float32, "dy_g": torch.bfloat16, "dhu": torch.bfloat16, "dhu_lo": torch.bfloat16,
               "gact": torch.bfloat16, "gact_lo": torch.bfloat16, "dx_g": torch.float32,
               "dg_part": torch.float32, "dlogits": torch.float32,
               "mx_dhu_r": torch.bfloat16, "mx_xg_r": torch.bfloat16, "mx_do_r": torch.bfloat16,
               "mx_a_r": torch.bfloat16, "mx_blk_off": torch.int32, "mx_xq": torch.uint8, "mx_xsf": torch.uint8,
               "mx_aq": torch.uint8, "mx_asf": torch.uint8, "mx_dyq": torch.uint8, "mx_dysf": torch.uint8,
               "mx_dhuq": torch.uint8, "mx_dhusf": torch.uint8}


def mx_rows_padded_bound(R: int, E: int) -> int:
    """Rows of the MXFP8 padded row space (include/mok.h, mok_layout.mx_xq): 32 (ceil(R / 32) + E)."""
    return 32 * ((R + 31) // 32 + E)


def mx_row_groups(R: int, E: int) -> int:
    """Row groups of the MXFP8 scale blocks: padded rows / 32 + 4."""
    return mx_rows_padded_bound(R, E) // 32 + 4


class MoELayer:
    """One layer descriptor with its ctx and ws buffers (torch-allocated device memory)."""

    def __init__(self, desc: LayerDesc, device="cuda"):
        self.desc = desc
        self.layout = get_layout(desc)
        self.ctx = torch.empty(self.layout["ctx_bytes"], dtype=torch.uint8, device=device)
        self.ws = torch.zeros(self.layout["ws_bytes"], dtype=torch.uint8, device=device)

    def ring_rows(self) -> int:
        """Rows of the ring forward's dispatched-row region (whole minibatches)."""
        d = self.desc
        R = d.T * d.k
        m = d.minibatch if d.minibatch > 0 else min_minibatch(0, d.I)
        m = min(m, R)
        return -(-R // m) * m

    def _shape(self, name):
        d = self.desc
        R = d.T * d.k
        if name == "ring":
            return (self.ring_rows(), d.H)
        return {"topk_idx": (d.T, d.k), "gates": (d.T, d.k), "scores": (d.T, d.E), "counts": (d.E,),
                "offsets": (d.E + 1,), "row_of": (R,), "src_of": (R,), "tile_off": (d.E + 1,), "gate_row": (R,),
                "x_g": (R, d.H), "hu": (R, 2 * d.I), "ring_stamp": (2,), "status": (4,), "logits": (d.T, d.E), "sched": (-(-R // 1024), d.E), "act": (R, d.I),
                "act_lo": (R, d.I), "expert_out": (R, d.H), "dy_g": (R, d.H), "dhu": (R, 2 * d.I),
                "dhu_lo": (R, 2 * d.I), "gact": (R, d.I), "gact_lo": (R, d.I),
                "dx_g": (R, d.H), "dg_part": (R, d.I // 128), "dlogits": (d.T, d.E), "mx_dhu_r": (R, 2 * d.I), "mx_xg_r": (R, d.H), "mx_do_r": (R, d.H), "mx_a_r": (R, d.I),
                "mx_blk_off": (d.E + 1,), "mx_xq": (mx_rows_padded_bound(R, d.E), d.H),
                "mx_xsf": (mx_row_groups(R, d.E), d.H // 128, 512), "mx_aq": (mx_rows_padded_bound(R, d.E), d.I),
                "mx_asf": (mx_row_groups(R, d.E), d.I // 128, 512), "mx_dyq": (mx_rows_padded_bound(R, d.E), d.H),
                "mx_dysf": (mx_row_groups(R, d.E), d.H // 128, 512),
                "mx_dhuq": (mx_rows_padded_bound(R, d.E), 2 * d.I),
                "mx_dhusf": (mx_row_groups(R, d.E), 2 * d.I // 128, 512)}[name]

    def view_split(self, name: str) -> torch.Tensor:
        """hi + lo of a split operand ("act", "dhu", "gact") as one float32 tensor."""
        return self.view(name).float() + self.view(name + "_lo").float()

    def view(self, name: str) -> torch.Tensor:
        """A typed view of one saved tensor (ctx) or temporary (ws)."""
        buf = self.ctx if name in CTX_FIELDS else self.ws
        off = self.layout[name]
        dt = _CTX_DTYPES[name]
        shape = self._shape(name)
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dt).element_size()
        return buf[off:off + nbytes].view(dt).view(shape)

    def forward(self, x, w_router, w13, w2, router_bias=None, given_topk=None, y=None, stream=None):
        if y is None:
            y = torch.empty((self.desc.T, self.desc.H), dtype=torch.bfloat16, device=x.device)
        moe_forward(self.desc, x, w_router, router_bias, given_topk, w13, w2, y, self.ctx, self.ws, stream)
        return y

    def backward(self, dy, x, w_router, w13, w2, out=None, stream=None):
        d = self.desc
        dev = dy.device
        if out is None:
            wdt = torch.bfloat16 if (d.flags & FLAG_WGRAD_BF16) else torch.float32
            out = {"dx": torch.empty((d.T, d.H), dtype=torch.bfloat16, device=dev),
                   "dw_router": torch.empty((d.E, d.H), dtype=torch.float32, device=dev),
                   "dw13": torch.empty((d.E, 2 * d.I, d.H), dtype=wdt, device=dev),
                   "dw2": torch.empty((d.E, d.H, d.I), dtype=wdt, device=dev),
                   "dgates": torch.empty((d.T, d.k), dtype=torch.float32, device=dev)}
        moe_backward(d, dy, x, w_router, w13, w2, self.ctx, out["dx"], out["dw_router"], out["dw13"], out["dw2"],
                     out["dgates"], self.ws, stream)
        return out

    def backward_mxfp8(self, dy, x, w_router, wb, out=None, stream=None):
        """mok_moe_backward_mxfp8 after forward_mxfp8; ``wb`` from quantize_weights_backward."""
        d = self.desc
        dev = dy.device
        if out is None:
            wdt = torch.bfloat16 if (d.flags & FLAG_WGRAD_BF16) else torch.float32
            out = {"dx": torch.empty((d.T, d.H), dtype=torch.bfloat16, device=dev),
                   "dw_router": torch.empty((d.E, d.H), dtype=torch.float32, device=dev),
                   "dw13": torch.empty((d.E, 2 * d.I, d.H), dtype=wdt, device=dev),
                   "dw2": torch.empty((d.E, d.H, d.I), dtype=wdt, device=dev),
                   "dgates": torch.empty((d.T, d.k), dtype=torch.float32, device=dev)}
        moe_backward_mxfp8(d, dy, x, w_router, wb, self.ctx, out["dx"], out["dw_router"], out["dw13"], out["dw2"],
                           out["dgates"], self.ws, stream)
        return out

    def status(self, stream=None):
        return read_status(self.ws, stream)


def schedule_noalloc(desc, x, w_router, router_bias, given_topk, topk_idx, gates, counts, offsets, row_of, src_of,
                     device_status=None, stream=None):
    """mok_schedule_noalloc: the router and schedule table with the library's own fixed scratch,
    for callers that cannot allocate a workspace.  Same outputs as ``schedule``;
    ``device_status`` (optional int32 [2] CUDA tensor) receives (code, site) of a device error."""
    lib = load()
    fn = lib.mok_schedule_noalloc
    if fn.argtypes is None:
        P = ctypes.c_void_p
        fn.argtypes = [ctypes.POINTER(LayerDesc), P, P, P, P, P, P, P, P, P, P, P, P]
        fn.restype = ctypes.c_int32
    R = desc.T * desc.k
    if x is not None:
        _expect(x, (desc.T, desc.H), torch.bfloat16, "x")
        _expect(w_router, (desc.E, desc.H), torch.bfloat16, "w_router")
    _expect(router_bias, (desc.E,), torch.float32, "router_bias", nullable=True)
    _expect(given_topk, (desc.T, desc.k), torch.int32, "given_topk", nullable=True)
    _expect(topk_idx, (desc.T, desc.k), torch.int32, "topk_idx")
    _expect(gates, (desc.T, desc.k), torch.float32, "gates", nullable=True)
    _expect(counts, (desc.E,), torch.int32, "counts")
    _expect(offsets, (desc.E + 1,), torch.int32, "offsets")
    _expect(row_of, (R,), torch.int32, "row_of")
    _expect(src_of, (R,), torch.int32, "src_of")
    _expect(device_status, (2,), torch.int32, "device_status", nullable=True)
    _check("mok_schedule_noalloc", fn(
        ctypes.byref(desc), _ptr(x), _ptr(w_router), _ptr(router_bias), _ptr(given_topk), _ptr(topk_idx),
        _ptr(gates), _ptr(counts), _ptr(offsets), _ptr(row_of), _ptr(src_of), _ptr(device_status),
        _stream(stream)))


def _mx_fn(name, nargs):
    fn = getattr(load(), name)
    if fn.argtypes is None:
        fn.argtypes = [ctypes.POINTER(LayerDesc)] + [ctypes.c_void_p] * nargs
        fn.restype = ctypes.c_int32
    return fn


def convert_f16(src, stream=None):
    """mok_convert_f16: an fp16 copy of a bf16 CUDA tensor (round to nearest even), e.g. W2 for
    MOK_FLAG_W2_F16."""
    if src is None or src.device.type != "cuda" or src.dtype != torch.bfloat16:
        raise ValueError("convert_f16 takes a bf16 CUDA tensor")
    out = torch.empty(src.shape, dtype=torch.float16, device=src.device)
    fn = load().mok_convert_f16
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    fn.restype = ctypes.c_int32
    _check("mok_convert_f16", fn(_ptr(src), _ptr(out), src.numel(), _stream(stream)))
    return out


def quantize_weights(desc, w13, w2, stream=None):
    """mok_quantize_weights: MXFP8 (E4M3 + E8M0 per 32 along K) copies of the expert weights.
    Returns {"w13_q", "w13_scale", "w2_q", "w2_scale"} as uint8 CUDA tensors."""
    _expect(w13, (desc.E, 2 * desc.I, desc.H), torch.bfloat16, "w13")
    _expect(w2, (desc.E, desc.H, desc.I), torch.bfloat16, "w2")
    dev = w13.device
    E, H, I = desc.E, desc.H, desc.I
    out = {"w13_q": torch.empty((E, 2 * I, H), dtype=torch.uint8, device=dev),
           "w13_scale": torch.empty((E, I // 64, H // 128, 512), dtype=torch.uint8, device=dev),
           "w2_q": torch.empty((E, H, I), dtype=torch.uint8, device=dev),
           "w2_scale": torch.empty((E, H // 128, I // 128, 512), dtype=torch.uint8, device=dev)}
    fn = load().mok_quantize_weights
    fn.argtypes = [ctypes.POINTER(LayerDesc)] + [ctypes.c_void_p] * 7
    fn.restype = ctypes.c_int32
    _check("mok_quantize_weights", fn(ctypes.byref(desc), _ptr(w13), _ptr(w2), _ptr(out["w13_q"]),
                                      _ptr(out["w13_scale"]), _ptr(out["w2_q"]), _ptr(out["w2_scale"]),
                                      _stream(stream)))
    return out


def moe_forward_mxfp8(desc, x, w_router, router_bias, given_topk, wq, y, ctx, ws, stream=None):
    """mok_moe_forward_mxfp8 with the weights of ``quantize_weights``."""
    E, H, I = desc.E, desc.H, desc.I
    _expect(x, (desc.T, H), torch.bfloat16, "x")
    _expect(w_router, (E, H), torch.bfloat16, "w_router")
    _expect(router_bias, (E,), torch.float32, "router_bias", nullable=True)
    _expect(given_topk, (desc.T, desc.k), torch.int32, "given_topk", nullable=True)
    _expect(wq["w13_q"], (E, 2 * I, H), torch.uint8, "w13_q")
    _expect(wq["w13_scale"], (E, I // 64, H // 128, 512), torch.uint8, "w13_scale")
    _expect(wq["w2_q"], (E, H, I), torch.uint8, "w2_q")
    _expect(wq["w2_scale"], (E, H // 128, I // 128, 512), torch.uint8, "w2_scale")
    _expect(y, (desc.T, H), torch.bfloat16, "y")
    fn = load().mok_moe_forward_mxfp8
    P, SZ = ctypes.c_void_p, ctypes.c_size_t
    fn.argtypes = [ctypes.POINTER(LayerDesc), P, P, P, P, P, P, P, P, P, P, SZ, P, SZ, P]
    fn.restype = ctypes.c_int32
    _check("mok_moe_forward_mxfp8", fn(
        ctypes.byref(desc), _ptr(x), _ptr(w_router), _ptr(router_bias), _ptr(given_topk), _ptr(wq["w13_q"]),
        _ptr(wq["w13_scale"]), _ptr(wq["w2_q"]), _ptr(wq["w2_scale"]), _ptr(y), *_buf(ctx, "ctx"),
        *_buf(ws, "ws"), _stream(stream)))
    return y


def quantize_weights_backward(desc, w13, w2, stream=None):
    """mok_quantize_weights_backward: W2 transposed to [E][I][H] and quantised along H, W13 transposed to
    [E][H][2I] and quantised along 2I (E4M3 + scale blocks).  Returns {"w13t_q", "w13t_scale", "w2t_q",
    "w2t_scale"} as uint8 CUDA tensors."""
    _expect(w13, (desc.E, 2 * desc.I, desc.H), torch.bfloat16, "w13")
    _expect(w2, (desc.E, desc.H, desc.I), torch.bfloat16, "w2")
    dev = w13.device
    E, H, I = desc.E, desc.H, desc.I
    out = {"w13t_q": torch.empty((E, H, 2 * I), dtype=torch.uint8, device=dev),
           "w13t_scale": torch.empty((E, H // 128, 2 * I // 128, 512), dtype=torch.uint8, device=dev),
           "w2t_q": torch.empty((E, I, H), dtype=torch.uint8, device=dev),
           "w2t_scale": torch.empty((E, I // 128, H // 128, 512), dtype=torch.uint8, device=dev)}
    fn = _mx_fn("mok_quantize_weights_backward", 7)
    _check("mok_quantize_weights_backward", fn(ctypes.byref(desc), _ptr(w13), _ptr(w2), _ptr(out["w13t_q"]),
                                               _ptr(out["w13t_scale"]), _ptr(out["w2t_q"]), _ptr(out["w2t_scale"]),
                                               _stream(stream)))
    return out


def moe_backward_mxfp8(desc, dy, x, w_router, wb, ctx, dx, dw_router, dw13, dw2, dgates, ws, stream=None):
    """mok_moe_backward_mxfp8 with the weights of ``quantize_weights_backward``."""
    E, H, I = desc.E, desc.H, desc.I
    wdt = torch.bfloat16 if (desc.flags & FLAG_WGRAD_BF16) else torch.float32
    _expect(x, (desc.T, H), torch.bfloat16, "x")
    _expect(w_router, (E, H), torch.bfloat16, "w_router")
    _expect(wb["w13t_q"], (E, H, 2 * I), torch.uint8, "w13t_q")
    _expect(wb["w13t_scale"], (E, H // 128, 2 * I // 128, 512), torch.uint8, "w13t_scale")
    _expect(wb["w2t_q"], (E, I, H), torch.uint8, "w2t_q")
    _expect(wb["w2t_scale"], (E, I // 128, H // 128, 512), torch.uint8, "w2t_scale")
    _expect(dy, (desc.T, H), torch.bfloat16, "dy")
    _expect(dx, (desc.T, H), torch.bfloat16, "dx")
    _expect(dw_router, (E, H), torch.float32, "dw_router")
    _expect(dw13, (E, 2 * I, H), wdt, "dw13")
    _expect(dw2, (E, H, I), wdt, "dw2")
    _expect(dgates, (desc.T, desc.k), torch.float32, "dgates", nullable=True)
    fn = load().mok_moe_backward_mxfp8
    P, SZ = ctypes.c_void_p, ctypes.c_size_t
    fn.argtypes = [ctypes.POINTER(LayerDesc), P, P, P, P, P, P, P, P, SZ, P, P, P, P, P, P, SZ, P]
    fn.restype = ctypes.c_int32
    _check("mok_moe_backward_mxfp8", fn(
        ctypes.byref(desc), _ptr(dy), _ptr(x), _ptr(w_router), _ptr(wb["w13t_q"]), _ptr(wb["w13t_scale"]),
        _ptr(wb["w2t_q"]), _ptr(wb["w2t_scale"]), *_buf(ctx, "ctx"), _ptr(dx), _ptr(dw_router), _ptr(dw13),
        _ptr(dw2), _ptr(dgates), *_buf(ws, "ws"), _stream(stream)))
