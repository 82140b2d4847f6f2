"""Single-GPU deterministic mixture-of-experts layer for GB300 (sm_103a).

The compute path is libmok.so (C ABI in include/mok.h, CUDA kernels under
csrc/); this package only binds it (``_native``) and draws seeded synthetic
workloads (``workloads``).
"""
from ._native import (FLAG_GEMM_PAIR, FLAG_GEMM_SINGLE, FLAG_RING_PERSISTENT, FLAG_W2_F16,  # noqa: F401
                      FLAG_WGRAD_BF16,
                      LayerDesc, MoELayer, MokError, convert_f16, desc_from_shape, get_layout, load, make_desc,
                      min_minibatch, moe_backward, moe_backward_mxfp8, moe_forward, moe_forward_mxfp8,
                      quantize_weights, quantize_weights_backward, read_status, schedule, status_string,
                      workspace_size)
