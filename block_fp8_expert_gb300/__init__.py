"""GB300-native block-FP8 (E4M3) Mixture-of-Experts FFN layer.

The layer runs in ``libmoe_fp8.so`` (hand-written sm_103a CUDA kernels behind
the C ABI in ``include/moe_fp8.h``).  This package is its thin Python binding:
``_lib`` (ctypes, one function per C entry point) and ``device`` (weights held
in HBM as PyTorch tensors, plus a forward call).  It never computes any part of
the layer itself and has no CPU fallback.
"""
from ._lib import (  # noqa: F401
    Dims, Fp8Ffn, Fp8Mat, MoeError, dims, ffn, lib, version, workspace_bytes,
    moe_route, moe_permute, moe_expert_ffn_fp8, moe_combine, moe_layer_forward,
    moe_layer_forward_gated, moe_layer_forward_act8,
    moe_read_device_status, kernel_launches, expert_uses_gemm,
)
