"""fp64 CPU oracle for the block-FP8 (E4M3) Mixture-of-Experts FFN layer.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import anything under ``oracle/``.  The CUDA library
never calls it and shares no code with it.

Every function states the layer from its plain definition, in float64, with
NumPy primitives (matmul, sort, exp) as its only helpers.  The pages this
follows name the ingredients of the layer but print no formulas; each reading
taken where they are silent is stated at the function that takes it.

Parity pins: every function here is pinned by a ``-m "not gpu"`` test against
something other than itself (closed forms, brute force, invariants, a library
FP8 decode).  The whole-layer output beyond the tiny workload is pinned by the
composition of those pinned parts plus a scalar brute-force loop on the tiny
workload; no page prints a layer output to compare against.
"""
from .moe_ref import (  # noqa: F401
    BLOCK,
    e4m3_decode,
    e4m3_table,
    bf16_to_f64,
    dequantize,
    router_logits,
    softmax,
    topk_renorm,
    permute,
    silu,
    expert_ffn,
    e4m3_encode_rne,
    act8_quantize,
    act8_dequantize,
    act8_round,
    expert_ffn_act8,
    combine,
    shared_gate_factor,
    moe_layer,
    moe_layer_sampled,
)
