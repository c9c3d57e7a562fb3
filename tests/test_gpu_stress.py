"""Repeated layer calls on the same inputs give bit-identical outputs.

Every cross-role or cross-CTA hand-off of the expert kernels is a bounded
wait on a barrier or counter: the GEMM's code/token/TMEM rings, its gate/up
to down completion counters, the streamed GEMV's combine tickets.  A missed
phase or a stale read shows as a wrong value in one call out of hundreds,
not as a fault, so each case runs the layer many times back to back (no
host synchronisation in between) and compares every output with the first,
bit for bit, on the device.  The first output is also checked against the
fp64 oracle, so a repeatable wrong value cannot pass either."""
import pytest

import moe_inputs as mi
import oracle
from gpu_common import assert_within_tol, bf16_bits, host_layer, require_gpu

pytestmark = pytest.mark.gpu

CALLS = 300

CASES = [
    # streamed GEMV, combine folded into the down kernel (tickets)
    ("qwen3moe_decode", 1, None, False),
    ("qwen3moe_decode", 8, None, False),
    # tensor-core GEMM as one launch (gate/up then down tiles per CTA)
    ("qwen3moe_decode", 64, None, False),
    # tensor-core GEMM as two launches, hot experts with full 128-row tiles
    ("skewed", 256, "2", False),
    # the shared expert beside 512 routed experts
    ("large_sparse", 256, None, False),
    # E4M3 activations
    ("qwen3moe_decode", 64, None, True),
]


@pytest.mark.parametrize("name,T,launches,act8", CASES)
def test_repeated_calls_are_bit_identical(monkeypatch, name, T, launches, act8):
    torch = require_gpu()
    import block_fp8_expert_gb300 as m
    from block_fp8_expert_gb300.device import DeviceLayer, x_to_device
    if launches:
        monkeypatch.setenv("MOE_FP8_GEMM_LAUNCHES", launches)
    L = host_layer(name)
    D = DeviceLayer.from_host(L)
    xb, _ = mi.make_tokens(L, T, seed=21)
    x = x_to_device(xb)
    ws = D.workspace(T)
    first = D.forward(x, ws=ws, act8=act8).clone()
    bad = torch.zeros((), dtype=torch.int32, device="cuda")
    for _ in range(CALLS):
        out = D.forward(x, ws=ws, act8=act8)
        bad += (~torch.eq(out.view(torch.int16), first.view(torch.int16))).any().to(torch.int32)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(ws) == 0
    assert bad.item() == 0, f"{bad.item()} of {CALLS} calls differed from the first"
    ref = oracle.moe_layer(xb, L, act8=act8, keep_intermediates=False)
    assert_within_tol(oracle.bf16_to_f64(bf16_bits(first)), ref["out"],
                      f"{name} T={T} first call")
