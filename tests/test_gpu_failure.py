"""Failure detection on the GPU without a fault: a bounded device wait that
runs out.

The layer call's down GEMM waits, per token tile, until the gate/up GEMM has
stored that tile's SwiGLU rows (a counter the gate/up epilogue raises).
MOE_FP8_TEST_STALL=down makes it wait for one more completion than will ever
come, and MOE_FP8_WAIT_LIMIT_US shortens every bounded wait of the GEMMs, so
the wait runs out after a few milliseconds.  The kernel must then record
MOE_DEV_WAIT_TIMEOUT and where it gave up, drain its copies, free its tensor
memory and exit; the context stays usable and the next call, without the
stall, is clean and correct.
"""
import numpy as np
import pytest

import moe_inputs as mi
import oracle
from gpu_common import assert_within_tol, bf16_bits, host_layer, require_gpu

pytestmark = pytest.mark.gpu


def test_down_gemm_wait_runs_out_then_next_call_is_clean(monkeypatch):
    torch = require_gpu()
    import block_fp8_expert_gb300 as m
    from block_fp8_expert_gb300 import _lib
    from block_fp8_expert_gb300.device import DeviceLayer, x_to_device
    L = host_layer("qwen3moe_decode")
    D = DeviceLayer.from_host(L)
    T = 64
    assert m.expert_uses_gemm(D.dims(T))  # the tensor-core GEMM regime
    xb, _ = mi.make_tokens(L, T, seed=13)
    x = x_to_device(xb)
    ws = D.workspace(T)

    monkeypatch.setenv("MOE_FP8_TEST_STALL", "down")
    monkeypatch.setenv("MOE_FP8_WAIT_LIMIT_US", "2000")
    D.forward(x, ws=ws)
    torch.cuda.synchronize()  # the kernels returned: nothing hangs
    words = ws[:64].view(torch.int32).cpu().numpy()[:16]
    assert words[0] & _lib.MOE_DEV_WAIT_TIMEOUT, words[:6]
    with pytest.raises(m.MoeError):
        m.moe_read_device_status(ws)
    # where the first wait of the grid gave up (word 1 = warp + 1, word 2 =
    # barrier id): the stalled token warp (warp 1, id 9: a token tile's hid
    # rows), or one of the roles waiting behind it in the same CTA, whose
    # budgets start at about the same time
    assert 1 <= words[1] <= 19 and 1 <= words[2] <= 9, words[:6]
    if words[2] == 9:
        # that tile had all of its real completions, but not the extra one
        assert words[1] == 2 and words[4] == (L.I // 128) * 8, words[:6]

    monkeypatch.delenv("MOE_FP8_TEST_STALL")
    monkeypatch.delenv("MOE_FP8_WAIT_LIMIT_US")
    out = D.forward(x, ws=ws)
    assert m.moe_read_device_status(ws) == 0
    ref = oracle.moe_layer(xb, L, keep_intermediates=False)
    assert_within_tol(oracle.bf16_to_f64(bf16_bits(out)), ref["out"], "after the timeout")


def test_short_wait_limit_alone_changes_nothing(monkeypatch):
    """A short limit without the stall: every wait still ends in time."""
    torch = require_gpu()
    import block_fp8_expert_gb300 as m
    from block_fp8_expert_gb300.device import DeviceLayer, x_to_device
    L = host_layer("qwen3moe_decode")
    D = DeviceLayer.from_host(L)
    xb, _ = mi.make_tokens(L, 64, seed=14)
    ws = D.workspace(64)
    monkeypatch.setenv("MOE_FP8_WAIT_LIMIT_US", "20000")
    out = D.forward(x_to_device(xb), ws=ws)
    assert m.moe_read_device_status(ws) == 0
    ref = oracle.moe_layer(xb, L, keep_intermediates=False)
    assert_within_tol(oracle.bf16_to_f64(bf16_bits(out)), ref["out"], "short wait limit")
    np.testing.assert_equal(torch.isfinite(out.float()).all().item(), True)
