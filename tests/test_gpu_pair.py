"""The tensor-core GEMM in CTA pairs (two SMs per tile, cta_group::2),
forced with MOE_FP8_GEMM_PAIR=1 on shapes where the host rule would not pick
it, and compared with the single-CTA GEMM (MOE_FP8_GEMM_PAIR=0) and with the
fp64 oracle.

A pair computes each output element from the same products, in the same K
order, as a single CTA does (the pair's M = 256 MMA is the single CTA's two
M = 128 MMAs side by side); both must be within the layer tolerance of the
oracle, and they must agree with each other much more closely than that.
The shapes cover full token tiles, ragged tails (N rounded to 32 and split
in halves between the two CTAs), experts with no rows, and the layer call.
"""
import numpy as np
import pytest

import moe_inputs as mi
import oracle
from gpu_common import W_REL, assert_within_tol, bf16_bits, host_layer, require_gpu

pytestmark = pytest.mark.gpu


def _ffn(torch, D, L, xb, ref):
    import block_fp8_expert_gb300 as m
    from block_fp8_expert_gb300.device import x_to_device
    T = xb.shape[0]
    ws = D.workspace(T)
    y = torch.full((T * L.k, L.H), float("nan"), dtype=torch.float32, device="cuda")
    m.moe_expert_ffn_fp8(x_to_device(xb), torch.from_numpy(ref["expert_off"]).cuda(),
                         torch.from_numpy(ref["row_token"]).cuda(), D.routed.abi(), D.dims(T), y,
                         ws)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(ws) == 0
    return y.cpu().numpy()


@pytest.mark.parametrize("T,E,k", [(200, 4, 2), (96, 8, 2), (1000, 16, 4)])
def test_pair_expert_ffn_matches_single_cta_and_oracle(monkeypatch, T, E, k):
    torch = require_gpu()
    import block_fp8_expert_gb300 as m
    from block_fp8_expert_gb300.device import DeviceLayer
    w_ = mi.Workload("pair_small", H=512, I=256, E=E, k=k)
    L = mi.make_layer(w_, seed=60 + T)
    D = DeviceLayer.from_host(L)
    xb, _ = mi.make_tokens(L, T, seed=61)
    ref = oracle.moe_layer(xb, L)
    monkeypatch.setenv("MOE_FP8_EXPERT_PATH", "gemm")
    assert m.expert_uses_gemm(D.dims(T))
    monkeypatch.setenv("MOE_FP8_GEMM_PAIR", "1")
    yp = _ffn(torch, D, L, xb, ref)
    monkeypatch.setenv("MOE_FP8_GEMM_PAIR", "0")
    ys = _ffn(torch, D, L, xb, ref)
    assert_within_tol(yp, ref["y_perm"], f"pair y_perm T={T} E={E}")
    assert_within_tol(ys, ref["y_perm"], f"single-CTA y_perm T={T} E={E}")
    # same products, same K order: agreement far inside the tolerance
    assert_within_tol(yp, ys, "pair vs single CTA", rel=1e-5)


@pytest.mark.parametrize("name,T", [("qwen3moe_decode", 64), ("skewed", 256),
                                    ("large_sparse", 256)])
def test_pair_layer_forced(monkeypatch, name, T):
    torch = require_gpu()
    from block_fp8_expert_gb300.device import DeviceLayer, x_to_device
    L = host_layer(name)
    D = DeviceLayer.from_host(L)
    xb, _ = mi.make_tokens(L, T, seed=62)
    monkeypatch.setenv("MOE_FP8_EXPERT_PATH", "gemm")
    monkeypatch.setenv("MOE_FP8_GEMM_PAIR", "1")
    idx = torch.empty((T, L.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, L.k), dtype=torch.float32, device="cuda")
    ws = D.workspace(T)
    out = D.forward(x_to_device(xb), ws=ws, topk_idx=idx, topk_w=w)
    torch.cuda.synchronize()
    words = ws[:32].view(torch.int32).cpu().numpy()
    assert words[0] == 0, f"device status {words[:6].tolist()}"
    ref = oracle.moe_layer(xb, L, keep_intermediates=False)
    assert np.array_equal(idx.cpu().numpy(), ref["topk_idx"])
    assert_within_tol(w.cpu().numpy(), ref["topk_w"], "topk_w", rel=W_REL)
    assert_within_tol(oracle.bf16_to_f64(bf16_bits(out)), ref["out"], f"pair {name} T={T}")


def test_pair_wait_runs_out_then_next_call_is_clean(monkeypatch):
    """The failure path of the pair GEMM: the down projection's token warps
    wait for a gate/up completion that never comes (MOE_FP8_TEST_STALL=down)
    with a 2 ms limit; both CTAs of every pair give up, drain and free their
    tensor memory, and the next call is clean."""
    torch = require_gpu()
    import block_fp8_expert_gb300 as m
    from block_fp8_expert_gb300 import _lib
    from block_fp8_expert_gb300.device import DeviceLayer, x_to_device
    w_ = mi.Workload("pair_small", H=512, I=256, E=4, k=2)
    L = mi.make_layer(w_, seed=63)
    D = DeviceLayer.from_host(L)
    T = 400
    xb, _ = mi.make_tokens(L, T, seed=64)
    x = x_to_device(xb)
    ws = D.workspace(T)
    monkeypatch.setenv("MOE_FP8_EXPERT_PATH", "gemm")
    monkeypatch.setenv("MOE_FP8_GEMM_PAIR", "1")
    monkeypatch.setenv("MOE_FP8_TEST_STALL", "down")
    monkeypatch.setenv("MOE_FP8_WAIT_LIMIT_US", "2000")
    D.forward(x, ws=ws)
    torch.cuda.synchronize()  # the kernels returned: nothing hangs
    words = ws[:64].view(torch.int32).cpu().numpy()[:16]
    assert words[0] & _lib.MOE_DEV_WAIT_TIMEOUT, words[:6]
    with pytest.raises(m.MoeError):
        m.moe_read_device_status(ws)
    monkeypatch.delenv("MOE_FP8_TEST_STALL")
    monkeypatch.delenv("MOE_FP8_WAIT_LIMIT_US")
    out = D.forward(x, ws=ws)
    assert m.moe_read_device_status(ws) == 0
    ref = oracle.moe_layer(xb, L, keep_intermediates=False)
    assert_within_tol(oracle.bf16_to_f64(bf16_bits(out)), ref["out"], "after the timeout")
