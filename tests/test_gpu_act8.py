"""The layer on E4M3 activations (moe_layer_forward_act8) against the
oracle's FP8-activation variant (reading R11 of the oracle): routing exact,
outputs within the layer tolerance.  x is quantised from the same bf16 bits
in the same float32 steps on both sides, so its codes agree exactly; hid is
quantised from float32 sums that the two sides form in different orders, so
an element near a rounding boundary can take the neighbouring code, which
moves its output row by well under the tolerance."""
import numpy as np
import pytest

import moe_inputs as mi
import oracle
from gpu_common import assert_within_tol, bf16_bits, host_layer, require_gpu

pytestmark = pytest.mark.gpu


def _run(name, T, seed=0, act8=True):
    torch = require_gpu()
    from block_fp8_expert_gb300.device import DeviceLayer, x_to_device
    L = host_layer(name)
    D = DeviceLayer.from_host(L)
    xb, _ = mi.make_tokens(L, T, seed=seed)
    x = x_to_device(xb)
    idx = torch.empty((T, L.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, L.k), dtype=torch.float32, device="cuda")
    ws = D.workspace(T)
    out = D.forward(x, ws=ws, topk_idx=idx, topk_w=w, act8=act8)
    torch.cuda.synchronize()
    import block_fp8_expert_gb300 as m
    assert m.moe_read_device_status(ws) == 0
    return L, xb, bf16_bits(out), idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("name,T", [("tiny", 8), ("qwen3moe_decode", 64), ("qwen3moe_decode", 1),
                                    ("qwen3moe_decode", 3), ("skewed", 16)])
def test_act8_layer_matches_oracle(name, T):
    L, xb, out, idx, w = _run(name, T)
    ref = oracle.moe_layer(xb, L, act8=True, keep_intermediates=False)
    assert np.array_equal(idx, ref["topk_idx"])
    assert_within_tol(oracle.bf16_to_f64(out), ref["out"], f"{name} T={T} act8")


@pytest.mark.parametrize("name,T", [("qwen3moe_prefill", 4096), ("skewed", 2048)])
def test_act8_layer_sampled_at_full_size(name, T):
    L, xb, out, idx, w = _run(name, T)
    tokens = np.linspace(0, T - 1, 24).astype(np.int64)
    ref = oracle.moe_layer_sampled(xb, L, tokens, act8=True)
    assert np.array_equal(idx, ref["topk_idx"])
    assert_within_tol(oracle.bf16_to_f64(out)[tokens], ref["out_sampled"], f"{name} T={T} act8")


def test_act8_differs_from_bf16_activations_by_the_quantisation():
    L, xb, out8, _, _ = _run("qwen3moe_decode", 64)
    _, _, out16, _, _ = _run("qwen3moe_decode", 64, act8=False)
    a, b = oracle.bf16_to_f64(out8), oracle.bf16_to_f64(out16)
    rms = np.sqrt(np.mean(b ** 2))
    e = np.sqrt(np.mean((a - b) ** 2)) / rms
    assert 0.02 < e < 0.08, e  # the oracle's own study: about 4.5%


def test_act8_rejects_a_shared_expert():
    require_gpu()
    import block_fp8_expert_gb300 as m
    with pytest.raises(m.MoeError):
        _run("large_sparse", 4)
