"""The runtime cross-check (moe_verify_layer): an independent GPU
recomputation of sampled tokens of a layer call.

It must (1) accept the library's own outputs (within the layer tolerance),
(2) agree with the fp64 oracle when handed the oracle's output rounded to
bf16 (so its reference is the layer, not an echo of the fast kernels), (3)
catch a corrupted output element, and (4) report a sample with an invalid
token index as an infinite error rather than reading out of bounds.
"""
import numpy as np
import pytest

import moe_inputs as mi
import oracle
from gpu_common import host_layer, require_gpu

pytestmark = pytest.mark.gpu


def _run(torch, L, T, seed, path=None, monkeypatch=None):
    from block_fp8_expert_gb300.device import DeviceLayer, x_to_device
    if path:
        monkeypatch.setenv("MOE_FP8_EXPERT_PATH", path)
    D = DeviceLayer.from_host(L)
    xb, _ = mi.make_tokens(L, T, seed=seed)
    x = x_to_device(xb)
    idx = torch.empty((T, L.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, L.k), dtype=torch.float32, device="cuda")
    out = D.forward(x, topk_idx=idx, topk_w=w)
    torch.cuda.synchronize()
    return D, xb, x, out, idx, w


@pytest.mark.parametrize("path", ["gemv", "gemm"])
def test_verify_accepts_the_layer_output(monkeypatch, path):
    torch = require_gpu()
    L = host_layer("qwen3moe_decode")
    D, xb, x, out, idx, w = _run(torch, L, 64, 21, path, monkeypatch)
    r = D.verify(x, out, idx, w, list(range(0, 64, 4)))
    assert 0 < r["max_err_over_tol"] <= 1.0, r
    assert r["rms_ref"] > 0


def test_verify_agrees_with_the_oracle_and_catches_a_corrupted_element():
    torch = require_gpu()
    w_ = mi.Workload("shared_mid", H=512, I=256, E=32, k=4, I_shared=256)
    L = mi.make_layer(w_, seed=22, shared_gated=True)
    D, xb, x, out, idx, w = _run(torch, L, 12, 22)
    toks = [0, 3, 7, 11]
    assert D.verify(x, out, idx, w, toks)["max_err_over_tol"] <= 1.0
    # the oracle's output, rounded to bf16: only that rounding (at most
    # 2^-8 relative, bf16 having 8 significant bits: 0.39 of the tolerance)
    # and the cross-check's own fp32 sums separate it from the reference
    ref = oracle.moe_layer(xb, L, keep_intermediates=False)["out"]
    ob = torch.from_numpy(mi.bf16_bits_rne(ref.astype(np.float32)).view(np.int16)).cuda().view(
        torch.bfloat16)
    r = D.verify(x, ob, idx, w, toks)
    assert r["max_err_over_tol"] <= 0.4, r
    # one element of a sampled token off by 20% of the output's rms (|ref|
    # is within a few rms, so that is several tolerances)
    bad = out.clone()
    rms = float(np.sqrt(np.mean(ref[toks] ** 2)))
    assert abs(ref[7, 100]) < 4 * rms
    bad[7, 100] = bad[7, 100].float() + 0.2 * rms
    assert D.verify(x, bad, idx, w, toks)["max_err_over_tol"] > 3.0
    # ... but not when that token is not in the sample
    assert D.verify(x, bad, idx, w, [0, 3, 11])["max_err_over_tol"] <= 1.0


def test_verify_reports_an_invalid_token_as_infinite():
    torch = require_gpu()
    L = host_layer("tiny")
    D, xb, x, out, idx, w = _run(torch, L, 8, 23)
    r = D.verify(x, out, idx, w, [1, 8])  # token 8 does not exist
    assert r["max_err_over_tol"] == float("inf")
    assert D.verify(x, out, idx, w, [1, 7])["max_err_over_tol"] <= 1.0
