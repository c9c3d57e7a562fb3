"""GPU parity across the value ranges block-FP8 checkpoints and activations
take: the layer call and moe_expert_ffn_fp8 on both regimes (the streamed
GEMV and the tensor-core GEMM, each forced with MOE_FP8_EXPERT_PATH) against
the fp64 oracle, with block scales far below and above the workloads'
U(0.005, 0.02), scales whose magnitudes mix inside one row block, codes spread
over the whole E4M3 range, and activations scaled by powers of ten.  Values
within |gpu - ref| <= 1e-2 (|ref| + rms(ref)); routing bit-exact.

Also the status bits for inputs the fp16 intermediates cannot hold
(MOE_DEV_FP16_RANGE on the tensor-core GEMM) and for non-finite inputs
(MOE_DEV_NONFINITE on both regimes).
"""
import numpy as np
import pytest

import moe_inputs as mi
import oracle
from gpu_common import W_REL, assert_within_tol, bf16_bits, require_gpu

pytestmark = pytest.mark.gpu

PATHS = ("gemv", "gemm")

# (label, scale range, distribution)
SCALES = [
    ("u5e-5_2e-4", (5e-5, 2e-4), "uniform"),
    ("u2e-4_8e-4", (2e-4, 8e-4), "uniform"),
    ("u1e-3_4e-3", (1e-3, 4e-3), "uniform"),
    ("u1e-6_1e-4", (1e-6, 1e-4), "uniform"),
    ("mix5e-5_4e-3", (5e-5, 4e-3), "loguniform"),  # magnitudes mix inside a row block
    ("u3e1_3e2", (30.0, 300.0), "uniform"),
]


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


_cache = {}


def _base(name):
    if name not in _cache:
        _cache.clear()
        _cache[name] = mi.make_layer(name, seed=0)
    return _cache[name]


def _device(L):
    from block_fp8_expert_gb300.device import DeviceLayer
    return DeviceLayer.from_host(L)


def _x(xb):
    from block_fp8_expert_gb300.device import x_to_device
    return x_to_device(xb)


def _layer(torch, D, xb):
    import block_fp8_expert_gb300 as m
    T = xb.shape[0]
    idx = torch.empty((T, D.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, D.k), dtype=torch.float32, device="cuda")
    ws = D.workspace(T)
    out = D.forward(_x(xb), ws=ws, topk_idx=idx, topk_w=w)
    status = m.moe_read_device_status(ws)  # raises when a bit is set
    return oracle.bf16_to_f64(bf16_bits(out)), idx.cpu().numpy(), w.cpu().numpy(), status


def _ffn(torch, D, xb, ref):
    """moe_expert_ffn_fp8 on the oracle's own permutation; returns y_perm
    and the raw status bits (no exception)."""
    import block_fp8_expert_gb300 as m
    T = xb.shape[0]
    d = D.dims(T)
    ws = D.workspace(T)
    y = torch.full((T * D.k, D.H), float("nan"), dtype=torch.float32, device="cuda")
    m.moe_expert_ffn_fp8(_x(xb), torch.from_numpy(ref["expert_off"]).cuda(),
                         torch.from_numpy(ref["row_token"]).cuda(), D.routed.abi(), d, y, ws)
    torch.cuda.synchronize()
    bits = int(ws[:4].view(torch.int32).item())
    return y.cpu().numpy(), bits


def _check_layer(torch, D, L, xb, what, ref=None):
    got, idx, w, _ = _layer(torch, D, xb)
    if ref is None:
        ref = oracle.moe_layer(xb, L, keep_intermediates=False)
    assert np.array_equal(idx, ref["topk_idx"]), what
    assert_within_tol(w, ref["topk_w"], what + " topk_w", rel=W_REL)
    return assert_within_tol(got, ref["out"], what)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("label,rng,dist", SCALES)
def test_block_scale_range_qwen3_decode(torch, monkeypatch, path, label, rng, dist):
    """The Qwen3-MoE decode layer at 64 tokens (the tensor-core GEMM's regime
    by default) on both paths, block scales from each range."""
    monkeypatch.setenv("MOE_FP8_EXPERT_PATH", path)
    L = mi.with_scales(_base("qwen3moe_decode"), seed=11, scale_range=rng, scale_dist=dist)
    D = _device(L)
    xb, _ = mi.make_tokens(L, 64, seed=7)
    ref = oracle.moe_layer(xb, L)
    _check_layer(torch, D, L, xb, f"layer {label} {path}", ref)
    y, bits = _ffn(torch, D, xb, ref)
    assert bits == 0, f"status 0x{bits:x}"
    P = int(ref["expert_off"][-1])
    assert_within_tol(y[:P], ref["y_perm"][:P], f"y_perm {label} {path}")


@pytest.mark.parametrize("path", PATHS)
def test_checkpoint_like_codes(torch, monkeypatch, path):
    """Codes spread over the whole E4M3 range (an amax-scaled checkpoint:
    |code| up to 448) with scales ~1e-4, so the weights keep a realistic
    magnitude while codes and scales each sit far from 1."""
    monkeypatch.setenv("MOE_FP8_EXPERT_PATH", path)
    L = mi.make_layer("tiny", seed=3, code_gain=100.0, scale_range=(5e-5, 2e-4))
    assert int((L.gate.codes & 0x7F).max()) == 0x7E  # saturated codes present
    D = _device(L)
    xb, _ = mi.make_tokens(L, 300, seed=3)
    _check_layer(torch, D, L, xb, f"checkpoint-like codes {path}")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("gain", [1e-3, 1e3])
def test_activation_magnitude(torch, monkeypatch, path, gain):
    """x scaled by 1e-3 and 1e3 (then rounded to bf16): the expert FFN is
    compared on the oracle's permutation, so routing ties from the shrunken
    logit gaps cannot enter."""
    monkeypatch.setenv("MOE_FP8_EXPERT_PATH", path)
    L = _base("tiny")
    D = _device(L)
    xb0, _ = mi.make_tokens(L, 300, seed=5)
    xb = mi.bf16_bits_rne(oracle.bf16_to_f64(xb0).astype(np.float32) * np.float32(gain))
    ref = oracle.moe_layer(xb, L)
    y, bits = _ffn(torch, D, xb, ref)
    assert bits == 0, f"status 0x{bits:x}"
    P = int(ref["expert_off"][-1])
    assert_within_tol(y[:P], ref["y_perm"][:P], f"y_perm x*{gain:g} {path}")


@pytest.mark.parametrize("path", PATHS)
def test_shared_expert_small_scales(torch, monkeypatch, path):
    """A layer with a shared expert (the 512-expert family's structure at a
    smaller size), scales U(5e-5, 2e-4), 64 tokens: routed and shared experts
    both on the forced path."""
    monkeypatch.setenv("MOE_FP8_EXPERT_PATH", path)
    w = mi.Workload("shared_mid", H=512, I=256, E=32, k=4, I_shared=256)
    L = mi.make_layer(w, seed=8, scale_range=(5e-5, 2e-4))
    D = _device(L)
    xb, _ = mi.make_tokens(L, 64, seed=8)
    _check_layer(torch, D, L, xb, f"shared expert small scales {path}")


def test_large_scales_are_exact(torch, monkeypatch):
    """Gate/up scales of 300 (SwiGLU outputs around 1e7, far beyond fp16's
    range) give correct values on both paths: nothing is flagged."""
    L = mi.make_layer("tiny", seed=6)
    L.gate.scales[:] = 300.0
    L.up.scales[:] = 300.0
    D = _device(L)
    xb, _ = mi.make_tokens(L, 100, seed=6)
    for path in PATHS:
        monkeypatch.setenv("MOE_FP8_EXPERT_PATH", path)
        _check_layer(torch, D, L, xb, f"scales 300 {path}")


def test_tiny_codes_flagged_on_gemm_exact_on_gemv(torch, monkeypatch):
    """Codes at the smallest E4M3 magnitude (2^-9) everywhere: the weights
    are 2^-9 of what their block scales suggest, so the tensor-core GEMM's
    fixed hid normalisation would leave every hid value in fp16's subnormal
    range.  It must raise MOE_DEV_FP16_RANGE; the streamed GEMV, whose hid
    exponent follows the values, stays exact."""
    import block_fp8_expert_gb300 as m
    L = mi.make_layer("tiny", seed=9)
    rng = np.random.default_rng(9)
    for mat in (L.gate, L.up, L.down):
        mat.codes[:] = np.where(rng.random(mat.codes.shape) < 0.5, 0x01, 0x81).astype(np.uint8)
    D = _device(L)
    xb, _ = mi.make_tokens(L, 300, seed=9)
    ref = oracle.moe_layer(xb, L)
    P = int(ref["expert_off"][-1])
    monkeypatch.setenv("MOE_FP8_EXPERT_PATH", "gemm")
    _, bits = _ffn(torch, D, xb, ref)
    assert bits & m._lib.MOE_DEV_FP16_RANGE, f"status 0x{bits:x}"
    monkeypatch.setenv("MOE_FP8_EXPERT_PATH", "gemv")
    y, bits = _ffn(torch, D, xb, ref)
    assert bits == 0, f"status 0x{bits:x}"
    assert_within_tol(y[:P], ref["y_perm"][:P], "tiny codes gemv")


def test_saturated_codes_and_positive_x_flagged_on_gemm_exact_on_gemv(torch, monkeypatch):
    """Every code +448 and every activation positive: the gate and up sums
    add coherently, and the GEMM's hid exceeds fp16's range.  It must raise
    MOE_DEV_FP16_RANGE; the GEMV stays exact."""
    import block_fp8_expert_gb300 as m
    L = mi.make_layer("tiny", seed=10)
    for mat in (L.gate, L.up, L.down):
        mat.codes[:] = 0x7E
    D = _device(L)
    xb0, _ = mi.make_tokens(L, 64, seed=10)
    xb = xb0 & np.uint16(0x7FFF)  # |x|
    ref = oracle.moe_layer(xb, L)
    P = int(ref["expert_off"][-1])
    monkeypatch.setenv("MOE_FP8_EXPERT_PATH", "gemm")
    _, bits = _ffn(torch, D, xb, ref)
    assert bits & m._lib.MOE_DEV_FP16_RANGE, f"status 0x{bits:x}"
    monkeypatch.setenv("MOE_FP8_EXPERT_PATH", "gemv")
    y, bits = _ffn(torch, D, xb, ref)
    assert bits == 0, f"status 0x{bits:x}"
    assert_within_tol(y[:P], ref["y_perm"][:P], "saturated codes gemv")


@pytest.mark.parametrize("path", PATHS)
def test_nonfinite_inputs_flagged(torch, monkeypatch, path):
    """An infinite block scale, or a NaN activation, raises
    MOE_DEV_NONFINITE; the next clean call clears it."""
    import block_fp8_expert_gb300 as m
    monkeypatch.setenv("MOE_FP8_EXPERT_PATH", path)
    L = _base("tiny")
    xb, _ = mi.make_tokens(L, 300, seed=12)
    ref = oracle.moe_layer(xb, L)
    D = _device(L)
    bad_scale = D.routed.up_scales.clone()
    bad_scale.view(-1)[5] = float("inf")
    good = D.routed.up_scales
    D.routed.up_scales = bad_scale
    _, bits = _ffn(torch, D, xb, ref)
    assert bits & m._lib.MOE_DEV_NONFINITE, f"status 0x{bits:x}"
    D.routed.up_scales = good
    xn = xb.copy()
    xn[int(ref["row_token"][0]), 3] = 0x7FC0  # bf16 NaN in a routed token
    _, bits = _ffn(torch, D, xn, ref)
    assert bits & m._lib.MOE_DEV_NONFINITE, f"status 0x{bits:x}"
    _, bits = _ffn(torch, D, xb, ref)
    assert bits == 0, f"status 0x{bits:x}"


@pytest.mark.parametrize("path,T", [("auto", 8), ("gemv", 64), ("gemm", 64), ("auto", 300)])
def test_gated_shared_expert(torch, monkeypatch, path, T):
    """moe_layer_forward_gated: the shared expert's output scaled by
    sigmoid(x . g) per token.  T = 8 runs the shared expert as one more
    expert of the streamed GEMV launches with the combine folded into the
    down kernel; T = 64 on each forced regime; T = 300 the default regime
    (tensor-core GEMM, token-major gather writing the shared rows)."""
    if path != "auto":
        monkeypatch.setenv("MOE_FP8_EXPERT_PATH", path)
    w = mi.Workload("shared_mid", H=512, I=256, E=32, k=4, I_shared=256)
    L = mi.make_layer(w, seed=15, shared_gated=True)
    D = _device(L)
    assert D.shared_gate_w is not None
    xb, _ = mi.make_tokens(L, T, seed=15)
    ref = oracle.moe_layer(xb, L, keep_intermediates=False)
    fac = oracle.shared_gate_factor(oracle.bf16_to_f64(xb), L)
    assert fac.max() - fac.min() > 0.05  # the gate really varies over the tokens
    _check_layer(torch, D, L, xb, f"gated shared expert {path} T={T}", ref)
