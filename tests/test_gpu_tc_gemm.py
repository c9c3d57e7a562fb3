"""GPU parity of the tensor-core (tcgen05) grouped GEMM path.  The path is
forced on small shapes with MOE_FP8_EXPERT_PATH=gemm and taken naturally at
prefill sizes; results are compared with the fp64 oracle under the same rule
as every layer test: routing bit-exact, |gpu - ref| <= 1e-2 (|ref| + rms)."""
import numpy as np
import pytest

import moe_inputs as mi
import oracle
from gpu_common import assert_within_tol, bf16_bits, host_layer, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


@pytest.fixture
def force_gemm(monkeypatch):
    monkeypatch.setenv("MOE_FP8_EXPERT_PATH", "gemm")


def _run(torch, L, T, seed=0):
    from block_fp8_expert_gb300.device import DeviceLayer, x_to_device
    D = DeviceLayer.from_host(L)
    xb, _ = mi.make_tokens(L, T, seed=seed)
    idx = torch.empty((T, L.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, L.k), dtype=torch.float32, device="cuda")
    ws = D.workspace(T)
    ws.zero_()
    out = D.forward(x_to_device(xb), ws=ws, topk_idx=idx, topk_w=w)
    torch.cuda.synchronize()
    _assert_clean_status(torch, ws)
    return xb, out, idx, w


def _assert_clean_status(torch, ws):
    words = ws[:32].view(torch.int32).cpu().numpy()
    # word 0: status bits; words 1-5: where a bounded wait ran out, if one did
    assert words[0] == 0, f"device status {words[:6].tolist()}"



@pytest.mark.parametrize("T", [8, 100, 300])
def test_tiny_layer_through_gemm(torch, force_gemm, T):
    L = host_layer("tiny")
    xb, out, idx, w = _run(torch, L, T)
    ref = oracle.moe_layer(xb, L, keep_intermediates=False)
    assert np.array_equal(idx.cpu().numpy(), ref["topk_idx"])
    assert_within_tol(oracle.bf16_to_f64(bf16_bits(out)), ref["out"], f"tiny T={T} gemm")


def test_expert_ffn_through_gemm_matches_oracle_y(torch, force_gemm):
    """moe_expert_ffn_fp8 alone: y for every permuted row, 3 m-tiles + a
    ragged tail per expert."""
    import block_fp8_expert_gb300 as m
    from block_fp8_expert_gb300.device import DeviceLayer, x_to_device
    w = mi.Workload("gemm_probe", H=512, I=256, E=4, k=2)
    L = mi.make_layer(w, seed=3)
    T = 700
    xb, _ = mi.make_tokens(L, T, seed=3)
    ref = oracle.moe_layer(xb, L)
    D = DeviceLayer.from_host(L)
    d = D.dims(T)
    ws = D.workspace(T)
    ws.zero_()
    y = torch.full((T * L.k, L.H), float("nan"), dtype=torch.float32, device="cuda")
    m.moe_expert_ffn_fp8(x_to_device(xb), torch.from_numpy(ref["expert_off"]).cuda(),
                         torch.from_numpy(ref["row_token"]).cuda(), D.routed.abi(), d, y, ws)
    torch.cuda.synchronize()
    _assert_clean_status(torch, ws)
    assert_within_tol(y.cpu().numpy(), ref["y_perm"], "y_perm (gemm)")


def test_identity_experts_through_gemm(torch, force_gemm):
    """H = 256, I = 128, every expert the identity-like matrix c*[I | 0]:
    closed form out = c^3 x^2 sigma(c x) on the first 128 features."""
    H, I, E = 256, 128, 2
    c = 0.5
    g = np.zeros((E, I, H), np.uint8)
    g[:, np.arange(I), np.arange(I)] = 0x38
    d = np.zeros((E, H, I), np.uint8)
    d[:, np.arange(I), np.arange(I)] = 0x38
    gs = np.full((E, 1, 2), c, np.float32)
    ds = np.full((E, 2, 1), c, np.float32)
    Wr = np.zeros((E, H), np.float32)
    Wr[0, 0] = 1.0
    L = mi.LayerWeights(H=H, I=I, E=E, k=1, I_shared=0, Wr=Wr, bias=None,
                        gate=mi.Fp8Mat(g, gs), up=mi.Fp8Mat(g.copy(), gs.copy()),
                        down=mi.Fp8Mat(d, ds))
    xf = np.random.default_rng(1).standard_normal((200, H)).astype(np.float32)
    xf[:, 0] = np.abs(xf[:, 0]) + 0.5
    xb = mi.bf16_bits_rne(xf)
    from block_fp8_expert_gb300.device import DeviceLayer, x_to_device
    D = DeviceLayer.from_host(L)
    out = D.forward(x_to_device(xb))
    torch.cuda.synchronize()
    x = oracle.bf16_to_f64(xb)
    expect = np.zeros_like(x)
    expect[:, :I] = c ** 3 * x[:, :I] ** 2 / (1 + np.exp(-c * x[:, :I]))
    assert_within_tol(oracle.bf16_to_f64(bf16_bits(out)), expect, "identity via gemm")


@pytest.mark.parametrize("name,T", [("qwen3moe_decode", 64), ("large_sparse", 256)])
def test_decode_shapes_through_gemm(torch, force_gemm, name, T):
    L = host_layer(name)
    xb, out, idx, w = _run(torch, L, T)
    ref = oracle.moe_layer(xb, L, keep_intermediates=False)
    assert np.array_equal(idx.cpu().numpy(), ref["topk_idx"])
    assert_within_tol(oracle.bf16_to_f64(bf16_bits(out)), ref["out"], f"{name} T={T} gemm")


def test_largest_gemm_shape(torch):
    """H = I = 4096, the largest shape the tensor-core GEMM takes (32 block
    scales of K per weight row block); 2 experts, top-1, 100 tokens = 50 rows
    per expert on average, so the GEMM is the natural regime (checked), each
    expert's only token tile ragged."""
    import block_fp8_expert_gb300 as m
    w = mi.Workload("gemm_max", H=4096, I=4096, E=2, k=1)
    L = mi.make_layer(w, seed=7)
    T = 100
    assert m.expert_uses_gemm(m.dims(T, w.H, w.I, w.E, w.k))
    xb, out, idx, wts = _run(torch, L, T, seed=7)
    ref = oracle.moe_layer(xb, L, keep_intermediates=False)
    assert np.array_equal(idx.cpu().numpy(), ref["topk_idx"])
    assert_within_tol(oracle.bf16_to_f64(bf16_bits(out)), ref["out"], "H = I = 4096 gemm")


@pytest.mark.parametrize("launches", ["1", "2"])
@pytest.mark.parametrize("name,T", [("qwen3moe_decode", 64), ("tiny", 300), ("skewed", 256)])
def test_one_or_two_launches_match_oracle(torch, monkeypatch, launches, name, T):
    """The tile list run by one launch (gate/up then down tiles in every CTA's
    sequence) or by two (gate/up, then down): same oracle, either form forced
    with MOE_FP8_GEMM_LAUNCHES, so both are covered at every size."""
    monkeypatch.setenv("MOE_FP8_EXPERT_PATH", "gemm")
    monkeypatch.setenv("MOE_FP8_GEMM_LAUNCHES", launches)
    L = host_layer(name)
    xb, out, idx, w = _run(torch, L, T)
    ref = oracle.moe_layer(xb, L, keep_intermediates=False)
    assert np.array_equal(idx.cpu().numpy(), ref["topk_idx"])
    assert_within_tol(oracle.bf16_to_f64(bf16_bits(out)), ref["out"],
                      f"{name} T={T}, {launches} launch(es)")


@pytest.mark.parametrize("name,T", [("qwen3moe_decode", 64), ("qwen3moe_decode", 1),
                                    ("tiny", 300), ("skewed", 256)])
def test_one_and_two_launches_bit_identical(torch, monkeypatch, name, T):
    """One launch (gate/up and down tiles in every CTA's sequence) and two
    launches run each tile with the same arithmetic, so the layer outputs
    agree bit for bit on the same inputs."""
    monkeypatch.setenv("MOE_FP8_EXPERT_PATH", "gemm")
    L = host_layer(name)
    outs = []
    for launches in ("1", "2"):
        monkeypatch.setenv("MOE_FP8_GEMM_LAUNCHES", launches)
        xb, out, idx, w = _run(torch, L, T, seed=3)
        outs.append(bf16_bits(out))
    assert np.array_equal(outs[0], outs[1]), f"{name} T={T}: one vs two launches"
