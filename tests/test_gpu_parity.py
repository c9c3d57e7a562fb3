"""GPU parity: every C-ABI call against the fp64 oracle on the same seeded
inputs.  Routing and permutation bit-exact; values within
|gpu - ref| <= 1e-2 (|ref| + rms(ref)) per element."""
import numpy as np
import pytest

import moe_inputs as mi
import oracle
from gpu_common import W_REL, assert_within_tol, bf16_bits, host_layer, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


_dev_layers = {}


def dev_layer(name, seed=0):
    from block_fp8_expert_gb300.device import DeviceLayer
    key = (name, seed)
    if key not in _dev_layers:
        _dev_layers.clear()  # keep at most one large layer resident
        _dev_layers[key] = DeviceLayer.from_host(host_layer(name, seed))
    return _dev_layers[key]


def _x(torch, x_bits):
    from block_fp8_expert_gb300.device import x_to_device
    return x_to_device(x_bits)


def _forward(torch, D, xd):
    T = xd.shape[0]
    idx = torch.empty((T, D.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, D.k), dtype=torch.float32, device="cuda")
    ws = D.workspace(T)
    out = D.forward(xd, ws=ws, topk_idx=idx, topk_w=w)
    torch.cuda.synchronize()
    # word 0: status bits; words 1-5: where a bounded wait ran out, if one did
    words = ws[:32].view(torch.int32).cpu().numpy()
    assert words[0] == 0, f"device status {words[:6].tolist()}"
    return out, idx, w


# ---------------------------------------------------------------------------
# single ABI calls
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,T", [("tiny", 8), ("tiny", 37), ("qwen3moe_decode", 64),
                                    ("large_sparse", 256), ("skewed", 256)])
def test_route(torch, name, T):
    import block_fp8_expert_gb300 as m
    L = host_layer(name)
    D = dev_layer(name)
    xb, _ = mi.make_tokens(L, T, seed=1)
    xd = _x(torch, xb)
    d = D.dims(T)
    ws = D.workspace(T)
    idx = torch.empty((T, L.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, L.k), dtype=torch.float32, device="cuda")
    m.moe_route(xd, D.Wr, D.bias, d, idx, w, ws)
    torch.cuda.synchronize()
    x = oracle.bf16_to_f64(xb)
    ridx, rw = oracle.topk_renorm(oracle.softmax(oracle.router_logits(x, L.Wr, L.bias)), L.k)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert_within_tol(w.cpu().numpy(), rw, "topk_w", rel=W_REL)


@pytest.mark.parametrize("T,E,k", [(1, 16, 2), (8, 16, 2), (13, 128, 8), (300, 512, 10),
                                   (4096, 128, 8), (333, 7, 3), (16384, 128, 8)])
def test_permute_bit_exact(torch, T, E, k):
    import block_fp8_expert_gb300 as m
    rng = np.random.default_rng(T + E)
    if T >= 4096:  # skewed expert load
        p = 1.0 / np.arange(1, E + 1) ** 1.2
        idx = np.stack([rng.choice(E, k, replace=False, p=p / p.sum()) for _ in range(T)])
    else:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    idx = idx.astype(np.int32)
    d = m.dims(T, 256, 128, E, k)
    ws = torch.empty(m.workspace_bytes(d), dtype=torch.uint8, device="cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    rt = torch.empty(T * k, dtype=torch.int32, device="cuda")
    tsr = torch.empty(T * k, dtype=torch.int32, device="cuda")
    m.moe_permute(torch.from_numpy(idx).cuda(), d, off, rt, tsr, ws)
    assert m.moe_read_device_status(ws) == 0
    r_off, r_rt, r_tsr = oracle.permute(idx, E)
    assert np.array_equal(off.cpu().numpy(), r_off)
    assert np.array_equal(rt.cpu().numpy(), r_rt)
    assert np.array_equal(tsr.cpu().numpy(), r_tsr)


def test_permute_empty(torch):
    import block_fp8_expert_gb300 as m
    d = m.dims(0, 256, 128, 16, 2)
    ws = torch.empty(m.workspace_bytes(d), dtype=torch.uint8, device="cuda")
    off = torch.full((17,), 7, dtype=torch.int32, device="cuda")
    dummy = torch.empty(4, dtype=torch.int32, device="cuda")
    m.moe_permute(dummy, d, off, dummy, dummy, ws)
    torch.cuda.synchronize()
    assert off.cpu().numpy().tolist() == [0] * 17


def test_permute_flags_bad_expert_index(torch):
    import block_fp8_expert_gb300 as m
    T, E, k = 4, 16, 2
    idx = np.array([[0, 1], [2, 16], [-1, 3], [4, 5]], dtype=np.int32)
    d = m.dims(T, 256, 128, E, k)
    ws = torch.empty(m.workspace_bytes(d), dtype=torch.uint8, device="cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    rt = torch.empty(T * k, dtype=torch.int32, device="cuda")
    tsr = torch.empty(T * k, dtype=torch.int32, device="cuda")
    m.moe_permute(torch.from_numpy(idx).cuda(), d, off, rt, tsr, ws)
    with pytest.raises(m.MoeError) as ei:
        m.moe_read_device_status(ws)
    assert "0x1" in str(ei.value)
    t = tsr.cpu().numpy()
    assert t[3] == -1 and t[4] == -1
    assert off.cpu().numpy()[-1] == 6
    # a clean call afterwards clears the word
    good = torch.from_numpy(np.array([[0, 1], [2, 3], [4, 5], [6, 7]], np.int32)).cuda()
    m.moe_permute(good, d, off, rt, tsr, ws)
    assert m.moe_read_device_status(ws) == 0


@pytest.mark.parametrize("name,T", [("tiny", 8), ("tiny", 29), ("qwen3moe_decode", 8),
                                    ("qwen3moe_decode", 64)])
def test_expert_ffn(torch, name, T):
    import block_fp8_expert_gb300 as m
    L = host_layer(name)
    D = dev_layer(name)
    xb, _ = mi.make_tokens(L, T, seed=2)
    ref = oracle.moe_layer(xb, L)
    d = D.dims(T)
    ws = D.workspace(T)
    y = torch.full((T * L.k, L.H), float("nan"), dtype=torch.float32, device="cuda")
    m.moe_expert_ffn_fp8(_x(torch, xb), torch.from_numpy(ref["expert_off"]).cuda(),
                         torch.from_numpy(ref["row_token"]).cuda(), D.routed.abi(), d, y, ws)
    torch.cuda.synchronize()
    assert_within_tol(y.cpu().numpy(), ref["y_perm"], "y_perm")


def test_combine(torch):
    import block_fp8_expert_gb300 as m
    rng = np.random.default_rng(9)
    T, H, k = 37, 256, 3
    y = rng.standard_normal((T * k, H)).astype(np.float32)
    tsr = rng.permutation(T * k).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    sh = rng.standard_normal((T, H)).astype(np.float32)
    d = m.dims(T, H, 128, 8, k)
    for shared in (None, sh):
        out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        m.moe_combine(torch.from_numpy(y).cuda(), torch.from_numpy(tsr).cuda(),
                      torch.from_numpy(w).cuda(),
                      None if shared is None else torch.from_numpy(shared).cuda(), d, out)
        torch.cuda.synchronize()
        ref = oracle.combine(y.astype(np.float64), tsr, w.astype(np.float64),
                             None if shared is None else shared.astype(np.float64))
        got = oracle.bf16_to_f64(bf16_bits(out))
        # one bf16 rounding of the fp32 sum
        assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)


# ---------------------------------------------------------------------------
# the whole layer
# ---------------------------------------------------------------------------

FULL = [("tiny", 8), ("tiny", 1), ("tiny", 3), ("tiny", 13), ("tiny", 100),
        ("qwen3moe_decode", 1), ("qwen3moe_decode", 8), ("qwen3moe_decode", 64),
        ("large_sparse", 1), ("large_sparse", 256),
        ("skewed", 1), ("skewed", 16), ("skewed", 256)]


@pytest.mark.parametrize("name,T", FULL)
def test_layer_forward_full(torch, name, T):
    L = host_layer(name)
    D = dev_layer(name)
    xb, _ = mi.make_tokens(L, T, seed=0)
    out, idx, w = _forward(torch, D, _x(torch, xb))
    ref = oracle.moe_layer(xb, L, keep_intermediates=False)
    assert np.array_equal(idx.cpu().numpy(), ref["topk_idx"])
    assert_within_tol(w.cpu().numpy(), ref["topk_w"], "topk_w", rel=W_REL)
    assert_within_tol(oracle.bf16_to_f64(bf16_bits(out)), ref["out"], f"out {name} T={T}")


# Shapes the regime rule sends to the tensor-core GEMM, forced through the
# streamed GEMV (MOE_FP8_EXPERT_PATH=gemv): the GEMV's 16-token variant and its
# hot-expert row loops stay covered.
GEMV_FORCED = [("tiny", 100), ("qwen3moe_decode", 64), ("skewed", 256), ("large_sparse", 256)]


@pytest.mark.parametrize("name,T", GEMV_FORCED)
def test_layer_forward_full_through_gemv(torch, monkeypatch, name, T):
    monkeypatch.setenv("MOE_FP8_EXPERT_PATH", "gemv")
    L = host_layer(name)
    D = dev_layer(name)
    xb, _ = mi.make_tokens(L, T, seed=0)
    out, idx, w = _forward(torch, D, _x(torch, xb))
    ref = oracle.moe_layer(xb, L, keep_intermediates=False)
    assert np.array_equal(idx.cpu().numpy(), ref["topk_idx"])
    assert_within_tol(w.cpu().numpy(), ref["topk_w"], "topk_w", rel=W_REL)
    assert_within_tol(oracle.bf16_to_f64(bf16_bits(out)), ref["out"], f"out {name} T={T} gemv")


# Full-size batches of the tensor-core GEMM regime, every output element
# compared (the fp64 oracle takes a few seconds per call on the host).
LARGE = [("qwen3moe_prefill", 4096), ("skewed", 2048), ("skewed", 16384)]


@pytest.mark.parametrize("name,T", LARGE)
def test_layer_forward_large(torch, name, T):
    L = host_layer(name if name != "qwen3moe_prefill" else "qwen3moe_decode")
    D = dev_layer(name if name != "qwen3moe_prefill" else "qwen3moe_decode")
    xb, _ = mi.make_tokens(L, T, seed=0)
    out, idx, w = _forward(torch, D, _x(torch, xb))
    ref = oracle.moe_layer(xb, L, keep_intermediates=False)
    assert np.array_equal(idx.cpu().numpy(), ref["topk_idx"])
    assert_within_tol(w.cpu().numpy(), ref["topk_w"], "topk_w", rel=W_REL)
    assert_within_tol(oracle.bf16_to_f64(bf16_bits(out)), ref["out"], f"out {name} T={T}")


def test_layer_forward_is_deterministic(torch):
    L = host_layer("qwen3moe_decode")
    D = dev_layer("qwen3moe_decode")
    xb, _ = mi.make_tokens(L, 64, seed=5)
    xd = _x(torch, xb)
    a = _forward(torch, D, xd)
    b = _forward(torch, D, xd)
    for u, v in zip(a, b):
        assert torch.equal(u.view(torch.uint8) if u.dtype == torch.bfloat16 else u,
                           v.view(torch.uint8) if v.dtype == torch.bfloat16 else v)


@pytest.mark.parametrize("name,T", [("tiny", 8), ("qwen3moe_decode", 1), ("qwen3moe_decode", 8),
                                    ("qwen3moe_decode", 64), ("large_sparse", 1)])
def test_layer_forward_dirty_workspace(torch, name, T):
    """Every counter a call relies on (the fused combine's tickets, the GEMM's
    completion counters, the status words) is cleared by the call itself: a
    workspace full of stale bytes gives the same output, twice in a row."""
    L = host_layer(name)
    D = dev_layer(name)
    xb, _ = mi.make_tokens(L, T, seed=3)
    xd = _x(torch, xb)
    ws = D.workspace(T)
    outs = []
    for fill in (0x5A, 0xFF):
        ws.fill_(fill)
        outs.append(D.forward(xd, ws=ws))
        torch.cuda.synchronize()
        assert ws[:4].view(torch.int32).item() == 0
    assert torch.equal(outs[0].view(torch.uint8), outs[1].view(torch.uint8))
    ref = oracle.moe_layer(xb, L, keep_intermediates=False)
    assert_within_tol(oracle.bf16_to_f64(bf16_bits(outs[0])), ref["out"], f"out {name} T={T}")


def test_layer_forward_empty_batch(torch):
    D = dev_layer("tiny")
    x = torch.empty((0, D.H), dtype=torch.bfloat16, device="cuda")
    out = D.forward(x)
    torch.cuda.synchronize()
    assert out.shape == (0, D.H)


def test_shared_expert_alone(torch):
    """Routed experts zeroed: the layer is the shared expert."""
    from block_fp8_expert_gb300.device import DeviceLayer
    w = mi.Workload("shared_small", H=256, I=128, E=8, k=2, I_shared=192)
    L = mi.make_layer(w, seed=4)
    for mat in (L.gate, L.up, L.down):
        mat.codes[:] = 0
    D = DeviceLayer.from_host(L)
    xb, _ = mi.make_tokens(L, 11, seed=4)
    out, _, _ = _forward(torch, D, _x(torch, xb))
    ref = oracle.moe_layer(xb, L)["out"]
    assert np.abs(ref).max() > 0
    assert_within_tol(oracle.bf16_to_f64(bf16_bits(out)), ref, "shared only")


def test_identity_expert_closed_form(torch):
    """H = I = 128, one expert wins, Wg = Wu = Wd = c*Id: out = c^3 x^2 sigma(c x)."""
    from block_fp8_expert_gb300.device import DeviceLayer
    H = 128
    c = 0.5
    eye = np.zeros((2, H, H), np.uint8)
    eye[0, np.arange(H), np.arange(H)] = 0x38
    sc = np.full((2, 1, 1), c, np.float32)
    mat = mi.Fp8Mat(eye, sc)
    Wr = np.zeros((2, H), np.float32)
    Wr[0, 0] = 1.0
    L = mi.LayerWeights(H=H, I=H, E=2, k=1, I_shared=0, Wr=Wr, bias=None, gate=mat, up=mat,
                        down=mat)
    D = DeviceLayer.from_host(L)
    xf = np.random.default_rng(0).standard_normal((5, H)).astype(np.float32)
    xf[:, 0] = np.abs(xf[:, 0]) + 0.5
    xb = mi.bf16_bits_rne(xf)
    out, idx, w = _forward(torch, D, _x(torch, xb))
    x = oracle.bf16_to_f64(xb)
    expect = c ** 3 * x ** 2 / (1 + np.exp(-c * x))
    assert idx.cpu().numpy().ravel().tolist() == [0] * 5
    assert_within_tol(oracle.bf16_to_f64(bf16_bits(out)), expect, "identity expert")


# Degenerate routing: a single expert (every token's one slot, weight 1),
# every expert selected (k = E: the weights are the full softmax) and top-1,
# on both expert paths, with a ragged token count.
DEGENERATE = [(1, 1), (8, 8), (32, 1)]


@pytest.mark.parametrize("path", ["gemv", "gemm"])
@pytest.mark.parametrize("E,k", DEGENERATE)
@pytest.mark.parametrize("T", [1, 37, 200])
def test_layer_forward_degenerate_routing(torch, monkeypatch, path, E, k, T):
    from block_fp8_expert_gb300.device import DeviceLayer
    monkeypatch.setenv("MOE_FP8_EXPERT_PATH", path)
    w = mi.Workload(f"degenerate_E{E}_k{k}", H=256, I=128, E=E, k=k)
    L = mi.make_layer(w, seed=11)
    D = DeviceLayer.from_host(L)
    xb, _ = mi.make_tokens(L, T, seed=11)
    out, idx, wts = _forward(torch, D, _x(torch, xb))
    ref = oracle.moe_layer(xb, L, keep_intermediates=False)
    assert np.array_equal(idx.cpu().numpy(), ref["topk_idx"])
    if k == E:
        # every expert once per token
        assert np.array_equal(np.sort(idx.cpu().numpy(), axis=1),
                              np.tile(np.arange(E), (T, 1)))
    if k == 1:
        assert np.all(wts.cpu().numpy() == 1.0)
    assert_within_tol(wts.cpu().numpy(), ref["topk_w"], "topk_w", rel=W_REL)
    assert_within_tol(oracle.bf16_to_f64(bf16_bits(out)), ref["out"],
                      f"out E={E} k={k} T={T} {path}")


# Token counts on both sides of every host-side switch of the layer call:
# T*k = 64 (tiny one-CTA permutation) / 72, 15 / 16 (top-k split into its own
# launch), 127 / 128 (mma.sync router / tensor-core router), T*k = 4096 /
# 4104 (one-CTA permutation / three permutation kernels).
@pytest.mark.parametrize("T", [8, 9, 15, 16, 127, 128, 512, 513])
def test_layer_forward_switch_boundaries(torch, T):
    L = host_layer("qwen3moe_decode")
    D = dev_layer("qwen3moe_decode")
    xb, _ = mi.make_tokens(L, T, seed=12)
    out, idx, w = _forward(torch, D, _x(torch, xb))
    ref = oracle.moe_layer(xb, L, keep_intermediates=False)
    assert np.array_equal(idx.cpu().numpy(), ref["topk_idx"])
    assert_within_tol(w.cpu().numpy(), ref["topk_w"], "topk_w", rel=W_REL)
    assert_within_tol(oracle.bf16_to_f64(bf16_bits(out)), ref["out"], f"out T={T}")
