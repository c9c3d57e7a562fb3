"""Pins for the oracle's expert FFN, combine and whole layer: closed forms
with identity / one-hot experts, a pure-Python scalar brute force of the tiny
workload, the shared-expert reductions, the sampled path, and the gap guard of
the generated inputs."""
import math

import numpy as np
import pytest
from scipy.special import expit

import oracle
import moe_inputs as mi


def test_silu_matches_library():
    z = np.linspace(-30, 30, 1001)
    assert np.allclose(oracle.silu(z), z * expit(z), rtol=1e-14, atol=1e-300)


def _identity_mat(n, c):
    codes = np.zeros((1, n, n), np.uint8)
    codes[0, np.arange(n), np.arange(n)] = 0x38  # 1.0
    scales = np.full((1, -(-n // 128), -(-n // 128)), c, np.float32)
    return mi.Fp8Mat(codes, scales)


def _onehot_router(E, H, winner):
    # x . Wr[winner] large and positive for any x with a positive first entry
    Wr = np.zeros((E, H), np.float32)
    Wr[winner, 0] = 1.0
    return Wr


def test_ffn_closed_form_identity_experts():
    """H = I = 128, E = 2, k = 1, Wg = Wu = Wd = c*Id: with one token routed to
    expert 0 (weight 1 after renormalisation), out = c^3 x^2 sigma(c x)."""
    H = I = 128
    c = 0.5  # exactly representable in fp32
    g = _identity_mat(H, c)
    zero = mi.Fp8Mat(np.zeros((1, H, H), np.uint8), np.full((1, 1, 1), c, np.float32))
    gate = mi.Fp8Mat(np.concatenate([g.codes, zero.codes]), np.concatenate([g.scales, g.scales]))
    layer = mi.LayerWeights(H=H, I=I, E=2, k=1, I_shared=0,
                            Wr=_onehot_router(2, H, 0), bias=None,
                            gate=gate, up=gate, down=gate)
    rng = np.random.default_rng(0)
    xf = rng.standard_normal((3, H)).astype(np.float32)
    xf[:, 0] = np.abs(xf[:, 0]) + 0.5
    xb = mi.bf16_bits_rne(xf)
    res = oracle.moe_layer(xb, layer)
    assert res["topk_idx"].ravel().tolist() == [0, 0, 0]
    assert np.array_equal(res["topk_w"], np.ones((3, 1)))
    x = oracle.bf16_to_f64(xb)
    expect = c ** 3 * x ** 2 * expit(c * x)
    assert np.allclose(res["out"], expect, rtol=1e-14, atol=1e-300)


def test_down_projection_layout_one_hot():
    """Wd a row permutation (Wd[h, pi(h)] = 1): y[h] = hid[pi(h)].  A
    transposed down matrix would give hid[pi^-1(h)] instead."""
    H, I = 256, 128
    rng = np.random.default_rng(2)
    pi = rng.integers(0, I, H)  # Wd[h, pi[h]] = 1, not a transpose-symmetric map
    dcodes = np.zeros((1, H, I), np.uint8)
    dcodes[0, np.arange(H), pi] = 0x38
    down = mi.Fp8Mat(dcodes, np.ones((1, 2, 1), np.float32))
    gc = rng.integers(0, 0x7E, (1, I, H)).astype(np.uint8)
    gate = mi.Fp8Mat(gc, np.full((1, 1, 2), 0.01, np.float32))
    uc = rng.integers(0, 0x7E, (1, I, H)).astype(np.uint8)
    up = mi.Fp8Mat(uc, np.full((1, 1, 2), 0.02, np.float32))
    x = rng.standard_normal((4, H))
    Wg = oracle.dequantize(gc[0], gate.scales[0])
    Wu = oracle.dequantize(uc[0], up.scales[0])
    Wd = oracle.dequantize(dcodes[0], down.scales[0])
    y = oracle.expert_ffn(x, Wg, Wu, Wd)
    hid = oracle.silu(x @ Wg.T) * (x @ Wu.T)
    assert np.allclose(y, hid[:, pi], rtol=1e-14, atol=0)


def _scalar_layer(x_bits, L):
    """The layer for every token with pure-Python scalar loops and math.fsum:
    no NumPy arithmetic, no BLAS."""
    T, H = x_bits.shape
    E, k, I = L.E, L.k, L.I

    def bf(b):
        return oracle.bf16_to_f64(np.array([b]))[0]

    def dec(code):
        s, e, m = code >> 7, (code >> 3) & 15, code & 7
        mag = (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        return -mag if s else mag

    def w(mat, e, r, c):
        return dec(int(mat.codes[e, r, c])) * float(mat.scales[e, r // 128, c // 128])

    outs = []
    for t in range(T):
        x = [bf(int(b)) for b in x_bits[t]]
        l = [math.fsum(x[h] * float(L.Wr[e, h]) for h in range(H))
             + (0.0 if L.bias is None else float(L.bias[e])) for e in range(E)]
        m = max(l)
        z = [math.exp(v - m) for v in l]
        Z = math.fsum(z)
        p = [v / Z for v in z]
        sel = sorted(range(E), key=lambda e: (-p[e], e))[:k]
        ps = math.fsum(p[e] for e in sel)
        out = [0.0] * H
        for e in sel:
            hid = []
            for i in range(I):
                g = math.fsum(x[h] * w(L.gate, e, i, h) for h in range(H))
                u = math.fsum(x[h] * w(L.up, e, i, h) for h in range(H))
                hid.append(g / (1 + math.exp(-g)) * u)
            for h in range(H):
                out[h] += p[e] / ps * math.fsum(hid[i] * w(L.down, e, h, i) for i in range(I))
        outs.append(out)
    return np.array(outs)


def test_tiny_layer_against_scalar_brute_force():
    L = mi.make_layer("tiny", seed=0)
    xb, _ = mi.make_tokens(L, 3, seed=0)
    ref = _scalar_layer(xb, L)
    got = oracle.moe_layer(xb, L)["out"]
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def _small_shared_layer(seed=0):
    w = mi.Workload("small_shared", H=256, I=128, E=8, k=2, I_shared=128)
    return mi.make_layer(w, seed=seed)


def test_shared_expert_alone_when_routed_experts_are_zero():
    L = _small_shared_layer()
    xb, _ = mi.make_tokens(L, 5)
    L.gate.codes[:] = 0
    L.up.codes[:] = 0
    L.down.codes[:] = 0
    res = oracle.moe_layer(xb, L)
    x = oracle.bf16_to_f64(xb)
    sh = oracle.expert_ffn(x, oracle.dequantize(L.shared_gate.codes[0], L.shared_gate.scales[0]),
                           oracle.dequantize(L.shared_up.codes[0], L.shared_up.scales[0]),
                           oracle.dequantize(L.shared_down.codes[0], L.shared_down.scales[0]))
    assert np.array_equal(res["out"], sh)
    assert np.abs(sh).max() > 0


def test_zero_shared_expert_reduces_to_routed_layer():
    L = _small_shared_layer(1)
    xb, _ = mi.make_tokens(L, 6)
    with_sh = oracle.moe_layer(xb, L)["out"]
    L.shared_down.codes[:] = 0
    zeroed = oracle.moe_layer(xb, L)["out"]
    L2 = mi.LayerWeights(H=L.H, I=L.I, E=L.E, k=L.k, I_shared=0, Wr=L.Wr, bias=None,
                         gate=L.gate, up=L.up, down=L.down)
    routed = oracle.moe_layer(xb, L2)["out"]
    assert np.array_equal(zeroed, routed)
    assert not np.allclose(with_sh, routed)


def _gated(L, g):
    import dataclasses
    return dataclasses.replace(L, shared_gate_w=np.asarray(g, dtype=np.float32))


def test_gated_shared_expert_limits():
    """Gate vector zero: the shared output is halved (sigmoid(0) = 1/2); a
    gate driven to +inf keeps it whole, to -inf removes it.  The difference
    to the ungated layer is exactly the shared expert's output times
    (1 - factor), which pins where and with which sign the gate enters."""
    L = _small_shared_layer(2)
    xb, _ = mi.make_tokens(L, 7, seed=2)
    x = oracle.bf16_to_f64(xb)
    plain = oracle.moe_layer(xb, L)
    sh = plain["shared_y"]
    assert np.abs(sh).max() > 0
    half = oracle.moe_layer(xb, _gated(L, np.zeros(L.H)))["out"]
    assert np.allclose(half, plain["out"] - 0.5 * sh, rtol=1e-13, atol=1e-13 * np.abs(sh).max())
    # a gate along the sum of the token vectors: x_t . g is dominated by
    # |x_t|^2 > 0 for every token (checked), so +g keeps the shared output
    # whole and -g removes it
    g = 1e4 * x.sum(axis=0)
    assert np.all(x @ g > 50)
    whole = oracle.moe_layer(xb, _gated(L, g))["out"]
    assert np.allclose(whole, plain["out"], rtol=1e-13, atol=1e-13 * np.abs(sh).max())
    none = oracle.moe_layer(xb, _gated(L, -g))["out"]
    assert np.allclose(none, plain["out"] - sh, rtol=1e-12, atol=1e-12 * np.abs(sh).max())


def test_gate_factor_against_scalar_loop():
    """sigmoid(x . g) per token, against a math.fsum dot and math.exp."""
    w = mi.Workload("small_shared", H=256, I=128, E=8, k=2, I_shared=128)
    L = mi.make_layer(w, seed=3, shared_gated=True)
    assert L.shared_gate_w is not None and L.shared_gate_w.shape == (L.H,)
    xb, _ = mi.make_tokens(L, 5, seed=3)
    x = oracle.bf16_to_f64(xb)
    got = oracle.shared_gate_factor(x, L)
    for t in range(5):
        z = math.fsum(float(x[t, h]) * float(L.shared_gate_w[h]) for h in range(L.H))
        assert abs(got[t] - 1.0 / (1.0 + math.exp(-z))) <= 1e-14
    # and the gated layer scales the shared output by it, token by token
    ungated = oracle.moe_layer(xb, _gated(L, np.zeros(L.H)))  # factor 1/2
    gated = oracle.moe_layer(xb, L)
    sh_half = ungated["shared_y"]  # already scaled by 1/2
    assert np.allclose(gated["out"] - (ungated["out"] - sh_half),
                       2.0 * sh_half * got[:, None], rtol=1e-12,
                       atol=1e-12 * np.abs(sh_half).max())


def test_sampled_path_equals_full_layer():
    L = mi.make_layer("tiny", seed=3)
    xb, _ = mi.make_tokens(L, 8, seed=3)
    full = oracle.moe_layer(xb, L)
    toks = [7, 0, 3]
    s = oracle.moe_layer_sampled(xb, L, toks)
    assert np.allclose(s["out_sampled"], full["out"][toks], rtol=1e-13, atol=1e-15)
    for key in ("topk_idx", "expert_off", "row_token", "tok_slot_row"):
        assert np.array_equal(s[key], full[key])


def test_combine_against_loop():
    rng = np.random.default_rng(4)
    T, k, H = 5, 3, 7
    y = rng.standard_normal((T * k, H))
    tsr = rng.permutation(T * k).astype(np.int32)
    w = rng.random((T, k))
    sh = rng.standard_normal((T, H))
    out = oracle.combine(y, tsr, w, sh)
    for t in range(T):
        for h in range(H):
            ref = math.fsum([w[t, j] * y[tsr[t * k + j], h] for j in range(k)] + [sh[t, h]])
            assert abs(out[t, h] - ref) < 1e-14


@pytest.mark.parametrize("name,T", [("tiny", 8), ("skewed", 64)])
def test_generated_inputs_keep_the_logit_gap(name, T):
    L = mi.make_layer(name, seed=0) if name == "tiny" else None
    if L is None:
        w = mi.WORKLOADS[name]
        # Only the router matters for the guard: a layer with tiny experts.
        L = mi.make_layer(mi.Workload("guard", H=w.H, I=128, E=w.E, k=w.k,
                                      zipf_s=w.zipf_s), seed=0)
    xb, _ = mi.make_tokens(L, T, seed=0)
    l = oracle.router_logits(oracle.bf16_to_f64(xb), L.Wr, L.bias)
    top = -np.sort(-l, axis=1)[:, :L.k + 1]
    assert np.all(np.diff(-top, axis=1) > 1e-4)
