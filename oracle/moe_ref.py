"""The oracle's arithmetic: one MoE FFN layer with block-FP8 expert weights.

Test infrastructure only (see ``oracle/__init__.py``).

Sources, cited by page title and section:

* colizig README (page "benmaster82/colizig"), model table under "What this
  project is trying to prove": experts with top-k routing, 128 experts top-8
  without a shared expert, or 512 experts top-10 plus one shared expert.
* colizig README, "Features": block-FP8 (E4M3) weights, dequantised inside a
  fused decode+FMA dot product; MoE per-expert evaluation.
* colizig README, "Status" table: "MoE (+shared expert)".
* The layer statement this build implements: router GEMM, softmax over
  experts, top-k with renormalisation, permutation of tokens by expert,
  per-expert gate/up projections with SwiGLU and a down projection, weights
  dequantised from E4M3 codes with one fp32 scale per 128x128 block, an
  optional always-on shared expert, and a weighted combine back to token
  order.

Readings where the pages are silent:

R1  "E4M3" is the OCP FP8 E4M3 variant without infinities (bias 7, codes
    0x7F/0xFF are NaN, largest finite 448), the format of block-FP8
    checkpoints.
R2  A block scale multiplies: W[r, c] = dec(C[r, c]) * S[r // 128, c // 128];
    rows are output features, columns input features (Linear [out, in]).
R3  The router is l = x Wr^T + b with Wr [E, H]; b is absent except for the
    skewed workload.
R4  Top-k takes the k largest softmax probabilities in descending order, ties
    to the lower expert index; renormalised weights are w_j = p_j / sum p_sel.
R5  The permutation is expert-major and, inside one expert's segment,
    ascending in token index.
R6  SwiGLU is silu(x Wg^T) * (x Wu^T) with silu(z) = z / (1 + exp(-z)).
R7  The shared expert sees every token with weight 1 (no gate) and is added
    after the routed combine.
R10 Gated variant (not on the pages, which say only "+ 1 shared"): when the
    layer carries a gate vector g [H], the shared expert's output for token
    t is scaled by sigmoid(x[t] . g) before it is added.
R11 FP8-activation variant (not on the pages, whose block-FP8 format covers
    weights only): the expert projections' inputs (x, then hid) are
    quantised to E4M3 per row and group of 128 consecutive input features,
    the grouping of the weights' 128-wide scale blocks.  For a group with
    largest magnitude a (float32): a == 0 gives codes 0 and scale 0;
    otherwise inv = fp32(448 / a), each value v becomes the E4M3 code
    nearest to fp32(v * inv) (ties to the even code, magnitudes at or above
    448 saturate to 448), and the scale is s = fp32(a / 448); the
    dequantised value is dec(code) * s.  hid is quantised from its float32
    value.  Everything else is as in the bf16-activation layer.
"""
from __future__ import annotations

import numpy as np

BLOCK = 128


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """E4M3 code -> float64, from the bit fields (reading R1).

    A code is s eeee mmm.  e == 0: (-1)^s 2^-6 (m/8) (zero and subnormals);
    e == 15 and m == 7: NaN; otherwise (-1)^s 2^(e-7) (1 + m/8).
    """
    c = np.asarray(codes).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 0x7
    sign = np.where(s == 1, -1.0, 1.0)
    sub = sign * np.ldexp(m / 8.0, -6)
    nrm = sign * np.ldexp(1.0 + m / 8.0, e - 7)
    v = np.where(e == 0, sub, nrm)
    return np.where((e == 15) & (m == 7), np.nan, v)


_TABLE = e4m3_decode(np.arange(256))


def e4m3_table() -> np.ndarray:
    """The 256 decoded values, indexed by code (a copy)."""
    return _TABLE.copy()


def bf16_to_f64(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64; exact (bf16 is the top half
    of an IEEE binary32)."""
    b = np.asarray(bits).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def dequantize(codes, scales, block: int = BLOCK) -> np.ndarray:
    """Block-FP8 matrix -> float64 (reading R2).

    codes [R, C] uint8, scales [ceil(R/block), ceil(C/block)] float32.
    Ragged edge blocks use the scale of the block they fall in.
    """
    codes = np.asarray(codes)
    R, C = codes.shape
    S = np.asarray(scales, dtype=np.float64)
    assert S.shape == (-(-R // block), -(-C // block)), S.shape
    full = np.repeat(np.repeat(S, block, axis=0), block, axis=1)[:R, :C]
    return _TABLE[codes] * full


def e4m3_encode_rne(v) -> np.ndarray:
    """float32 values -> E4M3 codes (uint8), rounded to the nearest finite
    E4M3 value, ties to the code with the even mantissa, magnitudes at or
    above 448 saturated to 448 (reading R11).  NaN is not accepted."""
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    assert not np.isnan(v).any()
    pos = _TABLE[:127]                      # codes 0x00 .. 0x7E, increasing
    a = np.minimum(np.abs(v), 448.0)
    hi = np.searchsorted(pos, a, side="left")  # first value >= a
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - pos[lo]
    d_hi = pos[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    return (code | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def act8_quantize(rows, group: int = BLOCK):
    """Per-row, per-128-group E4M3 quantisation of float32 activations
    (reading R11).  rows [n, K] (float32-representable), K % group == 0.
    Returns codes uint8 [n, K] and scales float32 [n, K / group]."""
    r = np.asarray(rows, dtype=np.float32)
    n, K = r.shape
    assert K % group == 0
    g = r.reshape(n, K // group, group)
    amax = np.abs(g).max(axis=2).astype(np.float32)
    safe = np.where(amax > 0, amax, np.float32(1))
    inv = (np.float32(448.0) / safe).astype(np.float32)
    v = (g * inv[:, :, None]).astype(np.float32)
    codes = e4m3_encode_rne(v).reshape(n, K)
    codes = np.where(np.repeat(amax, group, axis=1) > 0, codes, 0).astype(np.uint8)
    scales = np.where(amax > 0, (amax / np.float32(448.0)).astype(np.float32),
                      np.float32(0)).astype(np.float32)
    return codes, scales


def act8_dequantize(codes, scales, group: int = BLOCK) -> np.ndarray:
    """dec(code) * s per group, float64 [n, K]."""
    return _TABLE[np.asarray(codes)] * np.repeat(np.asarray(scales, np.float64), group, axis=1)


def act8_round(rows, group: int = BLOCK) -> np.ndarray:
    """Quantise then dequantise (reading R11), float64."""
    return act8_dequantize(*act8_quantize(rows, group), group)


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------

def router_logits(x, Wr, bias=None) -> np.ndarray:
    """l[t, e] = sum_h x[t, h] Wr[e, h] (+ b[e]) in float64 (reading R3)."""
    l = np.asarray(x, dtype=np.float64) @ np.asarray(Wr, dtype=np.float64).T
    if bias is not None:
        l = l + np.asarray(bias, dtype=np.float64)[None, :]
    return l


def softmax(l) -> np.ndarray:
    """Softmax over experts (last axis), shifted by the row maximum."""
    l = np.asarray(l, dtype=np.float64)
    z = np.exp(l - l.max(axis=-1, keepdims=True))
    return z / z.sum(axis=-1, keepdims=True)


def topk_renorm(p, k: int):
    """Top-k experts per token and their renormalised weights (reading R4).

    Returns (idx int32 [T, k], w float64 [T, k]); idx in descending p, ties
    to the lower expert index; w = p_sel / sum(p_sel).
    """
    p = np.asarray(p, dtype=np.float64)
    T, E = p.shape
    # Stable sort of -p keeps equal probabilities in ascending expert order.
    order = np.argsort(-p, axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(p, order, axis=1)
    w = sel / sel.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w


def permute(topk_idx, E: int):
    """Expert-contiguous segments of the (token, slot) pairs (reading R5).

    cnt[e] = #{(t, j) : idx[t, j] == e}; off = exclusive scan of cnt with
    off[E] = T*k.  Segment e holds its tokens in ascending t.  Returns
    (off int32 [E+1], row_token int32 [P], tok_slot_row int32 [T*k]) with
    row_token[r] the token of permuted row r and tok_slot_row[t*k + j] the
    row of pair (t, j).
    """
    idx = np.asarray(topk_idx, dtype=np.int64)
    T, k = idx.shape
    flat = idx.reshape(-1)
    cnt = np.bincount(flat, minlength=E)
    off = np.zeros(E + 1, dtype=np.int64)
    off[1:] = np.cumsum(cnt)
    # Sort the flattened pair index q = t*k + j by expert; a stable sort
    # keeps ascending q, which is ascending t inside one expert.
    order = np.argsort(flat, kind="stable")
    row_token = (order // k).astype(np.int32)
    tok_slot_row = np.empty(T * k, dtype=np.int32)
    tok_slot_row[order] = np.arange(T * k, dtype=np.int32)
    return off.astype(np.int32), row_token, tok_slot_row


# ---------------------------------------------------------------------------
# experts
# ---------------------------------------------------------------------------

def silu(z) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    # exp(-z) overflows to inf for z < -709; z / inf is then the limit 0
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def expert_ffn(xp, Wg, Wu, Wd) -> np.ndarray:
    """y = (silu(xp Wg^T) * (xp Wu^T)) Wd^T for the rows xp [n, H] of one
    expert (reading R6).  Wg, Wu [I, H], Wd [H, I], all float64."""
    g = xp @ Wg.T
    u = xp @ Wu.T
    return (silu(g) * u) @ Wd.T


def expert_ffn_act8(xp, Wg, Wu, Wd, quant=None) -> np.ndarray:
    """The FP8-activation expert (reading R11): the rows xp [n, H] and the
    float32 hid are each quantised per 128-group before their projection.
    ``quant`` replaces the quantise-dequantise step (tests only)."""
    q = act8_round if quant is None else quant
    xh = q(np.asarray(xp, dtype=np.float32))
    hid = silu(xh @ Wg.T) * (xh @ Wu.T)
    return q(hid.astype(np.float32)) @ Wd.T


def combine(y_perm, tok_slot_row, topk_w, shared_y=None) -> np.ndarray:
    """out[t] = sum_j w[t, j] y_perm[tok_slot_row[t*k + j]] (+ shared_y[t])
    (reading R7 for the shared term)."""
    w = np.asarray(topk_w, dtype=np.float64)
    T, k = w.shape
    rows = np.asarray(tok_slot_row).reshape(T, k)
    out = np.einsum("tj,tjh->th", w, np.asarray(y_perm)[rows])
    if shared_y is not None:
        out = out + shared_y
    return out


# ---------------------------------------------------------------------------
# the whole layer
# ---------------------------------------------------------------------------

def shared_gate_factor(x, layer) -> np.ndarray:
    """Per-token factor of the shared expert's output (readings R7, R10): 1
    without a gate vector, else sigmoid(x . g), float64 [T]."""
    g = getattr(layer, "shared_gate_w", None)
    x = np.asarray(x, dtype=np.float64)
    if g is None:
        return np.ones(x.shape[0])
    z = x @ np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def _expert_mats(mat, e):
    return dequantize(mat.codes[e], mat.scales[e])


def moe_layer(x_bits, layer, keep_intermediates: bool = True, act8: bool = False,
              quant=None) -> dict:
    """The full layer on every token, float64.  act8: the FP8-activation
    variant (reading R11) of every expert, routed and shared; the routing
    is the same.

    ``layer`` carries Wr, bias, gate/up/down (codes [E, ...], scales) and the
    optional shared expert (see ``moe_inputs.LayerWeights``).  Returns a dict
    with logits, p, topk_idx, topk_w, expert_off, row_token, tok_slot_row,
    y_perm, shared_y and out (all float64 except the integer arrays).
    """
    x = bf16_to_f64(x_bits)
    T = x.shape[0]
    k, E = layer.k, layer.E
    logits = router_logits(x, layer.Wr, layer.bias)
    p = softmax(logits)
    idx, w = topk_renorm(p, k)
    off, row_token, tok_slot_row = permute(idx, E)
    ffn = (lambda *m: expert_ffn_act8(*m, quant=quant)) if act8 else expert_ffn
    y_perm = np.zeros((T * k, layer.H), dtype=np.float64)
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        if a == b:
            continue
        y_perm[a:b] = ffn(x[row_token[a:b]],
                          _expert_mats(layer.gate, e),
                          _expert_mats(layer.up, e),
                          _expert_mats(layer.down, e))
    shared_y = None
    if layer.I_shared:
        shared_y = ffn(x, _expert_mats(layer.shared_gate, 0),
                       _expert_mats(layer.shared_up, 0),
                       _expert_mats(layer.shared_down, 0))
        shared_y = shared_y * shared_gate_factor(x, layer)[:, None]
    out = combine(y_perm, tok_slot_row, w, shared_y)
    res = dict(topk_idx=idx, topk_w=w, expert_off=off, row_token=row_token,
               tok_slot_row=tok_slot_row, out=out)
    if keep_intermediates:
        res.update(logits=logits, p=p, y_perm=y_perm, shared_y=shared_y)
    return res


def moe_layer_sampled(x_bits, layer, tokens, act8: bool = False) -> dict:
    """Routing and permutation for every token; the layer output only for the
    listed tokens (each computed from its own k experts, one by one).  act8:
    the FP8-activation variant (reading R11; quantisation is per row, so a
    token's rows do not depend on the other tokens).

    Returns the routing/permutation arrays of ``moe_layer`` plus
    out_sampled float64 [len(tokens), H] in the order of ``tokens``.
    """
    x = bf16_to_f64(x_bits)
    k, E = layer.k, layer.E
    logits = router_logits(x, layer.Wr, layer.bias)
    p = softmax(logits)
    idx, w = topk_renorm(p, k)
    off, row_token, tok_slot_row = permute(idx, E)
    tokens = np.asarray(tokens, dtype=np.int64)
    out = np.zeros((tokens.size, layer.H), dtype=np.float64)
    # Group the sampled (token, slot) pairs by expert so that each expert is
    # dequantised once.
    pairs = {}
    for n, t in enumerate(tokens):
        for j in range(k):
            pairs.setdefault(int(idx[t, j]), []).append((n, int(t), j))
    ffn = expert_ffn_act8 if act8 else expert_ffn
    for e, lst in pairs.items():
        rows = np.array([t for _, t, _ in lst])
        y = ffn(x[rows], _expert_mats(layer.gate, e),
                _expert_mats(layer.up, e), _expert_mats(layer.down, e))
        for (n, t, j), yr in zip(lst, y):
            out[n] += w[t, j] * yr
    if layer.I_shared:
        out += (expert_ffn(x[tokens], _expert_mats(layer.shared_gate, 0),
                           _expert_mats(layer.shared_up, 0),
                           _expert_mats(layer.shared_down, 0))
                * shared_gate_factor(x[tokens], layer)[:, None])
    return dict(topk_idx=idx, topk_w=w, expert_off=off, row_token=row_token,
                tok_slot_row=tok_slot_row, out_sampled=out)
