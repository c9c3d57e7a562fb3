"""Seeded synthetic inputs for the block-FP8 MoE FFN layer.

This module only draws data.  It holds none of the layer's arithmetic: no
E4M3 decode, no dequantisation, no softmax, routing, permutation or FFN.  It
is the one module that both the fp64 oracle (``oracle/``) and the CUDA path
(``block_fp8_expert_gb300``) are fed from, as plain arrays.

What it draws, per named workload (the layer shapes of the two model families
in the colizig README's model table, "What this project is trying to prove":
128 experts top-8 without a shared expert, and 512 experts top-10 plus one
shared expert):

* activations x ~ N(0, 1), rounded to bfloat16 (round-to-nearest-even);
* router weights Wr ~ N(0, 0.02^2), float32, layout [E, H];
* expert weights as E4M3 codes of z ~ N(0, 1) (the true weight is z times the
  block scale, so the code is the quantised w / scale), layouts
  gate/up [E, I, H] and down [E, H, I], uint8;
* one float32 scale per 128x128 block, ~ U(0.005, 0.02), layouts
  [E, ceil(I/128), ceil(H/128)] (gate/up) and [E, ceil(H/128), ceil(I/128)]
  (down); other scale distributions and a code gain can be asked for, to
  cover the scale range of real block-FP8 checkpoints;
* for the skewed workload, a router bias b[e] = ln q_{pi(e)} with
  q_r proportional to r^-1.2 (Zipf, s = 1.2) and pi a seeded permutation.

The encoder below is the quantiser that produced the checkpoint, not part of
the layer: it rounds to nearest-even on the E4M3 grid (the OCP FP8 E4M3
variant without infinities, largest finite magnitude 448) and saturates.

Gap guard: a token whose router logits (fp64, bias included) have any
adjacent gap among its k+1 largest values at or below 1e-4 is redrawn from the
same stream until none has.  That keeps the selected expert set and its
descending order unique, so both sides can be compared index for index.  The
guard needs the logits, so it evaluates x @ Wr^T + b with one fp64 matmul; that
product only decides which draws belong to the input domain.
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np

BLOCK = 128
GAP_MIN = 1e-4

# Stream tags: every tensor draws from its own counter-free numpy stream
# keyed by (seed, tag, index), so experts can be drawn in parallel and any one
# of them can be regenerated alone.
_TAG = {"wr": 1, "bias": 2, "gate": 3, "up": 4, "down": 5, "gate_s": 6,
        "up_s": 7, "down_s": 8, "sh_gate": 9, "sh_up": 10, "sh_down": 11,
        "sh_gate_s": 12, "sh_up_s": 13, "sh_down_s": 14, "x": 15, "sh_gate_w": 16}


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and distribution of one synthetic layer."""
    name: str
    H: int
    I: int
    E: int
    k: int
    I_shared: int = 0
    zipf_s: Optional[float] = None
    tokens: tuple = ()


WORKLOADS = {
    # 8 tokens, hidden 256, intermediate 128, 16 experts, top-2.
    "tiny": Workload("tiny", H=256, I=128, E=16, k=2, tokens=(8,)),
    # Qwen3-MoE-shaped layer (128 experts, top-8, no shared expert).
    "qwen3moe_decode": Workload("qwen3moe_decode", H=2048, I=768, E=128, k=8,
                                tokens=(1, 8, 64)),
    "qwen3moe_prefill": Workload("qwen3moe_prefill", H=2048, I=768, E=128, k=8,
                                 tokens=(4096,)),
    # 512 routed experts top-10 plus one always-on shared expert.
    "large_sparse": Workload("large_sparse", H=2048, I=512, E=512, k=10,
                             I_shared=512, tokens=(1, 256)),
    # Qwen3-MoE shape with a Zipf(1.2) router bias: few hot experts.
    "skewed": Workload("skewed", H=2048, I=768, E=128, k=8, zipf_s=1.2,
                       tokens=(1, 16, 256, 2048, 16384)),
}


@dataclasses.dataclass
class Fp8Mat:
    codes: np.ndarray   # uint8 [E, rows, cols]
    scales: np.ndarray  # float32 [E, ceil(rows/128), ceil(cols/128)]


@dataclasses.dataclass
class LayerWeights:
    H: int
    I: int
    E: int
    k: int
    I_shared: int
    Wr: np.ndarray                 # float32 [E, H]
    bias: Optional[np.ndarray]     # float32 [E] or None
    gate: Fp8Mat
    up: Fp8Mat
    down: Fp8Mat
    shared_gate: Optional[Fp8Mat] = None
    shared_up: Optional[Fp8Mat] = None
    shared_down: Optional[Fp8Mat] = None
    # gated shared expert only: float32 [H], the shared expert's output is
    # scaled per token by sigmoid(x . shared_gate_w)
    shared_gate_w: Optional[np.ndarray] = None

    @property
    def has_shared(self) -> bool:
        return self.I_shared > 0


def _rng(seed: int, tag: str, idx: int = 0) -> np.random.Generator:
    return np.random.default_rng([int(seed), _TAG[tag], int(idx)])


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


# --------------------------------------------------------------------------
# quantisers (data preparation, not layer arithmetic)
# --------------------------------------------------------------------------

def bf16_bits_rne(a: np.ndarray) -> np.ndarray:
    """float32 array -> bfloat16 bit patterns (uint16), round-to-nearest-even."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    return ((b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def e4m3_encode(z: np.ndarray) -> np.ndarray:
    """float32 array -> E4M3 codes, round-to-nearest-even, saturating at 448.

    Never emits the NaN codes 0x7F / 0xFF; emits 0x80 for -0.0 and for
    negative values that round to zero.
    """
    z = np.ascontiguousarray(z, dtype=np.float32)
    b = z.view(np.uint32)
    sign = ((b >> np.uint32(24)) & np.uint32(0x80)).astype(np.uint8)
    a = b & np.uint32(0x7FFFFFFF)
    # Normal E4M3 range (|z| >= 2^-6): keep 3 mantissa bits with RNE, then
    # move the exponent bias from 127 to 7.  A mantissa carry moves into the
    # exponent by itself.
    lsb = (a >> np.uint32(20)) & np.uint32(1)
    r = (a + np.uint32(0x7FFFF) + lsb) >> np.uint32(20)
    normal = np.minimum(r.astype(np.int64) - (120 << 3), 0x7E)
    # Subnormal range: multiples of 2^-9, rint is round-half-even.
    sub = np.rint(np.abs(z) * np.float32(512.0)).astype(np.int64)
    mag = np.where(a < np.uint32(121 << 23), sub, normal).astype(np.uint8)
    return mag | sign


# --------------------------------------------------------------------------
# drawing
# --------------------------------------------------------------------------

SCALE_RANGE = (0.005, 0.02)


def _draw_codes(seed: int, tag: str, e: int, rows: int, cols: int,
                code_gain: float = 1.0) -> np.ndarray:
    z = _rng(seed, tag, e).standard_normal((rows, cols), dtype=np.float32)
    if code_gain != 1.0:
        z = z * np.float32(code_gain)
    return e4m3_encode(z)


def _draw_scales(seed: int, tag: str, E: int, rows: int, cols: int,
                 scale_range=SCALE_RANGE, scale_dist: str = "uniform") -> np.ndarray:
    """One float32 scale per 128x128 block: U(lo, hi), or ("loguniform")
    exp(U(ln lo, ln hi)), which mixes magnitudes across the blocks of one
    row block."""
    shape = (E, _cdiv(rows, BLOCK), _cdiv(cols, BLOCK))
    lo, hi = scale_range
    rng = _rng(seed, tag)
    if scale_dist == "uniform":
        return rng.uniform(lo, hi, size=shape).astype(np.float32)
    if scale_dist == "loguniform":
        return np.exp(rng.uniform(math.log(lo), math.log(hi), size=shape)).astype(np.float32)
    raise ValueError(f"unknown scale distribution {scale_dist!r}")


def _draw_fp8(seed: int, tag: str, stag: str, E: int, rows: int, cols: int,
              pool: ThreadPoolExecutor, code_gain: float = 1.0, scale_range=SCALE_RANGE,
              scale_dist: str = "uniform") -> Fp8Mat:
    codes = np.empty((E, rows, cols), dtype=np.uint8)

    def one(e):
        codes[e] = _draw_codes(seed, tag, e, rows, cols, code_gain)

    list(pool.map(one, range(E)))
    return Fp8Mat(codes, _draw_scales(seed, stag, E, rows, cols, scale_range, scale_dist))


def zipf_bias(E: int, s: float, seed: int) -> np.ndarray:
    """b[e] = ln q_{pi(e)}, q_r = r^-s / sum_r r^-s, pi a seeded permutation."""
    ranks = np.arange(1, E + 1, dtype=np.float64)
    q = ranks ** (-s)
    q /= q.sum()
    perm = _rng(seed, "bias").permutation(E)
    return np.log(q[perm]).astype(np.float32)


def make_layer(workload: str | Workload, seed: int = 0,
               threads: Optional[int] = None, code_gain: float = 1.0,
               scale_range=SCALE_RANGE, scale_dist: str = "uniform",
               shared_gated: bool = False) -> LayerWeights:
    """Draw every weight of one layer of the named workload.

    The defaults are the workloads' distributions.  code_gain multiplies the
    N(0, 1) draw before it is encoded (100 gives codes spread over the whole
    E4M3 range, as an amax-scaled checkpoint has); scale_range and scale_dist
    choose the block scales' distribution (see _draw_scales); shared_gated
    adds a gate vector ~ N(0, 0.02^2) for the shared expert (layers with a
    shared expert only)."""
    w = WORKLOADS[workload] if isinstance(workload, str) else workload
    H, I, E = w.H, w.I, w.E
    threads = threads or min(32, os.cpu_count() or 1)
    Wr = (_rng(seed, "wr").standard_normal((E, H), dtype=np.float32)
          * np.float32(0.02))
    bias = zipf_bias(E, w.zipf_s, seed) if w.zipf_s else None
    kw = dict(code_gain=code_gain, scale_range=scale_range, scale_dist=scale_dist)
    with ThreadPoolExecutor(threads) as pool:
        gate = _draw_fp8(seed, "gate", "gate_s", E, I, H, pool, **kw)
        up = _draw_fp8(seed, "up", "up_s", E, I, H, pool, **kw)
        down = _draw_fp8(seed, "down", "down_s", E, H, I, pool, **kw)
        sg = su = sd = None
        if w.I_shared:
            Is = w.I_shared
            sg = _draw_fp8(seed, "sh_gate", "sh_gate_s", 1, Is, H, pool, **kw)
            su = _draw_fp8(seed, "sh_up", "sh_up_s", 1, Is, H, pool, **kw)
            sd = _draw_fp8(seed, "sh_down", "sh_down_s", 1, H, Is, pool, **kw)
    gw = None
    if shared_gated and w.I_shared:
        gw = (_rng(seed, "sh_gate_w").standard_normal(H, dtype=np.float32)
              * np.float32(0.02))
    return LayerWeights(H=H, I=I, E=E, k=w.k, I_shared=w.I_shared, Wr=Wr,
                        bias=bias, gate=gate, up=up, down=down,
                        shared_gate=sg, shared_up=su, shared_down=sd, shared_gate_w=gw)


def with_scales(layer: LayerWeights, seed: int, scale_range,
                scale_dist: str = "uniform") -> LayerWeights:
    """The same layer (same codes, router and bias arrays, shared not
    copied) with every block scale redrawn from another distribution."""
    def re(m: Optional[Fp8Mat], tag: str) -> Optional[Fp8Mat]:
        if m is None:
            return None
        E, nr, nc = m.scales.shape
        return Fp8Mat(m.codes, _draw_scales(seed, tag, E, nr * BLOCK, nc * BLOCK,
                                            scale_range, scale_dist))
    return dataclasses.replace(
        layer, gate=re(layer.gate, "gate_s"), up=re(layer.up, "up_s"),
        down=re(layer.down, "down_s"), shared_gate=re(layer.shared_gate, "sh_gate_s"),
        shared_up=re(layer.shared_up, "sh_up_s"), shared_down=re(layer.shared_down, "sh_down_s"))


def _bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _gap_ok(logits: np.ndarray, k: int) -> np.ndarray:
    """True per row where the k+1 largest logits are pairwise > GAP_MIN apart."""
    E = logits.shape[1]
    m = min(k + 1, E)
    top = -np.sort(-logits, axis=1)[:, :m]
    if m < 2:
        return np.ones(logits.shape[0], dtype=bool)
    return np.all(top[:, :-1] - top[:, 1:] > GAP_MIN, axis=1)


def make_tokens(layer: LayerWeights, T: int, seed: int = 0,
                max_rounds: int = 1000) -> tuple[np.ndarray, int]:
    """Draw x [T, H] as bfloat16 bits (uint16) under the gap guard.

    Returns (x_bits, redraws): redraws counts replaced rows.
    """
    rng = _rng(seed, "x", T)
    H = layer.H
    x = bf16_bits_rne(rng.standard_normal((T, H), dtype=np.float32))
    if T == 0:
        return x, 0
    Wr64 = layer.Wr.astype(np.float64)
    b64 = None if layer.bias is None else layer.bias.astype(np.float64)

    def logits_of(rows):
        l = _bf16_bits_to_f64(x[rows]) @ Wr64.T
        return l if b64 is None else l + b64

    bad = np.nonzero(~_gap_ok(logits_of(np.arange(T)), layer.k))[0]
    redraws = 0
    for _ in range(max_rounds):
        if bad.size == 0:
            return x, redraws
        for t in bad:  # ascending token order, one row at a time
            x[t] = bf16_bits_rne(rng.standard_normal(H, dtype=np.float32))
        redraws += bad.size
        bad = bad[~_gap_ok(logits_of(bad), layer.k)]
    raise RuntimeError("gap guard did not converge")


def total_bytes(layer: LayerWeights) -> int:
    """Host bytes of all weights of a layer (codes, scales, router)."""
    n = layer.Wr.nbytes + (0 if layer.bias is None else layer.bias.nbytes)
    for m in (layer.gate, layer.up, layer.down, layer.shared_gate,
              layer.shared_up, layer.shared_down):
        if m is not None:
            n += m.codes.nbytes + m.scales.nbytes
    return n
