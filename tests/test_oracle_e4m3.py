"""Pins for the oracle's E4M3 decode and dequantisation.

The decode is checked against the format's fixed points (tests/golden/
e4m3_spot.txt), against the FP8 decode of a library (torch.float8_e4m3fn),
and against structural facts of the format (monotone codes, sign symmetry,
value set).  The dequantisation is pinned by a probe whose every block has a
distinct scale, so a transposed or shifted scale index changes the result.
"""
import math
import os

import numpy as np
import pytest

import oracle
from moe_inputs import e4m3_encode, bf16_bits_rne

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_spot.txt")


def _read_spot():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            code, val = line.split()
            rows.append((int(code, 16), val))
    return rows


def test_spot_values():
    rows = _read_spot()
    assert len(rows) >= 12
    for code, val in rows:
        got = oracle.e4m3_decode(np.array([code]))[0]
        if val == "nan":
            assert math.isnan(got), hex(code)
        elif val == "-0":
            assert got == 0.0 and math.copysign(1.0, got) < 0, hex(code)
        else:
            assert got == float.fromhex(val) if val.startswith(("0x", "-0x")) \
                else got == float(val), (hex(code), got, val)


def test_all_codes_match_library_decode():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    mine = oracle.e4m3_decode(codes)
    nan_l, nan_m = np.isnan(lib), np.isnan(mine)
    assert np.array_equal(nan_l, nan_m)
    assert np.array_equal(lib[~nan_l], mine[~nan_m])
    assert set(np.nonzero(nan_m)[0]) == {0x7F, 0xFF}


def test_structure_of_the_value_set():
    v = oracle.e4m3_decode(np.arange(256))
    pos = v[:0x7F]
    # Codes 0x00..0x7E are strictly increasing magnitudes from 0 to 448.
    assert np.all(np.diff(pos) > 0)
    assert pos[0] == 0.0 and pos[-1] == 448.0
    # Sign symmetry.
    assert np.array_equal(v[0x80:0xFF], -pos)
    # Subnormals are evenly spaced by 2^-9; each binade e >= 1 holds 8
    # values evenly spaced by 2^(e-10).
    assert np.allclose(np.diff(pos[:9]), 2.0 ** -9, rtol=0, atol=0)
    for e in range(1, 16):
        seg = pos[8 * e: 8 * e + 8]
        assert np.all(np.diff(seg) == 2.0 ** (e - 10)), e


def test_encoder_roundtrips_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)],
                     dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(e4m3_encode(vals), codes)


def test_encoder_matches_library_rounding():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    z = np.concatenate([rng.standard_normal(200000).astype(np.float32),
                        (rng.standard_normal(20000) * 1e-3).astype(np.float32),
                        (rng.standard_normal(20000) * 100).astype(np.float32)])
    z = z[np.abs(z) < 448]
    lib = torch.from_numpy(z).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3_encode(z), lib)
    # Ties round to the even code: midpoints between neighbours.
    v = oracle.e4m3_decode(np.arange(0x7F)).astype(np.float64)
    mids = ((v[:-1] + v[1:]) / 2).astype(np.float32)
    got = e4m3_encode(mids)
    expect = np.where(np.arange(0x7E) % 2 == 0, np.arange(0x7E), np.arange(1, 0x7F))
    assert np.array_equal(got, expect.astype(np.uint8))
    # Saturation at 448.
    assert e4m3_encode(np.array([1e6, -500.0], np.float32)).tolist() == [0x7E, 0xFE]


def test_bf16_rounding_matches_library():
    torch = pytest.importorskip("torch")
    z = np.random.default_rng(3).standard_normal(100000).astype(np.float32)
    lib = torch.from_numpy(z).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf16_bits_rne(z), lib)
    back = oracle.bf16_to_f64(lib)
    assert np.array_equal(back, torch.from_numpy(lib.view(np.int16)).view(torch.bfloat16).double().numpy())


@pytest.mark.parametrize("R,C", [(256, 384), (300, 200), (128, 128), (1, 130)])
def test_dequant_block_scale_probe(R, C):
    """All codes 1.0 (0x38), scale S[a, b] = 1 + a + 16 b: W[r, c] must be
    S[r // 128, c // 128] exactly, and x one-hot at column h selects it."""
    nb_r, nb_c = -(-R // 128), -(-C // 128)
    a, b = np.meshgrid(np.arange(nb_r), np.arange(nb_c), indexing="ij")
    S = (1 + a + 16 * b).astype(np.float32)
    W = oracle.dequantize(np.full((R, C), 0x38, np.uint8), S)
    for r in range(0, R, max(1, R // 7)):
        for c in range(0, C, max(1, C // 5)):
            assert W[r, c] == 1 + (r // 128) + 16 * (c // 128)
    h = C - 1
    x = np.zeros(C)
    x[h] = 1.0
    g = W @ x
    assert np.array_equal(g, S[np.arange(R) // 128, h // 128].astype(np.float64))


def test_dequant_elementwise_against_scalar_loop():
    rng = np.random.default_rng(11)
    R, C = 200, 260
    codes = rng.integers(0, 256, (R, C), dtype=np.uint8)
    codes[codes == 0x7F] = 0x7E
    codes[codes == 0xFF] = 0xFE
    S = rng.uniform(0.005, 0.02, (2, 3)).astype(np.float32)
    W = oracle.dequantize(codes, S)
    for r in range(0, R, 13):
        for c in range(0, C, 17):
            code = int(codes[r, c])
            s, e, m = code >> 7, (code >> 3) & 15, code & 7
            mag = (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
            ref = (-mag if s else mag) * float(S[r // 128, c // 128])
            assert W[r, c] == ref
