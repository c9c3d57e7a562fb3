"""The seeded generator: determinism, shapes, value ranges and the Zipf skew."""
import numpy as np

import moe_inputs as mi
import oracle


def test_deterministic_and_seed_sensitive():
    a = mi.make_layer("tiny", seed=0)
    b = mi.make_layer("tiny", seed=0)
    c = mi.make_layer("tiny", seed=1)
    assert np.array_equal(a.gate.codes, b.gate.codes)
    assert np.array_equal(a.Wr, b.Wr)
    assert not np.array_equal(a.gate.codes, c.gate.codes)
    xa, _ = mi.make_tokens(a, 8, 0)
    xb, _ = mi.make_tokens(b, 8, 0)
    assert np.array_equal(xa, xb)


def test_shapes_and_ranges():
    L = mi.make_layer("tiny", seed=0)
    assert L.gate.codes.shape == (16, 128, 256) and L.gate.codes.dtype == np.uint8
    assert L.down.codes.shape == (16, 256, 128)
    assert L.gate.scales.shape == (16, 1, 2) and L.down.scales.shape == (16, 2, 1)
    for m in (L.gate, L.up, L.down):
        assert not np.any((m.codes == 0x7F) | (m.codes == 0xFF))
        assert m.scales.min() >= 0.005 and m.scales.max() <= 0.02
    # Codes of N(0, 1): the decoded values have unit spread.
    v = oracle.e4m3_decode(L.gate.codes)
    assert abs(v.std() - 1.0) < 0.02 and abs(v.mean()) < 0.02
    assert abs(L.Wr.std() - 0.02) < 0.002


def test_zipf_bias_skews_routing():
    w = mi.WORKLOADS["skewed"]
    b = mi.zipf_bias(w.E, w.zipf_s, 0)
    q = np.exp(b.astype(np.float64))
    assert abs(q.sum() - 1) < 1e-6
    qs = np.sort(q)[::-1]
    r = np.arange(1, w.E + 1)
    assert np.allclose(qs / qs[0], r ** -1.2, rtol=1e-5)
