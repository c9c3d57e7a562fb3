"""Pins for the oracle's router, softmax, top-k/renormalisation and
permutation: brute force on small inputs, a library softmax, closed-form
identities and the invariants of the permutation."""
import math

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

import oracle


def test_router_logits_scalar_loop():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 33))
    Wr = rng.standard_normal((7, 33))
    b = rng.standard_normal(7)
    l = oracle.router_logits(x, Wr, b)
    for t in range(5):
        for e in range(7):
            ref = math.fsum(x[t, h] * Wr[e, h] for h in range(33)) + b[e]
            assert abs(l[t, e] - ref) <= 1e-13 * (1 + abs(ref))
    assert np.array_equal(oracle.router_logits(x, Wr), x @ Wr.T)


def test_softmax_matches_library_and_sums_to_one():
    rng = np.random.default_rng(1)
    l = rng.standard_normal((64, 128)) * 3
    p = oracle.softmax(l)
    assert np.allclose(p, sp_softmax(l, axis=1), rtol=1e-14, atol=0)
    assert np.allclose(p.sum(1), 1.0, rtol=0, atol=1e-15)
    # Shift invariance and the huge-logit case stay finite.
    assert np.allclose(oracle.softmax(l + 1000.0), p, rtol=1e-13)


def _brute_topk(prow, k):
    order = sorted(range(len(prow)), key=lambda e: (-prow[e], e))[:k]
    sel = [prow[e] for e in order]
    s = math.fsum(sel)
    return order, [v / s for v in sel]


@pytest.mark.parametrize("E,k", [(16, 2), (128, 8), (512, 10), (5, 5), (3, 1)])
def test_topk_against_brute_force_sort(E, k):
    rng = np.random.default_rng(E * 100 + k)
    p = oracle.softmax(rng.standard_normal((40, E)))
    idx, w = oracle.topk_renorm(p, k)
    for t in range(40):
        o, ww = _brute_topk(list(p[t]), k)
        assert idx[t].tolist() == o
        assert np.allclose(w[t], ww, rtol=1e-15, atol=1e-16)
    assert np.allclose(w.sum(1), 1.0, rtol=0, atol=1e-15)


def test_topk_ties_go_to_lower_index():
    p = np.array([[0.1, 0.3, 0.3, 0.2, 0.3, 0.1],
                  [0.25, 0.25, 0.25, 0.25, 0.0, 0.0]])
    idx, w = oracle.topk_renorm(p, 3)
    assert idx.tolist() == [[1, 2, 4], [0, 1, 2]]
    assert np.allclose(w, [[1 / 3] * 3] * 2)


def test_renormalised_weights_equal_softmax_over_selected_logits():
    """w_j = p_j / sum(p_sel) = exp(l_j) / sum_sel exp(l): the normaliser of
    the full softmax cancels."""
    rng = np.random.default_rng(5)
    l = rng.standard_normal((50, 128))
    idx, w = oracle.topk_renorm(oracle.softmax(l), 8)
    sel = np.take_along_axis(l, idx.astype(np.int64), axis=1)
    assert np.allclose(w, sp_softmax(sel, axis=1), rtol=1e-13, atol=0)


def _brute_permute(idx, E):
    T, k = idx.shape
    off = [0]
    row_token = []
    tok_slot_row = [None] * (T * k)
    for e in range(E):
        for t in range(T):
            for j in range(k):
                if idx[t, j] == e:
                    tok_slot_row[t * k + j] = len(row_token)
                    row_token.append(t)
        off.append(len(row_token))
    return off, row_token, tok_slot_row


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (8, 16, 2), (7, 5, 3), (4, 4, 4)])
def test_permute_brute_force(T, E, k):
    rng = np.random.default_rng(T * 31 + E)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    off, rt, tsr = oracle.permute(idx, E)
    o2, rt2, tsr2 = _brute_permute(idx, E)
    assert off.tolist() == o2 and rt.tolist() == rt2 and tsr.tolist() == tsr2


@pytest.mark.parametrize("T,E,k", [(64, 128, 8), (1000, 512, 10), (333, 16, 2)])
def test_permute_invariants(T, E, k):
    rng = np.random.default_rng(T)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    off, rt, tsr = oracle.permute(idx, E)
    P = T * k
    assert off[0] == 0 and off[-1] == P and np.all(np.diff(off) >= 0)
    assert np.array_equal(np.diff(off), np.bincount(idx.ravel(), minlength=E))
    # Every token appears exactly k times.
    assert np.array_equal(np.bincount(rt, minlength=T), np.full(T, k))
    # tok_slot_row is a bijection onto the rows and points back to its token.
    assert np.array_equal(np.sort(tsr), np.arange(P))
    assert np.array_equal(rt[tsr], np.repeat(np.arange(T), k))
    # The row of pair (t, j) lies in expert idx[t, j]'s segment.
    e_of_row = np.repeat(np.arange(E), np.diff(off))
    assert np.array_equal(e_of_row[tsr], idx.ravel())
    # Tokens ascend inside every segment.
    for e in range(E):
        seg = rt[off[e]:off[e + 1]]
        assert np.all(np.diff(seg) > 0)


def test_permute_empty_and_single():
    off, rt, tsr = oracle.permute(np.zeros((0, 4), np.int32), 6)
    assert off.tolist() == [0] * 7 and rt.size == 0 and tsr.size == 0
    off, rt, tsr = oracle.permute(np.array([[3]], np.int32), 4)
    assert off.tolist() == [0, 0, 0, 0, 1] and rt.tolist() == [0] and tsr.tolist() == [0]
