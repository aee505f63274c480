"""Pins of the gating oracle (oracle/router.py) against facts that do not
come from the oracle itself: a pure-Python brute force with explicit tie
rules and math.exp, scipy's softmax for k = E, and the selection invariants."""
import math

import numpy as np
import pytest

from oracle import router as orr


def _brute(L, k, shared=None):
    """Per token: sort experts by (-logit, expert) in plain Python, softmax
    over the first k with math.exp and math.fsum."""
    ids, ws = [], []
    for row in L.tolist():
        sel = sorted(range(len(row)), key=lambda e: (-row[e], e))[:k]
        m = max(row[e] for e in sel)
        ex = [math.exp(row[e] - m) for e in sel]
        s = math.fsum(ex)
        w = [v / s for v in ex]
        if shared is not None:
            sel, w = sel + [shared], w + [1.0]
        ids.append(sel)
        ws.append(w)
    return np.array(ids, dtype=np.int32), np.array(ws)


@pytest.mark.parametrize("E,k", [(8, 1), (8, 3), (16, 6), (33, 7), (64, 16)])
def test_matches_brute_force_with_ties(E, k):
    g = np.random.default_rng(E * 100 + k)
    # a coarse grid makes many exact ties, including +0.0 vs -0.0
    L = (np.round(g.standard_normal((40, E)) * 2) / 2).astype(np.float32)
    L[0, :] = 0.0
    L[1, ::2] = -0.0
    ids, w = orr.router_topk(L, k)
    bi, bw = _brute(L, k)
    assert np.array_equal(ids, bi)
    np.testing.assert_allclose(w, bw, rtol=1e-13, atol=0)


def test_all_equal_logits_pick_lowest_experts_evenly():
    L = np.full((3, 10), 1.25, dtype=np.float32)
    ids, w = orr.router_topk(L, 4)
    assert (ids == np.arange(4)).all()
    np.testing.assert_allclose(w, 0.25, rtol=0, atol=1e-15)


def test_full_softmax_when_k_equals_E():
    scipy_special = pytest.importorskip("scipy.special")
    g = np.random.default_rng(3)
    L = g.standard_normal((20, 12)).astype(np.float32)
    ids, w = orr.router_topk(L, 12)
    ref = scipy_special.softmax(L.astype(np.float64), axis=1)
    np.testing.assert_allclose(np.take_along_axis(ref, ids.astype(np.int64), axis=1), w,
                               rtol=1e-12)


def test_selection_invariants():
    g = np.random.default_rng(7)
    L = g.standard_normal((200, 384)).astype(np.float32)
    k = 6
    ids, w = orr.router_topk(L, k)
    assert ids.shape == (200, k) and w.shape == (200, k)
    for t in range(200):
        assert len(set(ids[t].tolist())) == k
        chosen = L[t, ids[t]]
        rest = np.delete(L[t], ids[t])
        assert chosen.min() >= rest.max()
        assert (np.diff(chosen) <= 0).all()          # listed by descending logit
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert (np.diff(w, axis=1) <= 0).all()           # weights follow the logits


def test_shared_expert_column():
    g = np.random.default_rng(11)
    L = g.standard_normal((16, 384)).astype(np.float32)
    ids, w = orr.router_topk(L, 6, shared_id=384)
    bi, bw = _brute(L, 6, shared=384)
    assert np.array_equal(ids, bi)
    assert (ids[:, 6] == 384).all() and (w[:, 6] == 1.0).all()
    np.testing.assert_allclose(w[:, :6].sum(axis=1), 1.0, atol=1e-14)
    np.testing.assert_allclose(w, bw, rtol=1e-13)


def test_weights_are_shift_invariant():
    # softmax(L + c) = softmax(L) on the same selection (c exact in FP32)
    g = np.random.default_rng(5)
    L = np.round(g.standard_normal((30, 64)) * 64).astype(np.float32) / 64
    i0, w0 = orr.router_topk(L, 5)
    i1, w1 = orr.router_topk(L + np.float32(8.0), 5)
    assert np.array_equal(i0, i1)
    np.testing.assert_allclose(w0, w1, rtol=1e-13)


def test_rejects_bad_topk():
    with pytest.raises(ValueError):
        orr.router_topk(np.zeros((2, 4), np.float32), 5)


def test_shared_expert_pieces_take_consecutive_columns():
    L = np.random.default_rng(3).standard_normal((5, 12)).astype(np.float32)
    ids1, w1 = orr.router_topk(L, 3, shared_id=12)
    ids3, w3 = orr.router_topk(L, 3, shared_id=12, n_shared=3)
    assert np.array_equal(ids3[:, :4], ids1) and np.array_equal(w3[:, :4], w1)
    assert (ids3[:, 3:] == np.array([12, 13, 14])).all() and (w3[:, 3:] == 1.0).all()

