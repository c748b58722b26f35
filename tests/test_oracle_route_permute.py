"""Pins for the oracle's routing and counting-sort permute (CPU only)."""
import math

import numpy as np
import pytest

from oracle import moe as O


def _brute_topk(row, k):
    """Sort (−logit, index) tuples in Python and keep the first k."""
    order = sorted(range(len(row)), key=lambda e: (-float(row[e]), e))
    return order[:k]


@pytest.mark.parametrize("E,k", [(8, 2), (16, 4), (64, 8), (5, 5), (3, 1)])
def test_route_matches_brute_force_with_ties(E, k):
    rng = np.random.default_rng(E * 31 + k)
    # logits drawn from a small set so that ties are frequent; include -0.0 and +0.0
    pool = np.array([-1.5, -0.0, 0.0, 0.25, 0.25, 1.0, 2.0], dtype=np.float32)
    logits = pool[rng.integers(0, len(pool), (40, E))]
    logits = np.concatenate([logits, rng.standard_normal((40, E)).astype(np.float32)])
    idx, w = O.route_topk(logits, k)
    for t in range(logits.shape[0]):
        assert idx[t].tolist() == _brute_topk(logits[t], k), t


def test_route_weights_are_renormalised_softmax():
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((50, 32)).astype(np.float32) * 3
    idx, w = O.route_topk(logits, 6)
    assert np.all(w >= 0)
    assert np.allclose(w.astype(np.float64).sum(1), 1.0, atol=1e-6)
    for t in range(50):
        # full softmax over all E with math.fsum, then renormalise over the chosen k
        ex = [math.exp(float(v)) for v in logits[t]]
        z = math.fsum(ex)
        p = [v / z for v in ex]
        sel = [p[e] for e in idx[t]]
        ref = [s / math.fsum(sel) for s in sel]
        assert np.allclose(w[t], ref, rtol=1e-6, atol=0)
        assert np.all(np.diff(w[t]) <= 0)         # descending logits -> descending weights


def test_route_k1_weight_is_exactly_one():
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((20, 7)).astype(np.float32)
    idx, w = O.route_topk(logits, 1)
    assert np.all(w == 1.0)
    assert np.array_equal(idx[:, 0], np.argmax(logits, axis=1))


def test_permute_hand_example():
    idx = np.array([[2, 0], [0, 1], [2, 1]], dtype=np.int32)
    counts, offsets, perm, inv = O.permute(idx, 3)
    assert counts.tolist() == [2, 2, 2]
    assert offsets.tolist() == [0, 2, 4, 6]
    assert perm.tolist() == [1, 2, 3, 5, 0, 4]
    assert inv.tolist() == [4, 0, 1, 2, 5, 3]


def test_permute_dropped_pairs():
    idx = np.array([[1, -1], [-1, 0], [1, 0]], dtype=np.int32)
    counts, offsets, perm, inv = O.permute(idx, 3)
    assert counts.tolist() == [2, 2, 0]
    assert offsets.tolist() == [0, 2, 4, 4]
    assert perm.tolist() == [3, 5, 0, 4]
    assert inv.tolist() == [2, -1, -1, 0, 3, 1]


@pytest.mark.parametrize("T,E,k", [(1, 4, 1), (37, 8, 2), (64, 256, 8), (200, 5, 3)])
def test_permute_against_stable_argsort(T, E, k):
    rng = np.random.default_rng(T + E + k)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, perm, inv = O.permute(idx, E)
    flat = idx.reshape(-1)
    assert counts.sum() == T * k and offsets[-1] == T * k
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    ref = np.argsort(flat, kind="stable")        # library sort: stable by expert, then pair id
    assert np.array_equal(perm, ref)
    assert np.array_equal(np.sort(perm), np.arange(T * k))     # bijection
    assert np.array_equal(inv[perm], np.arange(T * k))
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)
        assert np.all(np.diff(seg // k) > 0)     # token-ascending: a token's k experts are distinct


# ---------------------------------------------------------------- routing variants
# Sigmoid scoring, softmax without renormalisation and raw scores (the MegaMoE
# test's topk of randn scores), pinned by closed forms and special cases.

def test_route_variants_select_the_same_experts():
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((30, 40)).astype(np.float32)
    ref, _ = O.route_topk(logits, 6)
    for scoring, renorm in [("softmax", False), ("sigmoid", True), ("sigmoid", False), ("raw", False)]:
        idx, _ = O.route_topk(logits, 6, scoring, renorm)
        assert np.array_equal(idx, ref), (scoring, renorm)
    for t in range(logits.shape[0]):
        assert ref[t].tolist() == _brute_topk(logits[t], 6)


def test_route_raw_weights_are_the_selected_logits():
    rng = np.random.default_rng(8)
    logits = rng.standard_normal((25, 12)).astype(np.float32)
    idx, w = O.route_topk(logits, 4, "raw", False)
    for t in range(logits.shape[0]):
        sel = _brute_topk(logits[t], 4)
        assert w[t].tolist() == [float(logits[t, e]) for e in sel]
    with pytest.raises(ValueError):
        O.route_topk(logits, 4, "raw", True)


def test_route_sigmoid_special_values():
    # sigmoid(0) = 1/2 exactly; sigmoid(ln 3) = 3/4; sigmoid(l) + sigmoid(-l) = 1
    l3 = np.float32(math.log(3.0))
    logits = np.array([[0.0, l3, -l3, 1.25, -1.25, -4.0]], dtype=np.float32)
    idx, w = O.route_topk(logits, 6, "sigmoid", False)
    got = dict(zip(idx[0].tolist(), w[0].astype(np.float64).tolist()))
    assert got[0] == 0.5
    assert abs(got[1] - 0.75) <= 1e-7
    assert abs(got[1] + got[2] - 1.0) <= 2 * 2.0 ** -24
    assert abs(got[3] + got[4] - 1.0) <= 2 * 2.0 ** -24
    assert 0.0 < got[5] < got[4] < got[0] < got[3]


def test_route_sigmoid_renormalised():
    rng = np.random.default_rng(9)
    logits = (rng.standard_normal((40, 20)) * 2).astype(np.float32)
    _, w = O.route_topk(logits, 5, "sigmoid", True)
    s = w.astype(np.float64).sum(axis=1)
    assert np.all(np.abs(s - 1.0) <= 5 * 2.0 ** -24)
    assert np.all(np.diff(w, axis=1) <= 0)              # descending with the logits
    _, w1 = O.route_topk(logits, 1, "sigmoid", True)
    assert np.all(w1 == 1.0)


def test_route_softmax_without_renormalisation():
    # all experts selected: the full softmax, which sums to one
    rng = np.random.default_rng(10)
    logits = rng.standard_normal((20, 9)).astype(np.float32)
    _, w = O.route_topk(logits, 9, "softmax", False)
    assert np.all(np.abs(w.astype(np.float64).sum(axis=1) - 1.0) <= 9 * 2.0 ** -24)
    # equal logits: every expert has probability 1/E
    _, w = O.route_topk(np.full((3, 16), 0.7, np.float32), 4, "softmax", False)
    assert np.all(w == np.float32(1.0 / 16))
    # two levels: m experts at a, E - m at b; p_a = 1 / (m + (E - m) e^(b - a))
    a, b, m, E = 1.5, -0.5, 3, 10
    row = np.array([[b] * (E - m) + [a] * m], dtype=np.float32)
    idx, w = O.route_topk(row, m + 1, "softmax", False)
    p_a = 1.0 / (m + (E - m) * math.exp(b - a))
    p_b = math.exp(b - a) * p_a
    assert idx[0].tolist() == [E - m, E - m + 1, E - m + 2, 0]
    assert np.allclose(w[0].astype(np.float64), [p_a] * m + [p_b], rtol=2.0 ** -23, atol=0)
    # a subset of the full softmax never sums above one
    _, w = O.route_topk(logits, 3, "softmax", False)
    assert np.all(w.astype(np.float64).sum(axis=1) < 1.0)
