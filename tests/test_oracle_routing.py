"""Pins for the oracle's router, top-k, gates and permutation."""
import itertools

import numpy as np
import pytest

from oracle import moe


def _beats(p, a, b):
    """Total order of the selection: larger p first, lower index on ties."""
    return p[a] > p[b] or (p[a] == p[b] and a < b)


def _brute_topk(p, k):
    E = len(p)
    winners = []
    for S in itertools.combinations(range(E), k):
        rest = [i for i in range(E) if i not in S]
        if all(_beats(p, a, b) for a in S for b in rest):
            winners.append(S)
    assert len(winners) == 1
    S = list(winners[0])
    # slot order: bubble by the same total order
    for i in range(len(S)):
        for j in range(len(S) - 1 - i):
            if _beats(p, S[j + 1], S[j]):
                S[j], S[j + 1] = S[j + 1], S[j]
    return S


@pytest.mark.parametrize("E", range(1, 9))
def test_topk_matches_brute_force(E):
    rng = np.random.default_rng(E)
    for trial in range(30):
        if trial % 3 == 0:
            p = rng.integers(0, 3, E).astype(float)  # many exact ties
        else:
            p = rng.normal(size=E)
        for k in range(1, E + 1):
            got = moe.topk_rows(p[None, :], k)[0].tolist()
            assert got == _brute_topk(p, k)


def test_topk_ties_go_to_lower_index():
    p = np.array([[0.1, 0.3, 0.3, 0.3, 0.0]])
    assert moe.topk_rows(p, 2)[0].tolist() == [1, 2]


def test_gates_closed_form_and_sum():
    rng = np.random.default_rng(11)
    l = rng.normal(0, 2, (16, 352))
    p = moe.softmax_rows(l)
    ids = moe.topk_rows(p, 8)
    g = moe.gates_rows(p, ids)
    assert np.abs(g.sum(axis=1) - 1).max() <= 1e-14
    # renormalising the full softmax equals a softmax restricted to the top-k
    for t in range(16):
        sel = l[t, ids[t]]
        direct = np.array([1.0 / sum(np.exp(s - v) for s in sel) for v in sel])
        assert np.allclose(g[t], direct, rtol=1e-13, atol=0)
    # descending slot order
    assert (np.diff(g, axis=1) <= 0).all()


def test_router_bias_enters_before_softmax():
    # E = 2, k = 2: gates are exactly softmax(l + b)
    x = np.array([[1.0, 2.0]])
    Wr = np.array([[0.5, -0.25], [0.25, 0.125]])
    b = np.array([0.75, -1.5])
    l = moe.router_logits(x, Wr, b)
    assert np.allclose(l, [[0.75, -1.5 + 0.5]], rtol=0, atol=1e-15)
    # without the bias expert 1 wins; the bias flips the order
    assert moe.topk_rows(moe.softmax_rows(moe.router_logits(x, Wr)), 1)[0, 0] == 1
    assert moe.topk_rows(moe.softmax_rows(l), 1)[0, 0] == 0
    g = moe.gates_rows(moe.softmax_rows(l), moe.topk_rows(moe.softmax_rows(l), 2))
    e0, e1 = np.exp(0.75), np.exp(-1.0)
    assert np.allclose(g[0], [e0 / (e0 + e1), e1 / (e0 + e1)], rtol=1e-15)


def test_router_is_x_times_w_transposed():
    # unit vector x = e_h picks column h of Wr (catches a transposed operand)
    rng = np.random.default_rng(12)
    Wr = rng.normal(size=(5, 7))
    for h in range(7):
        x = np.zeros((1, 7))
        x[0, h] = 1
        assert np.array_equal(moe.router_logits(x, Wr)[0], Wr[:, h])


@pytest.mark.parametrize("T,E,k", [(4, 16, 2), (4, 352, 8), (7, 5, 5), (64, 32, 8)])
def test_permutation_invariants(T, E, k):
    rng = np.random.default_rng(T * 1000 + E)
    p = moe.softmax_rows(rng.normal(size=(T, E)))
    ids = moe.topk_rows(p, k)
    off, perm, pos, act = moe.permutation(ids, E)
    assert off[0] == 0 and off[E] == T * k
    assert sorted(perm.tolist()) == list(range(T * k))
    flat = ids.reshape(-1)
    for e in range(E):
        seg = perm[off[e]:off[e + 1]]
        assert (flat[seg] == e).all()
        assert (np.diff(seg) > 0).all()
        assert (off[e + 1] > off[e]) == (e in act)
    for t in range(T):
        for j in range(k):
            assert perm[pos[t, j]] == t * k + j
    assert list(act) == sorted(set(flat.tolist()))


def test_near_tie_rule():
    l = np.array([[3.0, 2.0, 1.0, 1.00005], [3.0, 2.0, 1.0, 0.5]])
    assert moe.near_tie_tokens(l, 3).tolist() == [True, False]


def test_max_rel_err_is_per_row_then_max():
    # row 0: max |diff| 0.5 over max |y*| 10 -> 0.05; row 1: 0.3 / 1 -> 0.3
    y_ref = np.array([[10.0, -2.0, 0.0], [1.0, 0.5, -1.0]])
    y = y_ref + np.array([[0.5, -0.1, 0.0], [0.0, 0.3, 0.0]])
    assert moe.max_rel_err(y, y_ref) == pytest.approx(0.3, rel=1e-15)
    # a row's error is relative to that row's own scale, not the tensor's
    assert moe.max_rel_err(y[:1], y_ref[:1]) == pytest.approx(0.05, rel=1e-15)
    assert moe.max_rel_err(np.zeros((0, 3)), np.zeros((0, 3))) == 0.0


def test_max_rel_err_elementwise_floor():
    # element-wise ratios against max(|y*|, 1e-3 * row max):
    #   row 0: 0.1/10 = 0.01; 0.02/2 = 0.01; 1e-6 against the floor 1e-2 -> 1e-4
    #   row 1: 0.5 / 0.5 = 1.0 (the largest)
    y_ref = np.array([[10.0, -2.0, 0.0], [1.0, 0.5, -1.0]])
    y = y_ref + np.array([[0.1, -0.02, 1e-6], [0.0, 0.5, 0.0]])
    assert moe.max_rel_err_elementwise(y, y_ref) == pytest.approx(1.0, rel=1e-12)
    assert moe.max_rel_err_elementwise(y[:1], y_ref[:1]) == pytest.approx(0.01, rel=1e-12)
    # a near-zero reference element is measured against the row's floor, not itself
    y_ref = np.array([[1.0, 1e-9]])
    y = np.array([[1.0, 1e-9 + 5e-4]])
    assert moe.max_rel_err_elementwise(y, y_ref) == pytest.approx(0.5, rel=1e-9)
    assert moe.max_rel_err_elementwise(y, y_ref, floor=1e-2) == pytest.approx(0.05, rel=1e-9)
    # never below the row-max metric
    assert moe.max_rel_err_elementwise(y, y_ref) >= moe.max_rel_err(y, y_ref)
