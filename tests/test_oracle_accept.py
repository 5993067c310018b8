"""Pins for greedy acceptance: the PR's worked example and the edge cases."""
import os

import numpy as np

from oracle.accept import greedy_accept, argmax_lowest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "accept_worked_example.txt")


def _read_golden():
    d = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        d[key] = [int(v) for v in vals]
    return d


def _logits_with_argmax(argmaxes, V, seed=0):
    rng = np.random.default_rng(seed)
    L = rng.normal(0, 1, (len(argmaxes), V)).astype(np.float32)
    for i, a in enumerate(argmaxes):
        L[i, a] = L[i].max() + 1.0
    return L


def test_pr_worked_example():
    g = _read_golden()
    L = _logits_with_argmax(g["argmax"], g["V"][0])
    n, nxt, a = greedy_accept(g["draft"], L)
    assert n == g["n_accepted"][0]
    assert nxt == g["next"][0]
    assert g["draft"][:n] + [nxt] == g["accepted"]
    # the hidden state handed to the next round is verify_h[n_accepted]
    assert n == g["pending_h_index"][0]


def test_all_accepted_takes_bonus_row():
    L = _logits_with_argmax([3, 1, 4, 15], 16)
    assert greedy_accept([3, 1, 4], L)[:2] == (3, 15)


def test_first_reject():
    L = _logits_with_argmax([2, 1, 4, 15], 16)
    assert greedy_accept([3, 1, 4], L)[:2] == (0, 2)


def test_later_match_after_mismatch_does_not_count():
    L = _logits_with_argmax([3, 9, 4, 15], 16)
    assert greedy_accept([3, 1, 4], L)[:2] == (1, 9)


def test_argmax_ties_lowest_id():
    row = np.array([0.0, 2.0, 1.0, 2.0, 2.0])
    assert argmax_lowest(row) == 1
    L = np.zeros((2, 6), np.float32)  # all ties: argmax 0 everywhere
    assert greedy_accept([0], L)[:2] == (1, 0)
    assert greedy_accept([5], L)[:2] == (0, 0)


def test_k_zero():
    L = _logits_with_argmax([7], 10)
    assert greedy_accept([], L)[:2] == (0, 7)
