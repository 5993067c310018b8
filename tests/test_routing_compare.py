"""The routing comparison used by the GPU parity tests, checked on CPU with
planted mistakes."""
import numpy as np
import pytest

from tests.gpu_util import check_routing


def _r(logits, k):
    l = np.asarray(logits, np.float64)
    ids = np.argsort(-l, axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(l, ids, axis=1)
    g = np.exp(sel - sel[:, :1])
    return dict(logits=l, ids=ids, gates=g / g.sum(axis=1, keepdims=True))


def test_exact_match_passes():
    r = _r([[3.0, 1.0, 2.0, 0.0]], 2)
    assert check_routing(r["ids"].copy(), r["gates"].copy(), r, np.array([True])) == 0


def test_close_logits_may_swap_slots():
    r = _r([[1.0, 0.95012, 0.5, 0.95012 + 1e-7]], 3)
    ids = r["ids"].copy()
    gates = r["gates"].copy()
    ids[0, [1, 2]] = ids[0, [2, 1]]
    gates[0, [1, 2]] = gates[0, [2, 1]]
    assert check_routing(ids, gates, r, np.array([True])) == 1


def test_far_logits_must_keep_order():
    r = _r([[1.0, 0.9, 0.5, 0.0]], 3)
    ids = r["ids"].copy()
    ids[0, [1, 2]] = ids[0, [2, 1]]
    with pytest.raises(AssertionError, match="slot order"):
        check_routing(ids, r["gates"][:, [0, 2, 1]], r, np.array([True]))


def test_wrong_set_fails_and_excluded_token_is_skipped():
    r = _r([[1.0, 0.9, 0.5, 0.0], [0.0, 1.0, 2.0, 3.0]], 2)
    ids = r["ids"].copy()
    ids[1] = [0, 1]
    with pytest.raises(AssertionError, match="selected experts"):
        check_routing(ids, r["gates"], r, np.array([True, True]))
    check_routing(ids, r["gates"], r, np.array([True, False]))


def test_wrong_gate_fails():
    r = _r([[1.0, 0.9, 0.5, 0.0]], 2)
    g = r["gates"].copy()
    g[0, 1] *= 1.001
    with pytest.raises(AssertionError, match="gates"):
        check_routing(r["ids"].copy(), g, r, np.array([True]))
