"""Shared helpers of the GPU parity tests."""
import numpy as np
import torch

from oracle import moe as omoe


def to_np(t):
    return t.float().cpu().numpy()


def check_routing(ids, gates, r, keep, thr=1e-4, label=""):
    """GPU ids/gates [T, k] against the oracle routing ``r`` on tokens ``keep``.

    The selected set must match exactly.  The slot order (descending logit)
    must match wherever the oracle's selected logits are at least ``thr``
    apart; a run of selected experts whose logits are closer than that may
    come in either order (fp32 and fp64 can rank them differently), and is
    compared as a set.  Gates are compared per expert id.
    """
    T, k = ids.shape
    o_ids = r["ids"]
    ids = ids.astype(np.int64)
    assert np.array_equal(np.sort(ids[keep], axis=1), np.sort(o_ids[keep], axis=1)), \
        f"{label}: selected experts differ"
    lsel = np.take_along_axis(np.asarray(r["logits"], np.float64), o_ids, axis=1)
    close = np.zeros((T, k), bool)
    if k > 1:
        g = (lsel[:, :-1] - lsel[:, 1:]) < thr
        close[:, :-1] |= g
        close[:, 1:] |= g
    fixed = keep[:, None] & ~close
    assert np.array_equal(ids[fixed], o_ids[fixed]), f"{label}: slot order differs"
    og = np.take_along_axis(r["gates"], np.argsort(o_ids, axis=1), axis=1)
    gg = np.take_along_axis(np.asarray(gates, np.float64), np.argsort(ids, axis=1), axis=1)
    assert np.allclose(gg[keep], og[keep], rtol=2e-5, atol=1e-7), f"{label}: gates differ"
    return int((keep[:, None] & close).any(axis=1).sum())


def check_layer(layer, x, oracle_layer, k, E, tol, label=""):
    """Runs the CUDA layer on x and compares it with the oracle.

    Expert ids must match bit-exactly and gates closely (see check_routing),
    except on tokens whose k-th / (k+1)-th router logits are within 1e-4
    (reported); the permutation must equal the oracle's permutation of the
    GPU's own ids;
    outputs must be within ``tol`` max relative error per token row.
    Returns (max_rel_err, n_excluded, routing dict).
    """
    T = x.shape[0]
    y = layer.forward(x)
    torch.cuda.synchronize()
    layer.status()
    y_ref, r = omoe.forward(to_np(x), oracle_layer)
    keep = ~omoe.near_tie_tokens(r["logits"], k)
    ids, gates, offs, perm = (to_np(t) for t in layer.routing(T))
    ids = ids.astype(np.int64)
    check_routing(ids, gates, r, keep, label=label)
    o_off, o_perm, o_pos, _ = omoe.permutation(ids, E)
    assert np.array_equal(offs.astype(np.int64), o_off), f"{label}: offsets"
    assert np.array_equal(perm.astype(np.int64), o_perm), f"{label}: perm"
    yn = to_np(y)
    assert np.isfinite(yn).all()
    err = omoe.max_rel_err(yn[keep], y_ref[keep])
    assert err <= tol, f"{label}: max rel err {err:.3e} > {tol}"
    r["elementwise_err"] = omoe.max_rel_err_elementwise(yn[keep], y_ref[keep])
    print(f"{label}: max rel err {err:.3e} (element-wise, 1e-3 floor: {r['elementwise_err']:.3e}), "
          f"excluded {int((~keep).sum())} of {T} tokens")
    return err, int((~keep).sum()), r
