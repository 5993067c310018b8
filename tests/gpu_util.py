"""Shared helpers of the GPU parity tests."""
import numpy as np
import torch

from oracle import moe as omoe


def to_np(t):
    return t.float().cpu().numpy()


def check_layer(layer, x, oracle_layer, k, E, tol, label=""):
    """Runs the CUDA layer on x and compares it with the oracle.

    Expert ids must match bit-exactly and gates closely, except on tokens
    whose k-th / (k+1)-th router logits are within 1e-4 (reported); the
    permutation must equal the oracle's permutation of the GPU's own ids;
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
    assert np.array_equal(ids[keep], r["ids"][keep]), f"{label}: expert ids differ"
    assert np.allclose(gates[keep], r["gates"][keep], rtol=2e-5, atol=1e-7), f"{label}: gates differ"
    o_off, o_perm, o_pos, _ = omoe.permutation(ids, E)
    assert np.array_equal(offs.astype(np.int64), o_off), f"{label}: offsets"
    assert np.array_equal(perm.astype(np.int64), o_perm), f"{label}: perm"
    yn = to_np(y)
    assert np.isfinite(yn).all()
    err = omoe.max_rel_err(yn[keep], y_ref[keep])
    assert err <= tol, f"{label}: max rel err {err:.3e} > {tol}"
    return err, int((~keep).sum()), r
