"""Plain fp64 MoE FFN layer: router, top-k gates, permutation, SwiGLU experts,
shared expert and combine.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The layer (pages: "Step-5 Preview GGUF", "Model background" table -- sparse
MoE with 352 routed experts, 8 selected per token, hidden 4096 -- and
"Precision distribution" table -- routed gate/up/down, shared-expert gate/up/
down, F32 routers; "Step 3.7 Flash Mixed-Quant GGUF", "Tensor recipe").
The pages name the tensors but print no formula; the readings used here:

  router      l[t, e] = sum_h x[t, h] * Wr[e, h] + b[e]        (bias before softmax)
  gates       p = softmax(l[t, :]) over all E experts; the k largest p (ties to
              the lower expert index) in descending order; g = p_sel / sum p_sel
  experts     h = silu(Wg x) * (Wu x), silu(u) = u / (1 + exp(-u)); z = Wd h
  combine     y[t] = sum_{j=0}^{k-1} g[t, j] * z_e(t,j)(x_t) + shared(x_t)
              (the shared expert has weight 1)
  permutation pairs p = t*k + j stably sorted by expert: offsets[E+1] from the
              histogram, perm[] the sorted pair ids, pos[t, j] the inverse.

Weights are decoded with :mod:`oracle.formats` to fp32, then widened to fp64;
x (bf16 values) is widened exactly.  All sums are fp64 matrix products.
"""

from dataclasses import dataclass
from typing import Callable, Optional

import numpy as np

from . import formats

F64 = np.float64


@dataclass
class QTensor:
    """A serialised weight matrix [rows, cols]; blocks run along cols."""
    fmt: int
    rows: int
    cols: int
    data: np.ndarray  # uint8 [rows, row_bytes]

    def dense(self):
        return formats.dequantize(self.fmt, self.data, self.rows, self.cols).astype(F64)


@dataclass
class Expert:
    gate: QTensor  # [I, H]
    up: QTensor    # [I, H]
    down: QTensor  # [H, I]


@dataclass
class Layer:
    H: int
    E: int
    top_k: int
    I: int
    I_shared: int
    router_w: np.ndarray            # fp32 [E, H]
    router_b: Optional[np.ndarray]  # fp32 [E] or None
    expert: Callable[[int], Expert]  # e -> Expert (may build lazily)
    shared: Optional[Expert]


def router_logits(x, Wr, b=None):
    """l = x Wr^T + b in fp64.  x [T, H], Wr [E, H], b [E] -> [T, E]."""
    l = np.asarray(x, F64) @ np.asarray(Wr, F64).T
    if b is not None:
        l = l + np.asarray(b, F64)[None, :]
    return l


def softmax_rows(l):
    l = np.asarray(l, F64)
    e = np.exp(l - l.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def topk_rows(p, k):
    """Per row, the k experts with the largest p; ties go to the lower index.

    Returns int64 [T, k] in slot order: descending p, ascending index on ties.
    """
    p = np.asarray(p, F64)
    T, E = p.shape
    ids = np.empty((T, k), np.int64)
    idx = np.arange(E)
    for t in range(T):
        order = np.lexsort((idx, -p[t]))  # primary -p ascending, then index
        ids[t] = order[:k]
    return ids


def gates_rows(p, ids):
    sel = np.take_along_axis(np.asarray(p, F64), ids, axis=1)
    return sel / sel.sum(axis=1, keepdims=True)


def permutation(ids, E):
    """Stable grouping of the T*k (token, slot) pairs by expert.

    Returns offsets int64 [E+1], perm int64 [T*k] (pair ids p = t*k + j in
    (expert, p) order), pos int64 [T, k] with perm[pos[t, j]] = t*k + j, and
    the ascending list of active experts.
    """
    ids = np.asarray(ids, np.int64)
    T, k = ids.shape
    flat = ids.reshape(-1)
    counts = np.bincount(flat, minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    perm = np.argsort(flat, kind="stable").astype(np.int64)
    pos = np.empty(T * k, np.int64)
    pos[perm] = np.arange(T * k)
    act = np.nonzero(counts)[0].astype(np.int64)
    return offsets, perm, pos.reshape(T, k), act


def silu(u):
    with np.errstate(over="ignore"):
        return u / (1.0 + np.exp(-u))


def swiglu_expert(xr, ex: Expert):
    """xr [M, K] fp64 -> z [M, H_out] fp64 for one expert."""
    xr = np.asarray(xr, F64)
    u = xr @ ex.gate.dense().T
    v = xr @ ex.up.dense().T
    h = silu(u) * v
    return h @ ex.down.dense().T


def route(x, layer: Layer):
    """Router, softmax, top-k, gates and permutation for x [T, H]."""
    l = router_logits(x, layer.router_w, layer.router_b)
    p = softmax_rows(l)
    ids = topk_rows(p, layer.top_k)
    g = gates_rows(p, ids)
    offsets, perm, pos, act = permutation(ids, layer.E)
    return dict(logits=l, p=p, ids=ids, gates=g, offsets=offsets, perm=perm,
                pos=pos, act=act)


def forward(x, layer: Layer, routing=None, expert_fn=None):
    """y [T, H] fp64 and the routing dict for x [T, H].

    ``expert_fn(e, xr)``, if given, stands in for ``swiglu_expert(xr,
    layer.expert(e))`` (the same computation evaluated elsewhere, e.g. by
    worker processes holding the same weights)."""
    x = np.asarray(x, F64)
    T = x.shape[0]
    r = route(x, layer) if routing is None else routing
    k = layer.top_k
    if expert_fn is None:
        def expert_fn(e, xr):
            return swiglu_expert(xr, layer.expert(e))
    z = np.zeros((T, k, layer.H), F64)
    for e in r["act"]:
        e = int(e)
        sl = r["perm"][r["offsets"][e]:r["offsets"][e + 1]]
        toks, slots = sl // k, sl % k
        z[toks, slots] = expert_fn(e, x[toks])
    y = np.zeros((T, layer.H), F64)
    for j in range(k):
        y += r["gates"][:, j:j + 1] * z[:, j]
    if layer.shared is not None:
        y += swiglu_expert(x, layer.shared)
    r["z"] = z
    return y, r


def near_tie_tokens(logits, k, thr=1e-4):
    """Tokens whose k-th and (k+1)-th largest router logits differ by < thr.

    Their expert choice may legitimately differ between implementations that
    round differently, so ids / permutation / output comparisons skip them.
    """
    l = np.sort(np.asarray(logits, F64), axis=1)[:, ::-1]
    if l.shape[1] <= k:
        return np.zeros(l.shape[0], bool)
    return (l[:, k - 1] - l[:, k]) < thr


def max_rel_err(y, y_ref):
    """Per token row max_h |y - y*| / max_h |y*|; returns the max over rows."""
    y = np.asarray(y, F64)
    y_ref = np.asarray(y_ref, F64)
    den = np.maximum(np.abs(y_ref).max(axis=1), 1e-30)
    return float((np.abs(y - y_ref).max(axis=1) / den).max()) if y.size else 0.0


def max_rel_err_elementwise(y, y_ref, floor=1e-3):
    """Element-wise relative error, the second figure of the "max relative
    error" reading: |y - y*| / max(|y*|, floor * max_h |y*|) per element (the
    floor is taken per token row, so near-zero outputs do not dominate);
    returns the max over all elements."""
    y = np.asarray(y, F64)
    y_ref = np.asarray(y_ref, F64)
    if not y.size:
        return 0.0
    den = np.maximum(np.abs(y_ref), floor * np.abs(y_ref).max(axis=1, keepdims=True))
    den = np.maximum(den, 1e-30)
    return float((np.abs(y - y_ref) / den).max())


def forward_shard(x, layer: Layer, begin, count, with_shared, routing=None):
    """The part of y that one expert-parallel shard computes: the routing over
    all E experts is the layer's, but only pairs whose expert lies in
    [begin, begin + count) contribute (with their full gates), plus the shared
    expert if the shard holds it.  Summed over shards that cover every expert
    once with the shared expert on one of them, this is forward(x)."""
    x = np.asarray(x, F64)
    T = x.shape[0]
    r = route(x, layer) if routing is None else routing
    k = layer.top_k
    y = np.zeros((T, layer.H), F64)
    for e in r["act"]:
        e = int(e)
        if not begin <= e < begin + count:
            continue
        sl = r["perm"][r["offsets"][e]:r["offsets"][e + 1]]
        toks, slots = sl // k, sl % k
        z = swiglu_expert(x[toks], layer.expert(e))
        y[toks] += r["gates"][toks, slots][:, None] * z
    if with_shared and layer.shared is not None:
        y += swiglu_expert(x, layer.shared)
    return y, r
