"""Pins for the oracle's whole layer: dense special case, closed forms,
linearity and token independence."""
import math

import numpy as np
import pytest

from oracle import formats, moe
from tests._oracle_layer import expert_from_fp32, layer_from_fp32, qtensor


def _rand_layer(seed, H=64, E=6, k=2, I=32, I_sh=32, fmt=formats.FMT_Q8_0, bias=True):
    rng = np.random.default_rng(seed)
    Wr = rng.normal(0, 0.3, (E, H)).astype(np.float32)
    b = rng.normal(0, 0.5, E).astype(np.float32) if bias else None
    ws = [tuple(rng.normal(0, 0.05, s).astype(np.float32) for s in ((I, H), (I, H), (H, I)))
          for _ in range(E)]
    sh = tuple(rng.normal(0, 0.05, s).astype(np.float32) for s in ((I_sh, H), (I_sh, H), (H, I_sh)))
    return layer_from_fp32(H, E, k, I, I_sh, Wr, b, lambda e: ws[e], sh, fmt, formats.FMT_Q8_0), ws, sh


def _loop_ffn(x, G, U, D):
    """Straight-line SwiGLU FFN with Python loops (no matrix products)."""
    I, H = G.shape
    h = []
    for i in range(I):
        u = sum(float(G[i, c]) * float(x[c]) for c in range(H))
        v = sum(float(U[i, c]) * float(x[c]) for c in range(H))
        h.append(u / (1.0 + math.exp(-u)) * v)
    return [sum(float(D[r, i]) * h[i] for i in range(I)) for r in range(D.shape[0])]


def test_single_expert_top1_is_dense_swiglu_plus_shared():
    L, _, _ = _rand_layer(1, H=32, E=1, k=1, I=32, I_sh=32)
    rng = np.random.default_rng(2)
    x = rng.normal(size=(3, 32)).astype(np.float32)
    y, r = moe.forward(x, L)
    assert (r["ids"] == 0).all() and np.allclose(r["gates"], 1.0, rtol=0, atol=0)
    ex, sh = L.expert(0), L.shared
    for t in range(3):
        dense = _loop_ffn(x[t], ex.gate.dense(), ex.up.dense(), ex.down.dense())
        shared = _loop_ffn(x[t], sh.gate.dense(), sh.up.dense(), sh.down.dense())
        assert np.allclose(y[t], np.add(dense, shared), rtol=1e-12, atol=1e-15)


def test_unit_vector_selects_columns():
    rng = np.random.default_rng(3)
    G, U = rng.normal(0, 0.1, (32, 64)), rng.normal(0, 0.1, (32, 64))
    D = rng.normal(0, 0.1, (64, 32))
    ex = expert_from_fp32(formats.FMT_Q8_0, G, U, D)
    Gd, Ud, Dd = ex.gate.dense(), ex.up.dense(), ex.down.dense()
    for c in (0, 17, 63):
        x = np.zeros((1, 64))
        x[0, c] = 1.0
        u, v = Gd[:, c], Ud[:, c]
        want = Dd @ (u / (1 + np.exp(-u)) * v)
        assert np.allclose(moe.swiglu_expert(x, ex)[0], want, rtol=1e-14, atol=0)


def test_silu_values():
    u = np.array([0.0, 1.0, -1.0, 30.0, -800.0])
    want = [0.0, 1 / (1 + math.exp(-1)), -1 / (1 + math.e), 30 / (1 + math.exp(-30)), 0.0]
    assert np.allclose(moe.silu(u), want, rtol=1e-15, atol=0)


@pytest.mark.parametrize("fmt", [formats.FMT_Q8_0, formats.FMT_Q4KS])
def test_doubling_routed_down_doubles_routed_part(fmt):
    H, I = 256, 256
    L, ws, sh = _rand_layer(4, H=H, E=4, k=2, I=I, I_sh=32, fmt=fmt)
    x = np.random.default_rng(5).normal(size=(4, H)).astype(np.float32)
    y, r = moe.forward(x, L)
    y_sh = moe.swiglu_expert(x, L.shared)

    def doubled(e):
        ex = L.expert(e)
        blob = ex.down.data.copy()
        if fmt == formats.FMT_Q8_0:
            v = blob.reshape(H, -1, 34)
            d = np.ascontiguousarray(v[..., :2]).view("<f2") * np.float16(2)
            v[..., :2] = d.view(np.uint8)
        else:
            v = blob.reshape(H, -1, 144)
            for o in (0, 2):
                d = np.ascontiguousarray(v[..., o:o + 2]).view("<f2") * np.float16(2)
                v[..., o:o + 2] = d.view(np.uint8)
        return moe.Expert(ex.gate, ex.up, moe.QTensor(fmt, H, I, blob))
    L2 = moe.Layer(L.H, L.E, L.top_k, L.I, L.I_shared, L.router_w, L.router_b, doubled, L.shared)
    y2, _ = moe.forward(x, L2)
    assert np.allclose(y2 - y_sh, 2 * (y - y_sh), rtol=1e-12, atol=1e-14)


def test_tokens_are_independent_and_permute():
    L, _, _ = _rand_layer(6, H=64, E=8, k=3)
    x = np.random.default_rng(7).normal(size=(4, 64)).astype(np.float32)
    y, _ = moe.forward(x, L)
    for t in range(4):
        yt, _ = moe.forward(x[t:t + 1], L)
        assert np.allclose(yt[0], y[t], rtol=1e-13, atol=1e-15)
    order = [2, 0, 3, 1]
    yp, _ = moe.forward(x[order], L)
    assert np.allclose(yp, y[order], rtol=1e-13, atol=1e-15)


def test_combine_uses_gates_in_slot_order():
    L, _, _ = _rand_layer(8, H=64, E=5, k=3)
    x = np.random.default_rng(9).normal(size=(2, 64)).astype(np.float32)
    y, r = moe.forward(x, L)
    for t in range(2):
        want = moe.swiglu_expert(x[t:t + 1], L.shared)[0].copy()
        for j in range(3):
            want += r["gates"][t, j] * moe.swiglu_expert(x[t:t + 1], L.expert(int(r["ids"][t, j])))[0]
        assert np.allclose(y[t], want, rtol=1e-13, atol=1e-15)


def test_expert_shards_sum_to_the_layer():
    # shards covering every expert once, shared expert on one: their parts sum
    # to the layer's output; each part only holds its own experts' pairs
    L, ws, sh = _rand_layer(11, E=7, k=3)
    rng = np.random.default_rng(12)
    x = rng.normal(size=(5, 64)).astype(np.float32)
    y, r = moe.forward(x, L)
    for split in ([(0, 7)], [(0, 3), (3, 4)], [(0, 2), (2, 2), (4, 3)]):
        parts = [moe.forward_shard(x, L, b, n, i == 0)[0] for i, (b, n) in enumerate(split)]
        assert np.allclose(sum(parts), y, rtol=1e-12, atol=1e-14)
    # a shard's part by hand: the gates of its own pairs, and no shared expert
    part, _ = moe.forward_shard(x, L, 3, 4, False)
    want = np.zeros_like(part)
    for t in range(5):
        for j in range(3):
            e = int(r["ids"][t, j])
            if 3 <= e < 7:
                want[t] += r["gates"][t, j] * moe.swiglu_expert(x[t:t + 1], L.expert(e))[0]
    assert np.allclose(part, want, rtol=1e-13, atol=1e-15)
    # a shard none of whose experts is chosen, without the shared expert: zero
    unused = sorted(set(range(7)) - set(r["ids"][0].tolist()))
    z, _ = moe.forward_shard(x[:1], L, unused[0], 1, False)
    assert not z.any()
