"""Pins for the oracle's MTP round: the output norm and LM head against closed
forms, the residual stack against special cases, and the round's acceptance
against properties that fix how drafts and target rows line up."""
import numpy as np

from oracle import formats, moe, mtp
from tests._oracle_layer import layer_from_fp32, qtensor

H, E, K, I, V = 64, 6, 2, 32, 50


def _layer(seed, zero=False):
    rng = np.random.default_rng(seed)
    s = 0.0 if zero else 0.05
    Wr = rng.normal(0, 0.3, (E, H)).astype(np.float32)
    ws = [tuple((rng.normal(0, 1, sh) * s).astype(np.float32) for sh in ((I, H), (I, H), (H, I))) for _ in range(E)]
    sh = tuple((rng.normal(0, 1, q) * s).astype(np.float32) for q in ((I, H), (I, H), (H, I)))
    return layer_from_fp32(H, E, K, I, I, Wr, None, lambda e: ws[e], sh, formats.FMT_Q8_0, formats.FMT_Q8_0)


def _lm(seed):
    rng = np.random.default_rng(seed)
    # w = 2^-7 q with |q| <= 127 and one 127 per block: Q8_0 holds it exactly
    q = rng.integers(-127, 128, (V, H)).astype(np.float32)
    q[:, ::32] = 127
    return qtensor(formats.FMT_Q8_0, q / 128.0), q / 128.0


def test_rmsnorm_closed_forms():
    v = np.array([[3.0, 4.0]])
    assert np.allclose(mtp.rmsnorm(v, eps=0.25), v / np.sqrt(12.5 + 0.25), rtol=1e-15)
    c = np.full((1, 16), -2.5)
    assert np.allclose(mtp.rmsnorm(c, eps=1e-6), -2.5 / np.sqrt(6.25 + 1e-6), rtol=1e-15)
    # rows are independent; the mean square of the output is ms / (ms + eps)
    rng = np.random.default_rng(0)
    x = rng.normal(size=(3, 40))
    y = mtp.rmsnorm(x, eps=1e-3)
    ms = np.mean(x * x, axis=1)
    assert np.allclose(np.mean(y * y, axis=1), ms / (ms + 1e-3), rtol=1e-13)
    assert np.allclose(mtp.rmsnorm(x[1:2], eps=1e-3), y[1:2], rtol=0, atol=0)


def test_lm_logits_unit_vector_picks_a_column():
    lm, w = _lm(1)
    s, h, eps = 3.0, 17, 1e-6
    x = np.zeros((1, H))
    x[0, h] = s
    want = w[:, h].astype(np.float64) * s / np.sqrt(s * s / H + eps)
    assert np.allclose(mtp.lm_logits(x, lm, eps)[0], want, rtol=1e-14, atol=0)


def test_target_stack_residual():
    rng = np.random.default_rng(2)
    x = rng.normal(size=(4, H)).astype(np.float32).astype(np.float64)
    zero = _layer(3, zero=True)
    assert np.array_equal(mtp.target_stack(x, [zero, zero]), x)  # zero experts: h stays x
    L = _layer(4)
    y, _ = moe.forward(mtp.rmsnorm(x), L)
    assert np.allclose(mtp.target_stack(x, [L]), x + y, rtol=0, atol=0)
    y2, _ = moe.forward(mtp.rmsnorm(x + y), L)
    assert np.allclose(mtp.target_stack(x, [L, L]), x + y + y2, rtol=0, atol=0)
    # the blocks see normalised inputs: scaling x by 4 (exact in binary, eps 0)
    # scales the skip path only
    y0, _ = moe.forward(mtp.rmsnorm(x, eps=0.0), L)
    assert np.allclose(mtp.target_stack(4.0 * x, [L], eps=0.0) - 4.0 * x, y0, rtol=1e-12, atol=1e-12)


def _round(noise_scale, k=3, seed=5):
    rng = np.random.default_rng(seed)
    layers = [_layer(10 + i) for i in range(2)]
    heads = [_layer(20 + j) for j in range(k)]
    lm, _ = _lm(6)
    x = rng.normal(size=(k + 1, H))
    noise = rng.normal(size=(k, k, H)) * noise_scale
    return mtp.mtp_round(x, layers, heads, lm, noise), x, layers, heads, lm, noise


def test_round_without_noise_accepts_every_draft():
    # drafts come from rows 0..k-1 of the target's hidden states: with no noise
    # draft j+1 is the target's argmax of row j, so every draft is accepted
    r, *_ = _round(0.0)
    assert r["drafts"] == r["argmax"][:3]
    assert r["n_accepted"] == 3 and r["next_token"] == r["argmax"][3]


def test_round_draft_rows_are_normalised():
    # scaling a row does not change rmsnorm (up to eps): noise = 0.5 * h_tgt
    r0, x, layers, heads, lm, _ = _round(0.0)
    k = 3
    noise = np.stack([0.5 * r0["h_tgt"][:k] for _ in range(k)])
    r = mtp.mtp_round(x, layers, heads, lm, noise)
    assert r["drafts"] == r0["drafts"] and r["n_accepted"] == 3


def test_round_head_outputs_and_acceptance():
    r, x, layers, heads, lm, noise = _round(3.0)
    for j in range(3):
        y, _ = moe.forward(mtp.rmsnorm(r["h_tgt"][: j + 1] + noise[j][: j + 1]), heads[j])
        assert np.allclose(r["head_out"][j], y, rtol=0, atol=0)
    # the acceptance is the greedy rule on the drafts and the target logits
    n = 0
    while n < 3 and r["drafts"][n] == r["argmax"][n]:
        n += 1
    assert r["n_accepted"] == n and r["next_token"] == r["argmax"][n]
