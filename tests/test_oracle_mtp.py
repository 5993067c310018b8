"""Pins for the oracle's MTP round: the output norm and LM head against closed
forms, the residual stack against special cases, and the round's acceptance
against properties that fix how drafts and target rows line up."""
import numpy as np
import pytest

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


def test_draft_probability_closed_forms():
    # two tokens with logits 0 and -ln 3: p = 1 / (1 + 1/3) = 3/4
    assert mtp.draft_probability([0.0, -np.log(3.0)]) == pytest.approx(0.75, rel=1e-15)
    # a uniform row: 1 / V, whatever the common value
    assert mtp.draft_probability(np.full(40, 7.5)) == pytest.approx(1 / 40, rel=1e-15)
    # shift invariance, and the probability of the argmax, not of index 0
    row = np.array([0.3, 2.0, -1.0, 1.5])
    p = np.exp(row) / np.exp(row).sum()
    assert mtp.draft_probability(row) == pytest.approx(p.max(), rel=1e-14)
    assert mtp.draft_probability(row + 100.0) == pytest.approx(p.max(), rel=1e-13)


def test_cut_drafts_is_a_prefix_rule():
    d, pr = [11, 22, 33], [0.9, 0.5, 0.95]
    assert mtp.cut_drafts(d, pr, 0.0) == ([11, 22, 33], 3)
    assert mtp.cut_drafts(d, pr, 0.5) == ([11, 22, 33], 3)   # p >= p_min is kept
    assert mtp.cut_drafts(d, pr, 0.6) == ([11], 1)           # a later confident draft is cut too
    assert mtp.cut_drafts(d, pr, 0.95) == ([], 0)
    assert mtp.cut_drafts([], [], 0.7) == ([], 0)


def test_round_p_min_zero_changes_nothing_and_one_drafts_nothing():
    r, x, layers, heads, lm, noise = _round(3.0)
    r0 = mtp.mtp_round(x, layers, heads, lm, noise, p_min=0.0)
    assert r0["drafts"] == r["drafts"] and r0["n_drafted"] == 3
    assert (r0["n_accepted"], r0["next_token"]) == (r["n_accepted"], r["next_token"])
    # p <= 1 always and < 1 for a row of finite logits over V > 1 tokens
    r1 = mtp.mtp_round(x, layers, heads, lm, noise, p_min=1.0)
    assert r1["n_drafted"] == 0 and r1["drafts"] == [-1, -1, -1]
    assert r1["n_accepted"] == 0 and r1["next_token"] == r["argmax"][0]


def test_round_p_min_just_above_and_below_a_draft():
    # no noise: every draft matches the target, so the accepted count equals
    # the number of drafts the cut keeps
    r, x, layers, heads, lm, noise = _round(0.0)
    probs = r["draft_probs"]
    assert r["n_accepted"] == 3
    j = int(np.argmin(probs))  # the least confident draft decides the cut
    below = mtp.mtp_round(x, layers, heads, lm, noise, p_min=probs[j] * (1 - 1e-9))
    above = mtp.mtp_round(x, layers, heads, lm, noise, p_min=probs[j] * (1 + 1e-9))
    assert below["n_drafted"] == 3 and below["n_accepted"] == 3
    want = min(i for i in range(3) if probs[i] < probs[j] * (1 + 1e-9))
    assert above["n_drafted"] == want == above["n_accepted"]
    assert above["drafts"][:want] == r["drafts"][:want] and above["drafts"][want:] == [-1] * (3 - want)
    # the next token is the target's argmax at the first row past the kept drafts
    assert above["next_token"] == r["argmax"][want]


def test_round_bf16_is_nearest_even():
    import torch
    # 8 significant bits: halfway cases go to the even neighbour
    assert mtp.round_bf16(1.0 + 2.0 ** -8) == 1.0
    assert mtp.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert mtp.round_bf16(-(1.0 + 2.0 ** -8 + 2.0 ** -30)) == -(1.0 + 2.0 ** -7)
    assert mtp.round_bf16(0.0) == 0.0 and mtp.round_bf16(3.0) == 3.0
    # on fp32 values it agrees with torch's fp32 -> bf16 conversion (RNE)
    rng = np.random.default_rng(3)
    v = (rng.normal(size=20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    want = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(mtp.round_bf16(v.astype(np.float64)), want)


def test_round_bf16_mode_rounds_the_layer_inputs():
    r, x, layers, heads, lm, noise = _round(3.0)
    rb = mtp.mtp_round(x, layers, heads, lm, noise, act="bf16")
    # by hand: each layer sees a bf16 input; outputs keep full precision
    h = np.asarray(x, np.float64)
    for L in layers:
        y, _ = moe.forward(mtp.round_bf16(mtp.rmsnorm(h)), L)
        h = h + y
    assert np.array_equal(rb["h_tgt"], h)
    for j in range(3):
        y, _ = moe.forward(mtp.round_bf16(mtp.rmsnorm(h[: j + 1] + noise[j][: j + 1])), heads[j])
        assert np.array_equal(rb["head_out"][j], y)
    # and the f64 mode is the unrounded round
    assert np.array_equal(mtp.mtp_round(x, layers, heads, lm, noise, act="f64")["h_tgt"], r["h_tgt"])
