"""The output head and one MTP draft/verify round against the oracle."""
import numpy as np
import pytest
import torch

import block_quantized_moe_layer_gb300 as pkg
from block_quantized_moe_layer_gb300 import synth
from block_quantized_moe_layer_gb300.workloads import synthetic_layer, synthetic_lm_head, synthetic_round
from oracle import accept as oacc
from oracle import formats, moe as omoe, mtp as omtp
from tests._oracle_layer import qtensor, synth_oracle_layer
from tests.gpu_util import to_np

pytestmark = pytest.mark.gpu

XDT = {pkg.ACT_BF16: torch.bfloat16, pkg.ACT_F32: torch.float32}
TOL = {pkg.ACT_BF16: 2e-2, pkg.ACT_F32: 1e-3}
# Router margin below which a layer's expert choice for a token may differ
# between the GPU chain and the fp64 oracle chain: the GPU's hidden state
# carries the rounding of every earlier layer (bf16: ~2^-8 relative per
# element), so its router logits differ from the oracle's by far more than
# within one layer.  A token whose top-k boundary margin is below this in any
# layer is reported and left out of the value comparisons (the per-layer
# near-tie rule, widened to the chain's input perturbation).
CHAIN_TIE = {pkg.ACT_BF16: 5e-2, pkg.ACT_F32: 1e-3}


def _oracle_lm(r):
    return qtensor(formats.FMT_Q8_0, synth.lm_weight(r, "cuda").cpu().numpy())


def _decided(o_row, err, rel=1e-3):
    """The oracle's argmax of a row cannot move under an error of `err` per logit."""
    s = np.sort(o_row)[::-1]
    return (s[0] - s[1]) > 2 * err + rel * np.abs(o_row).max()


@pytest.mark.parametrize("act", [pkg.ACT_BF16, pkg.ACT_F32], ids=["bf16", "f32"])
def test_lm_head_matches_oracle(act):
    r = synth.replace(synth.ROUNDS["tiny_round"], V=1001)
    lm = synthetic_lm_head(r, act, T_max=8)
    ol = _oracle_lm(r)
    try:
        for T in (1, 3, 4, 5, 8):
            x = synth.activations(r.layers[0], "cuda", T=T, variant=T).to(XDT[act])
            y = to_np(lm.forward(x))
            ref = omtp.lm_logits(to_np(x), ol)
            err = np.abs(y - ref).max() / np.abs(ref).max()
            assert err < 1e-3, f"T={T}: logits rel err {err:.2e}"
            for t in range(T):
                if _decided(ref[t], np.abs(y[t] - ref[t]).max()):
                    assert oacc.argmax_lowest(y[t]) == oacc.argmax_lowest(ref[t])
    finally:
        lm.close()


@pytest.mark.parametrize("act", [pkg.ACT_BF16, pkg.ACT_F32], ids=["bf16", "f32"])
def test_residual_forward(act):
    w = synth.with_T(synth.WORKLOADS["tiny"], 8)
    L, _ = synthetic_layer(w, act, T_max=8)
    try:
        ol = synth_oracle_layer(w, "cuda")
        x = synth.activations(w, "cuda", T=5).to(XDT[act])
        y = to_np(L.forward(x, residual=True))
        torch.cuda.synchronize()
        L.status()
        ref, _ = omoe.forward(to_np(x), ol)
        assert omoe.max_rel_err(y, to_np(x) + ref) <= TOL[act]
    finally:
        L.close()


def _check_round(r, act, report):
    layers, heads, lm = synthetic_round(r, act)
    try:
        x, noise = synth.round_inputs(r, "cuda")
        x = x.to(XDT[act])
        out = pkg.mtp_round(layers, heads, lm, x, noise)
        torch.cuda.synchronize()
        for L in layers + heads:
            L.status()
        logits, drafts = to_np(out["logits"]), out["drafts"].cpu().tolist()
        n_gpu, next_gpu = out["accept"].cpu().tolist()
        # acceptance is the greedy rule on the GPU's own drafts and logits (pure function: exact)
        n_self, next_self, amax_gpu = oacc.greedy_accept(drafts, logits)
        assert (n_gpu, next_gpu) == (n_self, next_self)
        # the oracle round on the same inputs
        ref = omtp.mtp_round(to_np(x), [synth_oracle_layer(w, "cuda") for w in r.layers],
                             [synth_oracle_layer(w, "cuda") for w in r.heads], _oracle_lm(r), to_np(noise))
        # rows whose routing in some target layer sits within the chain's perturbation
        T = r.k + 1
        chain = np.zeros(T, bool)
        for rt, w in zip(ref["target_routes"], r.layers):
            chain |= omoe.near_tie_tokens(rt["logits"], w.top_k, CHAIN_TIE[act])
        ok = ~chain
        assert ok.sum() >= 1, "every verify row has a routing near tie: nothing left to compare"
        lerr = np.abs(logits - ref["logits"]).max(axis=1)
        scale = np.abs(ref["logits"]).max()
        assert lerr[ok].max() / scale <= TOL[act], f"target logits rel err {lerr[ok].max() / scale:.2e}"
        hout = to_np(out["head_out"])
        head_ok = []
        for j in range(r.k):
            rows = ok[: j + 1] & ~omoe.near_tie_tokens(ref["head_routes"][j]["logits"], r.heads[j].top_k,
                                                        CHAIN_TIE[act])
            head_ok.append(rows)
            if rows.any():
                e = omoe.max_rel_err(hout[j, : j + 1][rows], ref["head_out"][j][rows])
                assert e <= TOL[act], f"head {j}: max rel err {e:.2e}"
        # drafts: the LM head on the noisy rows, checked where the decision is unique
        d_err = [np.abs(lm.forward(torch.from_numpy(ref["draft_rows"][j:j + 1]).to(XDT[act]).cuda())
                        .cpu().numpy()[0] - ref["draft_logits"][j]).max() for j in range(r.k)]
        near = [f"chain-row{i}" for i in range(T) if chain[i]]
        for j in range(r.k):
            if not ok[j]:
                near.append(f"draft{j}")
            elif _decided(ref["draft_logits"][j], 4 * max(d_err[j], lerr[ok].max())):
                assert drafts[j] == ref["drafts"][j], f"draft {j}"
            else:
                near.append(f"draft{j}")
        for i in range(r.k + 1):
            if ok[i] and _decided(ref["logits"][i], lerr[i]):
                assert amax_gpu[i] == ref["argmax"][i], f"target argmax row {i}"
            else:
                near.append(f"row{i}")
        rows = set(range(min(ref["n_accepted"], n_gpu) + 1))
        if not any(f"row{i}" in near or f"draft{i}" in near for i in rows):
            assert (n_gpu, next_gpu) == (ref["n_accepted"], ref["next_token"])
        report(f"{r.name} act={act}: n_accepted gpu {n_gpu} oracle {ref['n_accepted']}, next {next_gpu}/"
               f"{ref['next_token']}, logits rel err {lerr[ok].max() / scale:.2e} over {ok.sum()}/{T} rows, "
               f"near ties {near}")
    finally:
        for L in layers + heads:
            L.close()
        lm.close()


@pytest.mark.parametrize("act", [pkg.ACT_BF16, pkg.ACT_F32], ids=["bf16", "f32"])
def test_tiny_round(act):
    _check_round(synth.ROUNDS["tiny_round"], act, print)


def test_tiny_round_without_noise_accepts_all():
    r = synth.replace(synth.ROUNDS["tiny_round"], noise_std=0.0)
    layers, heads, lm = synthetic_round(r, pkg.ACT_F32)
    try:
        x, noise = synth.round_inputs(r, "cuda")
        out = pkg.mtp_round(layers, heads, lm, x.float(), noise)
        assert out["accept"].cpu().tolist()[0] == r.k
    finally:
        for L in layers + heads:
            L.close()
        lm.close()


def test_mtp_round_full_size_check_mode():
    _check_round(synth.ROUNDS["mtp_round"], pkg.ACT_F32, print)


def test_mtp_round_full_size_bf16():
    _check_round(synth.ROUNDS["mtp_round"], pkg.ACT_BF16, print)
