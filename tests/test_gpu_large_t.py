"""Parity of the prefill-sized (T > 8) tensor-core path with the oracle.

Small layers and the 352-expert layer at T = 1024 are compared in full:
every token's routing and output."""
import numpy as np
import pytest
import torch

import block_quantized_moe_layer_gb300 as pkg
from block_quantized_moe_layer_gb300 import synth
from block_quantized_moe_layer_gb300.workloads import synthetic_layer
from oracle import moe as omoe
from tests._oracle_layer import synth_oracle_layer
from tests.gpu_util import check_layer, check_routing, to_np

pytestmark = pytest.mark.gpu

TOL = 2e-2

# several router row tiles are not needed here: E_pad = 128
LT_Q8 = synth.Workload("lt_q8", 31, T=300, H=512, E=40, top_k=3, I=256, I_shared=256, bias_std=0.5)
LT_Q4 = synth.Workload("lt_q4", 32, T=300, H=512, E=40, top_k=3, I=256, I_shared=256, bias_std=0.5,
                       routed_fmt=synth.FMT_Q4KS)
# few experts, many tokens each: experts span several 128-token tiles
LT_SKEW = synth.Workload("lt_skew", 33, T=700, H=256, E=8, top_k=2, I=128, I_shared=128, bias_std=1.0)
# E above 128 (two router row tiles), no shared expert
LT_NOSH = synth.Workload("lt_nosh", 34, T=160, H=256, E=150, top_k=4, I=192, I_shared=0, bias_std=0.5)


def _layer(w, T_max):
    L, _ = synthetic_layer(w, pkg.ACT_BF16, T_max=T_max)
    return L


@pytest.fixture(scope="module")
def lt_q8():
    L = _layer(LT_Q8, 300)
    yield LT_Q8, L, synth_oracle_layer(LT_Q8, "cuda")
    L.close()


@pytest.mark.parametrize("T", [9, 16, 37, 128, 129, 300])
def test_lt_q8_parity(lt_q8, T):
    w, L, ol = lt_q8
    x = synth.activations(w, "cuda", T=T)
    err, excl, _ = check_layer(L, x, ol, w.top_k, w.E, TOL, f"lt_q8 T={T}")
    print(f"lt_q8 T={T}: max rel err {err:.3e}, excluded {excl}")


def test_lt_q8_small_and_large_T_interleaved(lt_q8):
    w, L, ol = lt_q8
    for T in (4, 200, 8, 9, 1):
        x = synth.activations(w, "cuda", T=T, variant=T)
        check_layer(L, x, ol, w.top_k, w.E, TOL, f"lt_q8 interleaved T={T}")


def test_lt_q8_deterministic_and_graph(lt_q8):
    w, L, _ = lt_q8
    x = synth.activations(w, "cuda", T=250)
    y1 = L.forward(x).clone()
    y2 = L.forward(x).clone()
    assert torch.equal(y1, y2)
    s = torch.cuda.Stream()
    y3 = torch.empty_like(x)
    with torch.cuda.stream(s):
        L.forward(x, y3, stream=s)  # warm up on the capture stream
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            L.forward(x, y3, stream=s)
    y3.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y1, y3)
    L.status()


@pytest.mark.parametrize("T", [9, 64, 300])
def test_lt_q4_parity(T):
    L = _layer(LT_Q4, 300)
    try:
        x = synth.activations(LT_Q4, "cuda", T=T)
        err, excl, _ = check_layer(L, x, synth_oracle_layer(LT_Q4, "cuda"), LT_Q4.top_k, LT_Q4.E, TOL,
                                   f"lt_q4 T={T}")
        print(f"lt_q4 T={T}: max rel err {err:.3e}, excluded {excl}")
    finally:
        L.close()


def test_lt_skewed_multi_tile_experts():
    L = _layer(LT_SKEW, 700)
    try:
        x = synth.activations(LT_SKEW, "cuda", T=700)
        err, excl, r = check_layer(L, x, synth_oracle_layer(LT_SKEW, "cuda"), LT_SKEW.top_k, LT_SKEW.E, TOL,
                                   "lt_skew")
        counts = np.diff(r["offsets"])
        assert counts.max() > 128, "the case should put more than one token tile on an expert"
        print(f"lt_skew: max rel err {err:.3e}, tokens per expert {counts.tolist()}")
    finally:
        L.close()


def test_lt_no_shared_two_router_tiles():
    L = _layer(LT_NOSH, 160)
    try:
        x = synth.activations(LT_NOSH, "cuda", T=160)
        check_layer(L, x, synth_oracle_layer(LT_NOSH, "cuda"), LT_NOSH.top_k, LT_NOSH.E, TOL, "lt_nosh")
    finally:
        L.close()


def test_lt_create_rejects_check_mode_and_odd_I():
    with pytest.raises(pkg.MoEError):
        synthetic_layer(LT_Q8, pkg.ACT_F32, T_max=16)
    odd = synth.Workload("lt_odd", 35, T=16, H=256, E=8, top_k=2, I=96, I_shared=96)
    with pytest.raises(pkg.MoEError):
        synthetic_layer(odd, pkg.ACT_BF16, T_max=16)
    L, _ = synthetic_layer(odd, pkg.ACT_BF16, T_max=8)  # the T <= 8 path takes I % 32 == 0
    L.close()


@pytest.fixture(scope="module")
def prefill():
    w = synth.WORKLOADS["prefill_q8"]
    L = _layer(w, w.T)
    yield w, L, synth_oracle_layer(w, "cuda")
    L.close()


def test_prefill_q8_full_size_every_token(prefill):
    """All 1024 tokens' routing and outputs against the oracle (its experts
    evaluated in worker processes); tokens within the near-tie rule are
    excluded and reported.  Every tile position of the grouped GEMMs is
    covered: every expert's tokens, in every 64-token tile, with every
    partial last tile."""
    from tests._oracle_pool import OraclePool
    w, L, ol = prefill
    x = synth.activations(w, "cuda")
    T = x.shape[0]
    y = to_np(L.forward(x))
    torch.cuda.synchronize()
    L.status()
    xn = to_np(x)
    r = omoe.route(xn, ol)
    keep = ~omoe.near_tie_tokens(r["logits"], w.top_k)
    ids, gates, offs, perm = (to_np(t) for t in L.routing(T))
    ids = ids.astype(np.int64)
    n_close = check_routing(ids, gates, r, keep, label="prefill_q8")
    o_off, o_perm, _, _ = omoe.permutation(ids, w.E)
    assert np.array_equal(offs.astype(np.int64), o_off)
    assert np.array_equal(perm.astype(np.int64), o_perm)
    counts = np.diff(o_off)
    with OraclePool() as pool:
        y_ref, _ = pool.forward(xn, ol, w, routing=r)
    assert np.isfinite(y).all()
    err = omoe.max_rel_err(y[keep], y_ref[keep])
    ew = omoe.max_rel_err_elementwise(y[keep], y_ref[keep])
    # the worst token, and the worst token of each expert-load class
    row_err = np.abs(y - y_ref).max(axis=1) / np.abs(y_ref).max(axis=1)
    assert err <= TOL, f"prefill max rel err {err:.3e} (token {int(np.argmax(np.where(keep, row_err, 0)))})"
    print(f"prefill_q8: {keep.sum()} of {T} tokens compared (excluded {(~keep).sum()}), close selected pairs "
          f"{n_close}, max tokens/expert {counts.max()}, max rel err {err:.3e}, element-wise {ew:.3e}")
