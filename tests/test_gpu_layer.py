"""Parity of the CUDA MoE layer (T <= 8 path) with the oracle."""
import numpy as np
import pytest
import torch

import block_quantized_moe_layer_gb300 as pkg
from block_quantized_moe_layer_gb300 import synth
from block_quantized_moe_layer_gb300.workloads import synthetic_layer
from oracle import moe as omoe
from tests._oracle_layer import synth_oracle_layer
from tests.gpu_util import check_layer, to_np

pytestmark = pytest.mark.gpu

TOL = {pkg.ACT_BF16: 2e-2, pkg.ACT_F32: 1e-3}
XDT = {pkg.ACT_BF16: torch.bfloat16, pkg.ACT_F32: torch.float32}

# a small layer with the 4-bit routed format, E not a multiple of 32, k = 3
SMALL_Q4 = synth.Workload("small_q4", 21, T=8, H=512, E=40, top_k=3, I=256, I_shared=256,
                          bias_std=0.5, routed_fmt=synth.FMT_Q4KS)


@pytest.fixture(scope="module", params=[pkg.ACT_BF16, pkg.ACT_F32], ids=["bf16", "f32"])
def tiny(request):
    w = synth.with_T(synth.WORKLOADS["tiny"], 8)
    L, _ = synthetic_layer(w, request.param, T_max=8)
    yield w, L, synth_oracle_layer(w, "cuda"), request.param
    L.close()


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8])
def test_tiny_parity(tiny, T):
    w, L, ol, act = tiny
    x = synth.activations(w, "cuda", T=T).to(XDT[act])
    check_layer(L, x, ol, w.top_k, w.E, TOL[act], f"tiny T={T}")


def test_tiny_T0_and_bounds(tiny):
    w, L, ol, act = tiny
    x = torch.zeros(0, w.H, dtype=XDT[act], device="cuda")
    assert L.forward(x).shape == (0, w.H)
    with pytest.raises(pkg.MoEError):
        L.forward(torch.zeros(9, w.H, dtype=XDT[act], device="cuda"))


@pytest.fixture(scope="module", params=[pkg.ACT_BF16, pkg.ACT_F32], ids=["bf16", "f32"])
def small_q4(request):
    L, _ = synthetic_layer(SMALL_Q4, request.param, T_max=8)
    yield SMALL_Q4, L, synth_oracle_layer(SMALL_Q4, "cuda"), request.param
    L.close()


@pytest.mark.parametrize("T", [1, 4, 7, 8])
def test_small_q4_parity(small_q4, T):
    w, L, ol, act = small_q4
    x = synth.activations(w, "cuda", T=T).to(XDT[act])
    check_layer(L, x, ol, w.top_k, w.E, TOL[act], f"small_q4 T={T}")


@pytest.fixture(scope="module")
def verify_q8():
    w = synth.WORKLOADS["verify_q8"]
    L, _ = synthetic_layer(w, pkg.ACT_BF16, T_max=8)
    yield w, L, synth_oracle_layer(w, "cuda")
    L.close()


@pytest.mark.parametrize("T", [4, 1, 8])
def test_verify_q8_full_size(verify_q8, T):
    w, L, ol = verify_q8
    x = synth.activations(w, "cuda", T=T)
    err, excl, r = check_layer(L, x, ol, w.top_k, w.E, TOL[pkg.ACT_BF16], f"verify_q8 T={T}")
    print(f"verify_q8 T={T}: max rel err {err:.3e}, excluded {excl}, unique experts {len(r['act'])}")


def test_verify_q8_deterministic_and_graph(verify_q8):
    w, L, _ = verify_q8
    x = synth.activations(w, "cuda")
    y1 = L.forward(x).clone()
    y2 = L.forward(x).clone()
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    s = torch.cuda.Stream()
    y3 = torch.empty_like(y1)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        L.forward(x, y3, stream=s)  # warm on the capture stream
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            L.forward(x, y3, stream=s)
    y3.zero_()
    g.replay()
    torch.cuda.synchronize()
    L.status()
    assert torch.equal(y1, y3)


@pytest.fixture(scope="module")
def verify_mixed():
    w = synth.WORKLOADS["verify_mixed"]
    L, _ = synthetic_layer(w, pkg.ACT_BF16, T_max=8)
    yield w, L, synth_oracle_layer(w, "cuda")
    L.close()


@pytest.mark.parametrize("T", [4, 3])
def test_verify_mixed_full_size(verify_mixed, T):
    w, L, ol = verify_mixed
    x = synth.activations(w, "cuda", T=T)
    err, excl, r = check_layer(L, x, ol, w.top_k, w.E, TOL[pkg.ACT_BF16], f"verify_mixed T={T}")
    print(f"verify_mixed T={T}: max rel err {err:.3e}, excluded {excl}")


@pytest.mark.parametrize("T", [1, 4, 8])
def test_forward_resnorm_is_residual_add_then_rmsnorm(tiny, T):
    """moe_forward_resnorm, one step of the residual stream: h_out = h_in + y
    with y the fp32 output of moe_forward_f32, bit for bit (the same combine
    sum, then one fp32 add); xn = rmsnorm(h_out) (weight 1, eps) up to the
    fp32 summation order and, in bf16 mode, one rounding; y and xn against
    the oracle within the layer's tolerance; in place (h_in is h_out) the
    same; overlapping outputs are refused."""
    w, L, ol, act = tiny
    eps = 1e-6
    g = torch.Generator(device="cuda").manual_seed(1234 + T)
    h_in = torch.randn(T, w.H, generator=g, device="cuda", dtype=torch.float32)
    x = (h_in / torch.sqrt((h_in * h_in).mean(dim=-1, keepdim=True) + eps)).to(XDT[act])
    y32 = L.forward(x, out_f32=True)
    h_out, xn = L.forward_resnorm(x, h_in, eps=eps)
    torch.cuda.synchronize()
    L.status()
    assert torch.equal(h_out, h_in + y32)
    ref_xn = h_out / torch.sqrt((h_out * h_out).mean(dim=-1, keepdim=True) + eps)
    d = (xn.float() - ref_xn).abs()
    if act == pkg.ACT_F32:
        assert d.max().item() <= 1e-5 * ref_xn.abs().max().item()
    else:
        assert bool((d <= ref_xn.abs() * 2.0 ** -8 + 1e-6).all())
    y_ref, r = omoe.forward(to_np(x), ol)
    keep = ~omoe.near_tie_tokens(r["logits"], w.top_k)
    assert omoe.max_rel_err(to_np(h_out - h_in)[keep], y_ref[keep]) <= TOL[act]
    h_ref = to_np(h_in).astype(np.float64) + y_ref
    xn_ref = h_ref / np.sqrt((h_ref * h_ref).mean(axis=-1, keepdims=True) + eps)
    assert omoe.max_rel_err(to_np(xn)[keep], xn_ref[keep]) <= TOL[act]
    h2 = h_in.clone()
    _, xn2 = L.forward_resnorm(x, h2, h_out=h2, eps=eps)
    torch.cuda.synchronize()
    assert torch.equal(h2, h_out) and torch.equal(xn2, xn)
    with pytest.raises(pkg.MoEError):
        L.forward_resnorm(x, h_in, xn=x)


@pytest.mark.parametrize("T", [1, 4, 8])
def test_forward_f32_is_the_unrounded_output(tiny, T):
    """moe_forward_f32 stores the combine's fp32 sum: in bf16 mode its rounding
    to bf16 is moe_forward's output bit for bit; in check mode it is that output."""
    w, L, ol, act = tiny
    x = synth.activations(w, "cuda", T=T, variant=7).to(XDT[act])
    y = L.forward(x)
    y32 = L.forward(x, out_f32=True)
    torch.cuda.synchronize()
    L.status()
    assert y32.dtype == torch.float32
    assert torch.equal(y32.to(y.dtype), y)
    ref, r = omoe.forward(to_np(x), ol)
    keep = ~omoe.near_tie_tokens(r["logits"], w.top_k)
    assert omoe.max_rel_err(to_np(y32)[keep], ref[keep]) <= TOL[act]
