"""Expert-parallel shards of one layer on one GPU: layers holding
complementary expert ranges (the shared expert on one of them) give parts
whose sum is the whole layer's output, and each part matches the oracle's
shard forward.  Shards with no work for a batch (none of their experts
chosen, no shared expert) return zero, or x with the residual."""
import numpy as np
import pytest
import torch

import block_quantized_moe_layer_gb300 as pkg
from block_quantized_moe_layer_gb300 import ep, synth
from block_quantized_moe_layer_gb300.workloads import synthetic_layer
from oracle import moe as omoe
from tests._oracle_layer import synth_oracle_layer
from tests.gpu_util import to_np

pytestmark = pytest.mark.gpu

TOL = {pkg.ACT_BF16: 2e-2, pkg.ACT_F32: 1e-3}
XDT = {pkg.ACT_BF16: torch.bfloat16, pkg.ACT_F32: torch.float32}

SMALL = synth.Workload("ep_small", 41, T=8, H=512, E=40, top_k=3, I=256, I_shared=256, bias_std=0.5)
SMALL_Q4 = synth.Workload("ep_small_q4", 42, T=8, H=512, E=40, top_k=3, I=256, I_shared=256, bias_std=0.5,
                          routed_fmt=synth.FMT_Q4KS)
LARGE_T = synth.Workload("ep_lt", 43, T=200, H=512, E=40, top_k=3, I=256, I_shared=256, bias_std=0.5)


def _shards(w, act, world, T_max):
    return [synthetic_layer(w, act, T_max=T_max, experts_held=r, with_shared=ep.holds_shared(i))[0]
            for i, r in enumerate(ep.expert_ranges(w.E, world))]


def _check_split(w, act, world, Ts, T_max):
    full, _ = synthetic_layer(w, act, T_max=T_max)
    shards = _shards(w, act, world, T_max)
    ol = synth_oracle_layer(w, "cuda")
    try:
        for T in Ts:
            x = synth.activations(w, "cuda", T=T, variant=T).to(XDT[act])
            yf = to_np(full.forward(x))
            parts = [to_np(L.forward(x)) for L in shards]
            torch.cuda.synchronize()
            for L in shards + [full]:
                L.status()
            xn = to_np(x)
            y_ref, r = omoe.forward(xn, ol)
            keep = ~omoe.near_tie_tokens(r["logits"], w.top_k)
            # every shard routes like the whole layer
            ids_full = to_np(full.routing(T)[0])
            for L in shards:
                assert np.array_equal(to_np(L.routing(T)[0]), ids_full)
            for i, ((b, n), p) in enumerate(zip(ep.expert_ranges(w.E, world), parts)):
                want, _ = omoe.forward_shard(xn, ol, b, n, ep.holds_shared(i), routing=r)
                # a part is a piece of y: measure it on the whole output's scale
                err = np.abs(p[keep] - want[keep]).max() / np.abs(y_ref[keep]).max()
                assert err <= TOL[act], f"shard {i} T={T}: err {err:.2e}"
            total = sum(parts)
            e_full = omoe.max_rel_err(total[keep], yf[keep])
            e_ref = omoe.max_rel_err(total[keep], y_ref[keep])
            # check mode: the parts add up to the whole layer up to fp32 rounding
            bound = 1e-5 if act == pkg.ACT_F32 else 2 * TOL[act]
            assert e_full <= bound and e_ref <= TOL[act], (T, e_full, e_ref)
            print(f"{w.name} act={act} world={world} T={T}: sum of parts vs layer {e_full:.2e}, vs oracle {e_ref:.2e}")
    finally:
        for L in shards + [full]:
            L.close()


@pytest.mark.parametrize("act", [pkg.ACT_F32, pkg.ACT_BF16], ids=["f32", "bf16"])
@pytest.mark.parametrize("world", [2, 3])
def test_shards_sum_to_the_layer(act, world):
    _check_split(SMALL, act, world, (1, 4, 8), 8)


def test_shards_sum_to_the_layer_q4():
    _check_split(SMALL_Q4, pkg.ACT_F32, 2, (3, 8), 8)


def test_shards_sum_to_the_layer_prefill_path():
    _check_split(LARGE_T, pkg.ACT_BF16, 2, (9, 200), 200)


@pytest.mark.parametrize("act", [pkg.ACT_F32, pkg.ACT_BF16], ids=["f32", "bf16"])
def test_shard_with_no_work(act):
    w = SMALL
    ol = synth_oracle_layer(w, "cuda")
    x = synth.activations(w, "cuda", T=1, variant=99).to(XDT[act])
    r = omoe.route(to_np(x), ol)
    unused = sorted(set(range(w.E)) - set(r["ids"][0].tolist()))[0]
    idle, _ = synthetic_layer(w, act, T_max=8, experts_held=(unused, 1), with_shared=False)
    shared_only, _ = synthetic_layer(w, act, T_max=8, experts_held=(unused, 1), with_shared=True)
    try:
        for _ in range(2):  # twice: the counters are reset between launches
            y = idle.forward(x)
            yr = idle.forward(x, residual=True)
            ys = to_np(shared_only.forward(x))
            torch.cuda.synchronize()
            idle.status()
            shared_only.status()
            assert not to_np(y).any()
            assert torch.equal(yr, x)
            want = omoe.swiglu_expert(to_np(x), ol.shared)
            assert omoe.max_rel_err(ys, want) <= TOL[act]
    finally:
        idle.close()
        shared_only.close()


def test_bad_expert_ranges_are_rejected():
    w = synth.WORKLOADS["tiny"]
    for rng in ((-1, 4), (10, 7), (0, -2)):
        with pytest.raises(pkg.MoEError):
            synthetic_layer(w, pkg.ACT_BF16, T_max=4, experts_held=rng)
