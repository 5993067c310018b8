"""Edge cases of the T <= 8 path against the oracle: every expert selected
(k = E), k = 1, the largest expert count and top-k the layer accepts
(E = 1024, k = 16: 128 (token, slot) pairs at T = 8, the general
permutation path), no shared expert, no router bias."""
import pytest
import torch

import block_quantized_moe_layer_gb300 as pkg
from block_quantized_moe_layer_gb300 import synth
from block_quantized_moe_layer_gb300.workloads import synthetic_layer
from tests._oracle_layer import synth_oracle_layer
from tests.gpu_util import check_layer

pytestmark = pytest.mark.gpu

TOL = {pkg.ACT_BF16: 2e-2, pkg.ACT_F32: 1e-3}
XDT = {pkg.ACT_BF16: torch.bfloat16, pkg.ACT_F32: torch.float32}

CASES = {
    "all_experts": synth.Workload("edge_all", 31, T=8, H=256, E=8, top_k=8, I=128, I_shared=128, bias_std=0.5),
    "top1": synth.Workload("edge_top1", 32, T=8, H=256, E=16, top_k=1, I=128, I_shared=128, bias_std=0.5),
    "max_e_k": synth.Workload("edge_max", 33, T=8, H=256, E=1024, top_k=16, I=64, I_shared=64, bias_std=0.5),
    "no_shared_no_bias": synth.Workload("edge_noshared", 34, T=8, H=512, E=24, top_k=4, I=96, I_shared=0),
    "q4_top1": synth.Workload("edge_q4_top1", 35, T=8, H=512, E=40, top_k=1, I=256, I_shared=256,
                              bias_std=0.5, routed_fmt=synth.FMT_Q4KS),
}


@pytest.mark.parametrize("act", [pkg.ACT_BF16, pkg.ACT_F32], ids=["bf16", "f32"])
@pytest.mark.parametrize("name", list(CASES))
def test_edge_case(name, act):
    w = CASES[name]
    L, _ = synthetic_layer(w, act, T_max=8)
    try:
        ol = synth_oracle_layer(w, "cuda")
        for T in (1, 5, 8):
            x = synth.activations(w, "cuda", T=T).to(XDT[act])
            err, excl, r = check_layer(L, x, ol, w.top_k, w.E, TOL[act], f"{name} T={T}")
            print(f"{name} act={act} T={T}: max rel err {err:.2e}, excluded {excl}, experts {len(r['act'])}")
    finally:
        L.close()
