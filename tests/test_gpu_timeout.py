"""The bounded device-side waits end a launch with an error instead of a
hang: with a 1 ms wait limit, a forward whose routing publication never comes
(the moe_layer_inject_timeout hook: the work-claiming threads wait for a flag
value the kernel never writes) reports MOE_ETIMEOUT with its wait site
through moe_layer_status, and the next forward is bit-identical to one taken
before.  No fault, trap or endless loop is involved."""
import time

import pytest
import torch

import block_quantized_moe_layer_gb300 as pkg
from block_quantized_moe_layer_gb300 import synth
from block_quantized_moe_layer_gb300.workloads import synthetic_layer

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,act", [("tiny", pkg.ACT_BF16), ("tiny", pkg.ACT_F32), ("verify_q8", pkg.ACT_BF16)])
def test_routing_wait_times_out_and_the_layer_recovers(name, act):
    w = synth.WORKLOADS[name]
    L, _ = synthetic_layer(w, act, T_max=8, wait_limit_us=1000)
    try:
        x = synth.activations(w, "cuda").to(torch.bfloat16 if act == pkg.ACT_BF16 else torch.float32)
        y0 = L.forward(x).clone()
        L.status()
        L.inject_timeout(1)
        t0 = time.perf_counter()
        L.forward(x)
        with pytest.raises(pkg.MoEError) as ei:
            L.status()
        dt = time.perf_counter() - t0
        assert ei.value.code == pkg.MOE_ETIMEOUT
        assert "routing flag" in str(ei.value)
        assert dt < 5.0, f"the timed-out launch took {dt:.2f} s"
        L.status()  # cleared
        for _ in range(2):
            y = L.forward(x)
            torch.cuda.synchronize()
            L.status()
            assert torch.equal(y, y0)
        print(f"{name} act={act}: timed-out launch and status read in {dt * 1e3:.1f} ms")
    finally:
        L.close()


def test_inject_rejects_unknown_sites():
    w = synth.WORKLOADS["tiny"]
    L, _ = synthetic_layer(w, pkg.ACT_BF16, T_max=4)
    try:
        with pytest.raises(pkg.MoEError):
            L.inject_timeout(2)
    finally:
        L.close()
