"""The synthetic input recipe (no GPU): the prefill workload's x carries, on
exactly `offset_dims` hidden dims, a per-token AR(1) offset with coefficient
`offset_rho` and stationary std `offset_std`, added before the bf16 rounding;
every other dim is the plain N(0, 1) draw."""
import dataclasses

import numpy as np

from block_quantized_moe_layer_gb300 import synth


def test_prefill_offsets_follow_the_ar1_recipe():
    w = synth.WORKLOADS["prefill_q8"]
    assert (w.offset_dims, w.offset_std, w.offset_rho) == (64, 0.3, 0.99)
    x = synth.activations(w).float().numpy().astype(np.float64)
    x0 = synth.activations(dataclasses.replace(w, offset_dims=0)).float().numpy().astype(np.float64)
    d = x - x0
    cols = np.flatnonzero(np.abs(d).max(axis=0) > 0)
    assert cols.size == w.offset_dims  # dims drawn without replacement; the rest untouched, bit for bit
    o = d[:, cols]  # the offsets plus the bf16 rounding of x + o (|x| ~ 1: ulp 2^-7)
    assert abs(o.std() / w.offset_std - 1.0) < 0.25
    lag1 = np.mean([np.corrcoef(o[1:, j], o[:-1, j])[0, 1] for j in range(o.shape[1])])
    assert lag1 > 0.95  # slowly varying: successive tokens' offsets nearly equal


def test_other_workloads_have_plain_normal_inputs():
    w = synth.WORKLOADS["verify_q8"]
    assert w.offset_dims == 0
    x = synth.activations(w).float().numpy()
    assert x.shape == (w.T, w.H)
    assert abs(x.std() - 1.0) < 0.05 and abs(x.mean()) < 0.05
