"""Host-side helpers of bench.py (no GPU)."""
import numpy as np

import bench


def test_expert_load_summary():
    # 5 experts: loads 0, 1, 3, 0, 8 -> three used; bins [1], [2,4), [8,16)
    offs = np.cumsum([0, 0, 1, 3, 0, 8])
    s = bench.expert_load_summary(offs)
    assert s == {"experts_used": 3, "pairs": 12, "min": 1, "median": 3.0, "max": 8, "pow2_hist": [1, 1, 0, 1]}
    assert bench.expert_load_summary(np.zeros(4, dtype=np.int64)) == {"experts_used": 0}


def test_algorithmic_bytes_of_the_verify_workloads():
    # the roofline numerator, from the formats' block sizes: Q8_0 stores 32
    # weights in 34 bytes, Q4KS 256 weights in 144; fp32 router and bias;
    # bf16 x and y of T = 4 tokens
    from block_quantized_moe_layer_gb300 import synth
    H, I, E, T = 4096, 1280, 352, 4
    router = E * H * 4 + E * 4
    q8_expert = 3 * (I * H // 32 * 34)
    q4_expert = 3 * (I * H // 256 * 144)
    act = 2 * T * H * 2
    assert bench.algorithmic_bytes(synth.WORKLOADS["verify_q8"], 30) == router + 31 * q8_expert + act == 523_896_192
    assert bench.algorithmic_bytes(synth.WORKLOADS["verify_mixed"], 30) == router + 30 * q4_expert + q8_expert + act


def test_traffic_record_needs_the_captured_kernel_sources(monkeypatch):
    import json
    import os
    records = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    for key, r in records.items():
        assert r["bytes_per_launch"] == r["read_bytes_per_launch"] + r["write_bytes_per_launch"], key
        assert abs(r["small_case"]["read_over_algorithmic"] - 1.0) < 1e-2, key
    # a record taken on other sources is never reported
    monkeypatch.setattr(bench, "kernel_hash", lambda path: "0" * 16)
    assert bench.traffic_record("small_t", "verify_q8") is None
