"""Host-side helpers of bench.py (no GPU)."""
import numpy as np

import bench


def test_expert_load_summary():
    # 5 experts: loads 0, 1, 3, 0, 8 -> three used; bins [1], [2,4), [8,16)
    offs = np.cumsum([0, 0, 1, 3, 0, 8])
    s = bench.expert_load_summary(offs)
    assert s == {"experts_used": 3, "pairs": 12, "min": 1, "median": 3.0, "max": 8, "pow2_hist": [1, 1, 0, 1]}
    assert bench.expert_load_summary(np.zeros(4, dtype=np.int64)) == {"experts_used": 0}
