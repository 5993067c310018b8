"""The library's quantiser is bit-exact with the oracle's."""
import numpy as np
import pytest
import torch

import block_quantized_moe_layer_gb300 as pkg
from oracle import formats as F

pytestmark = pytest.mark.gpu


def _inputs(K, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    w = torch.randn(64, K, generator=g, device="cuda") * 0.02
    w[0] = 0.0                                    # zero rows
    w[1] = 0.5                                    # constant positive
    w[2] = -0.25                                  # constant negative
    w[3, :32] = torch.arange(-16, 16, device="cuda") * 0.5  # exact halves after scaling
    w[4] *= 1e-30                                 # tiny values
    w[5] *= 1e3
    return w.contiguous()


@pytest.mark.parametrize("fmt,K", [(pkg.FMT_Q8_0, 256), (pkg.FMT_Q8_0, 4096), (pkg.FMT_Q4KS, 512),
                                   (pkg.FMT_Q4KS, 4096)])
def test_quantiser_bit_exact(fmt, K):
    w = _inputs(K, K + fmt)
    got = pkg.quantize(fmt, w).cpu().numpy()
    want = F.quantize(fmt, w.cpu().numpy()).reshape(-1)
    assert got.shape == want.shape
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[:8]}"
