"""Parity of the acceptance kernel with the oracle (bit-exact)."""
import numpy as np
import pytest
import torch

import block_quantized_moe_layer_gb300 as pkg
from oracle.accept import greedy_accept

pytestmark = pytest.mark.gpu


def _run(draft, logits, ws=None):
    d = torch.tensor(draft, dtype=torch.int32, device="cuda")
    L = torch.as_tensor(logits, dtype=torch.float32).cuda().contiguous()
    return pkg.verify_accept(d, L, workspace=ws).cpu().tolist()


@pytest.mark.parametrize("V", [1, 7, 1000, 32768, 100_003])
@pytest.mark.parametrize("k", [0, 1, 3, 7])
def test_accept_random(V, k):
    rng = np.random.default_rng(V * 31 + k)
    for trial in range(6):
        L = rng.normal(size=(k + 1, V)).astype(np.float32)
        a = L.argmax(axis=1)
        draft = a[:k].copy()
        if k and trial % 3:
            j = rng.integers(0, k)
            draft[j] = (draft[j] + 1) % V if V > 1 else draft[j]
        n, nxt, _ = greedy_accept(draft.tolist(), L)
        assert _run(draft.tolist(), L) == [n, nxt]


def test_accept_ties_and_worked_example():
    V = 50_000
    L = np.zeros((4, V), np.float32)
    L[0, [5, 17, 40_000]] = 3.0   # tie: lowest id 5 wins
    L[1, [4, 30_000]] = 1.0
    L[2, 23] = 2.0
    L[3, 5] = 1.0
    assert _run([5, 4, 9], L) == list(greedy_accept([5, 4, 9], L)[:2]) == [2, 23]
    assert _run([17, 4, 9], L) == [0, 5]
    L[2, 9] = 5.0
    assert _run([5, 4, 9], L) == [3, 5]


def test_accept_workspace_reuse():
    ws = pkg.accept_workspace(3, 32768)
    rng = np.random.default_rng(0)
    for _ in range(5):
        L = rng.normal(size=(4, 32768)).astype(np.float32)
        d = L.argmax(axis=1)[:3].tolist()
        assert _run(d, L, ws) == list(greedy_accept(d, L)[:2])
    assert int(ws[:4].view(torch.int32).item()) == 0
