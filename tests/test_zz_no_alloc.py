"""The allocation-free acceptance entry point (static scratch inside the
library), its size limit, and its results against the oracle's greedy
acceptance and against the workspace entry point.

Some callers cannot allocate device memory: a C runtime that drives the
draft/verify loop with no device allocator of its own, for which cudaMalloc /
cudaFree would also synchronise the device between verify rounds.  This file
checks the entry point made for them.  It is named to be collected last, so
that it also runs after every other test has used the library on the same
device."""
import numpy as np
import pytest

import block_quantized_moe_layer_gb300 as pkg
from oracle import accept as oacc


def test_noalloc_rejects_sizes_beyond_static_scratch():
    # 16 + 8 * 16 * ceil(600000 / 16384) = 4752 bytes > 4096: refused on the
    # host before any CUDA call.
    L = pkg.lib()
    # (the pointers are never dereferenced: the size check refuses first)
    rc = L.mtp_verify_accept_noalloc(16, 15, 16, 600_000, 16, 20, None)
    assert rc == pkg.MOE_EINVAL
    msg = L.moe_last_error().decode()
    assert "static scratch holds 4096" in msg and "V=600000" in msg
    # the stated limit: every V <= 507904 fits for k = 15, the next does not
    assert L.mtp_verify_accept_workspace_bytes(15, 507_904) == 16 + 8 * 16 * 31 <= 4096
    assert L.mtp_verify_accept_workspace_bytes(15, 507_905) > 4096


def _case(rng, k, V, reject_at):
    logits = rng.normal(size=(k + 1, V)).astype(np.float32)
    draft = logits.argmax(axis=1)[:k].copy()
    if reject_at is not None and k:
        draft[reject_at] = (draft[reject_at] + 1) % V
    return draft, logits


@pytest.mark.gpu
@pytest.mark.parametrize("k,V", [(0, 1), (3, 32768), (7, 151_936), (15, 507_904), (4, 1_000)])
def test_noalloc_matches_oracle_and_workspace_entry_two_calls_in_a_row(k, V):
    import torch
    rng = np.random.default_rng(k * 1009 + V)
    cases = [_case(rng, k, V, None), _case(rng, k, V, (k // 2) if k else None)]
    # the oracle's greedy acceptance on the same host arrays
    want = []
    for draft, logits in cases:
        n, nxt, _ = oacc.greedy_accept(draft.tolist(), logits)
        want.append([n, nxt])
    dev = []
    for draft, logits in cases:
        dev.append((torch.tensor(draft, dtype=torch.int32, device="cuda"),
                    torch.from_numpy(logits).cuda().contiguous()))
    outs = [torch.full((2,), -7, dtype=torch.int32, device="cuda") for _ in cases]
    # two calls back to back on one stream, read only afterwards
    for (d, lg), o in zip(dev, outs):
        pkg.verify_accept_noalloc(d, lg, out=o)
    torch.cuda.synchronize()
    for (d, lg), o, w in zip(dev, outs, want):
        got = o.cpu().tolist()
        assert got == w, (got, w)
        assert got == pkg.verify_accept(d, lg).cpu().tolist()
    # and again, each call interleaved with the workspace entry point
    for (d, lg), o, w in zip(dev, outs, want):
        o.fill_(-7)
        pkg.verify_accept_noalloc(d, lg, out=o)
        ref = pkg.verify_accept(d, lg)
        got = o.cpu().tolist()
        assert got == w, (got, w)
        assert got == ref.cpu().tolist()
