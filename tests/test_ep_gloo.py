"""Expert parallelism on the host: two gloo ranks on the CPU each compute
their shard's part of the layer (here with the oracle, since no GPU is
involved) on the balanced expert ranges of ``ep.expert_ranges``, with the
shared expert on rank 0, and ``ep.all_reduce_output`` sums the parts; the
sum must be the whole layer's output."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from block_quantized_moe_layer_gb300 import ep


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _layer():
    from oracle import formats
    from tests._oracle_layer import layer_from_fp32
    rng = np.random.default_rng(7)
    H, E, k, I = 64, 9, 3, 32
    Wr = rng.normal(0, 0.3, (E, H)).astype(np.float32)
    b = rng.normal(0, 0.5, E).astype(np.float32)
    ws = [tuple(rng.normal(0, 0.05, s).astype(np.float32) for s in ((I, H), (I, H), (H, I))) for _ in range(E)]
    sh = tuple(rng.normal(0, 0.05, s).astype(np.float32) for s in ((I, H), (I, H), (H, I)))
    x = rng.normal(size=(6, H)).astype(np.float32)
    return layer_from_fp32(H, E, k, I, I, Wr, b, lambda e: ws[e], sh, formats.FMT_Q8_0, formats.FMT_Q8_0), x


def _rank_main(rank, world, port, dtype, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    from oracle import moe
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        L, x = _layer()
        begin, count = ep.expert_ranges(L.E, world)[rank]
        part, _ = moe.forward_shard(x, L, begin, count, ep.holds_shared(rank))
        y = torch.from_numpy(part.astype(np.float32)).to(dtype)
        ep.all_reduce_output(y)
        q.put((rank, begin, count, y.float().numpy()))
    finally:
        dist.destroy_process_group()


def test_expert_ranges_cover_every_expert_once():
    for E in (1, 7, 16, 352):
        for world in range(1, min(E, 8) + 1):
            rs = ep.expert_ranges(E, world)
            assert len(rs) == world and rs[0][0] == 0
            assert all(b0 + n0 == b1 for (b0, n0), (b1, _) in zip(rs, rs[1:]))
            assert sum(n for _, n in rs) == E and max(n for _, n in rs) - min(n for _, n in rs) <= 1
    with pytest.raises(ValueError):
        ep.expert_ranges(3, 4)
    assert [ep.holds_shared(r) for r in range(3)] == [True, False, False]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_two_ranks_sum_to_the_layer(dtype):
    from oracle import moe
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, dtype, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted((q.get(timeout=5) for _ in range(world)), key=lambda g: g[0])
    assert [(b, n) for _, b, n, _ in got] == [(0, 5), (5, 4)]
    L, x = _layer()
    y, _ = moe.forward(x, L)
    tol = 1e-6 if dtype == torch.float32 else 2e-2
    for _, _, _, ys in got:  # every rank holds the sum
        assert moe.max_rel_err(ys, y) <= tol
