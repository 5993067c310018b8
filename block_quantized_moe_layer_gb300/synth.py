"""Seeded synthetic inputs for the MoE layer workloads.

This module holds random-number generation and tensor shapes only: no
quantisation, routing or FFN arithmetic.  Both the CUDA path (tests, bench)
and the oracle (tests) take their inputs from here.  Weights are drawn as
fp32 on the requested device with torch's generator for that device; every
tensor has its own seed derived from (workload seed, tensor kind, expert), so
any single expert can be regenerated without drawing the others.  CPU and
CUDA generators give different streams: a test that compares the two paths
draws on one device and copies to the other.

Workloads (shapes of the pages' Step-5 layer: hidden 4096, 352 routed
experts, 8 selected, plus a shared expert -- "Step-5 Preview GGUF", "Model
background" table; T = 4 is id_last plus three MTP drafts -- "Support
Step3.5/3.7 flash mtp3", "Overview", Round 1 step 1; T = 1024 is one
``-ub 1024`` micro-batch -- "Step-3.5-Flash MTP GGUF", "Usage").  The expert
intermediate size 1280 is a synthetic choice: the pages do not give it.
"""

from dataclasses import dataclass, field, replace
from typing import Optional, Tuple

import torch

FMT_F32, FMT_BF16, FMT_Q8_0, FMT_Q4KS = 0, 1, 2, 3

# tensor-kind tags for per-tensor seeds
_ROUTER_W, _ROUTER_B, _GATE, _UP, _DOWN, _SH_GATE, _SH_UP, _SH_DOWN, _X, _OFFS, _NOISE, _LM = range(12)


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    T: int
    H: int
    E: int
    top_k: int
    I: int
    I_shared: int
    w_std: float = 0.02
    router_std: float = 0.02
    bias_std: Optional[float] = None      # per-expert router bias N(0, bias_std)
    routed_fmt: int = FMT_Q8_0            # gate/up/down of routed experts
    shared_fmt: int = FMT_Q8_0
    offset_dims: int = 0                  # slowly varying per-token offset (prefill)
    offset_std: float = 0.0
    offset_rho: float = 0.99
    extra: dict = field(default_factory=dict, compare=False, hash=False)


WORKLOADS = {
    # tiny layer for small-case checks
    "tiny": Workload("tiny", 0, T=4, H=256, E=16, top_k=2, I=128, I_shared=128),
    # one Step-5-shaped layer on the T=4 verify batch, all Q8_0, biased router
    "verify_q8": Workload("verify_q8", 1, T=4, H=4096, E=352, top_k=8, I=1280,
                          I_shared=1280, bias_std=0.5),
    # same shapes, routed experts in the 4-bit Q4KS format, shared Q8_0
    "verify_mixed": Workload("verify_mixed", 2, T=4, H=4096, E=352, top_k=8, I=1280,
                             I_shared=1280, bias_std=0.5, routed_fmt=FMT_Q4KS),
    # prefill-sized micro-batch on the verify_q8 layer shapes
    "prefill_q8": Workload("prefill_q8", 3, T=1024, H=4096, E=352, top_k=8, I=1280,
                           I_shared=1280, bias_std=0.5, offset_dims=64, offset_std=0.3),
}


def _seed(w: Workload, kind: int, index: int = 0) -> int:
    return (w.seed * 1_000_003 + kind * 65_537 + index * 7 + 12_345) & 0x7FFF_FFFF_FFFF


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, std, device, seed) -> torch.Tensor:
    g = _gen(device, seed)
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * std


def router(w: Workload, device="cpu") -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Router weight fp32 [E, H] and optional bias fp32 [E]."""
    Wr = normal((w.E, w.H), w.router_std, device, _seed(w, _ROUTER_W))
    b = None
    if w.bias_std is not None:
        b = normal((w.E,), w.bias_std, device, _seed(w, _ROUTER_B))
    return Wr, b


def expert(w: Workload, e: int, device="cpu"):
    """fp32 (gate [I, H], up [I, H], down [H, I]) of routed expert e."""
    return (normal((w.I, w.H), w.w_std, device, _seed(w, _GATE, e)),
            normal((w.I, w.H), w.w_std, device, _seed(w, _UP, e)),
            normal((w.H, w.I), w.w_std, device, _seed(w, _DOWN, e)))


def shared(w: Workload, device="cpu"):
    """fp32 (gate [I_sh, H], up [I_sh, H], down [H, I_sh]) of the shared expert."""
    return (normal((w.I_shared, w.H), w.w_std, device, _seed(w, _SH_GATE)),
            normal((w.I_shared, w.H), w.w_std, device, _seed(w, _SH_UP)),
            normal((w.H, w.I_shared), w.w_std, device, _seed(w, _SH_DOWN)))


def activations(w: Workload, device="cpu", T: Optional[int] = None, variant: int = 0) -> torch.Tensor:
    """x bf16 [T, H]: N(0, 1), plus (prefill workload) a per-token offset on
    ``offset_dims`` hidden dims drawn without replacement, each an AR(1)
    sequence over tokens with stationary std ``offset_std`` and coefficient
    ``offset_rho``; the offset is added in fp32 before the bf16 rounding.
    ``variant`` selects an independent draw of the same distribution.
    """
    T = w.T if T is None else T
    s = _seed(w, _X, variant)
    x = normal((T, w.H), 1.0, "cpu", s)
    if w.offset_dims:
        g = _gen("cpu", _seed(w, _OFFS, variant))
        dims = torch.randperm(w.H, generator=g)[: w.offset_dims]
        z = torch.randn(T, w.offset_dims, generator=g, dtype=torch.float64)
        o = torch.empty(T, w.offset_dims, dtype=torch.float64)
        rho = w.offset_rho
        o[0] = w.offset_std * z[0]
        inov = (1.0 - rho * rho) ** 0.5 * w.offset_std
        for t in range(1, T):
            o[t] = rho * o[t - 1] + inov * z[t]
        x[:, dims] += o.to(torch.float32)
    return x.to(torch.bfloat16).to(device)


def noise(seed: int, head: int, shape, std, device="cpu") -> torch.Tensor:
    """N(0, std^2) fp32 noise for draft head ``head`` (MTP round workload)."""
    return normal(shape, std, device, (seed * 1_000_003 + _NOISE * 65_537 + head * 7 + 99) & 0x7FFF_FFFF_FFFF)


def with_T(w: Workload, T: int) -> Workload:
    return replace(w, T=T)
