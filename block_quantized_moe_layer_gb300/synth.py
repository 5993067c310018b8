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


@dataclass(frozen=True)
class RoundWorkload:
    """One MTP draft/verify round: k drafts (verify batch k + 1), target
    layers, k draft heads (head j runs at T = j + 1), a Q8_0 LM head [V, H]
    and the draft noise std ("Support Step3.5/3.7 flash mtp3", "Overview":
    three chained heads, a four-row verify batch)."""
    name: str
    seed: int
    k: int
    V: int
    layers: Tuple[Workload, ...]
    heads: Tuple[Workload, ...]
    lm_std: float = 0.02
    noise_std: float = 0.05


def round_workload(name, seed, H, E, top_k, I, I_sh, k=3, n_layers=8, V=32768, bias_std=0.5, q8_layers=(0, 7),
                   noise_std=0.05) -> RoundWorkload:
    """Target layers in the mixed recipe (routed Q4KS, shared Q8_0) except
    ``q8_layers`` (all Q8_0); draft heads in the mixed recipe."""
    layers = tuple(Workload(f"{name}_L{l}", seed * 100 + l, T=k + 1, H=H, E=E, top_k=top_k, I=I, I_shared=I_sh,
                            bias_std=bias_std, routed_fmt=FMT_Q8_0 if l in q8_layers else FMT_Q4KS)
                   for l in range(n_layers))
    heads = tuple(Workload(f"{name}_D{j}", seed * 100 + 50 + j, T=j + 1, H=H, E=E, top_k=top_k, I=I, I_shared=I_sh,
                           bias_std=bias_std, routed_fmt=FMT_Q4KS) for j in range(k))
    return RoundWorkload(name, seed, k, V, layers, heads, noise_std=noise_std)


ROUNDS = {
    # the Step-5-shaped round: 8 target layers, 3 heads, vocab 32768
    "mtp_round": round_workload("mtp_round", 4, 4096, 352, 8, 1280, 1280),
    # a small round for full comparisons
    "tiny_round": round_workload("tiny_round", 5, 512, 16, 2, 256, 256, n_layers=3, V=1000, q8_layers=(0,)),
}


def lm_weight(r: RoundWorkload, device="cpu") -> torch.Tensor:
    """fp32 [V, H] LM head weights N(0, lm_std^2)."""
    return normal((r.V, r.layers[0].H), r.lm_std, device, (r.seed * 1_000_003 + _LM * 65_537 + 12_345) & 0x7FFF_FFFF_FFFF)


def round_inputs(r: RoundWorkload, device="cpu", variant: int = 0):
    """(x bf16 [k+1, H], noise fp32 [k, k, H]): the verify batch and, for head j,
    rows 0..j of noise[j]."""
    x = activations(r.layers[0], device, T=r.k + 1, variant=variant)
    H = r.layers[0].H
    nz = torch.stack([noise(r.seed + 1000 * variant, j, (r.k, H), r.noise_std, device) for j in range(r.k)])
    return x, nz
