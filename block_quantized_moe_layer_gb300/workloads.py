"""Builds resident layers for the synthetic workloads in :mod:`.synth`.

Weights are drawn on the GPU, quantised by the library's own quantiser
(``moe_quantize``) and handed to ``moe_layer_create``; the serialised copies
are freed afterwards.
"""
import torch

from . import FMT_F32, FMT_Q8_0, Layer, LmHead, quantize, synth


def synthetic_layer(w: synth.Workload, act, T_max=None, device="cuda", keep_serialised=False, experts_held=None,
                    with_shared=True, wait_limit_us=0):
    """Returns (Layer, serialised dict or None) for workload ``w``.
    ``experts_held`` = (begin, count) makes one expert-parallel shard holding
    those routed experts (default: all); ``with_shared`` puts the shared
    expert on it."""
    T_max = w.T if T_max is None else T_max
    Wr, b = synth.router(w, device)
    begin, count = experts_held if experts_held is not None else (0, w.E)
    experts = []
    ser = {}
    for e in range(begin, begin + count):
        g, u, d = synth.expert(w, e, device)
        q = (w.routed_fmt, quantize(w.routed_fmt, g), quantize(w.routed_fmt, u),
             quantize(w.routed_fmt, d))
        experts.append(q)
        del g, u, d
    shared = None
    I_sh = w.I_shared if with_shared else 0
    if I_sh:
        g, u, d = synth.shared(w, device)
        shared = (w.shared_fmt, quantize(w.shared_fmt, g), quantize(w.shared_fmt, u),
                  quantize(w.shared_fmt, d))
    L = Layer(w.H, w.E, w.top_k, w.I, I_sh, T_max, act, Wr.contiguous(),
              None if b is None else b.contiguous(), experts, shared, expert_begin=begin,
              wait_limit_us=wait_limit_us)
    if keep_serialised:
        ser = dict(experts=experts, shared=shared, router=Wr, bias=b)
        return L, ser
    del experts, shared
    torch.cuda.synchronize()
    return L, None


def synthetic_lm_head(r: synth.RoundWorkload, act, T_max=8, device="cuda"):
    """LmHead for round workload ``r`` (weights drawn on the device, Q8_0)."""
    w = synth.lm_weight(r, device)
    q = quantize(FMT_Q8_0, w)
    del w
    lm = LmHead(q, r.V, r.layers[0].H, T_max, act)
    del q
    torch.cuda.synchronize()
    return lm


def synthetic_round(r: synth.RoundWorkload, act, device="cuda"):
    """(target layers, draft heads, LM head) for round workload ``r``."""
    layers = [synthetic_layer(w, act, T_max=r.k + 1, device=device)[0] for w in r.layers]
    heads = [synthetic_layer(w, act, T_max=j + 1, device=device)[0] for j, w in enumerate(r.heads)]
    return layers, heads, synthetic_lm_head(r, act, T_max=r.k + 1, device=device)
