"""Builds resident layers for the synthetic workloads in :mod:`.synth`.

Weights are drawn on the GPU, quantised by the library's own quantiser
(``moe_quantize``) and handed to ``moe_layer_create``; the serialised copies
are freed afterwards.
"""
import torch

from . import FMT_F32, Layer, quantize, synth


def synthetic_layer(w: synth.Workload, act, T_max=None, device="cuda", keep_serialised=False):
    """Returns (Layer, serialised dict or None) for workload ``w``."""
    T_max = w.T if T_max is None else T_max
    Wr, b = synth.router(w, device)
    experts = []
    ser = {}
    for e in range(w.E):
        g, u, d = synth.expert(w, e, device)
        q = (w.routed_fmt, quantize(w.routed_fmt, g), quantize(w.routed_fmt, u),
             quantize(w.routed_fmt, d))
        experts.append(q)
        del g, u, d
    shared = None
    if w.I_shared:
        g, u, d = synth.shared(w, device)
        shared = (w.shared_fmt, quantize(w.shared_fmt, g), quantize(w.shared_fmt, u),
                  quantize(w.shared_fmt, d))
    L = Layer(w.H, w.E, w.top_k, w.I, w.I_shared, T_max, act, Wr.contiguous(),
              None if b is None else b.contiguous(), experts, shared)
    if keep_serialised:
        ser = dict(experts=experts, shared=shared, router=Wr, bias=b)
        return L, ser
    del experts, shared
    torch.cuda.synchronize()
    return L, None
