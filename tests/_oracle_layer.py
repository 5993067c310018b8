"""Builds oracle layers from fp32 weights with the oracle's own quantiser."""
import functools

import numpy as np

from oracle import formats, moe


def qtensor(fmt, w):
    w = np.ascontiguousarray(np.asarray(w, np.float32))
    return moe.QTensor(fmt, w.shape[0], w.shape[1], formats.quantize(fmt, w))


def expert_from_fp32(fmt, gate, up, down):
    return moe.Expert(qtensor(fmt, gate), qtensor(fmt, up), qtensor(fmt, down))


def layer_from_fp32(H, E, k, I, I_sh, Wr, b, expert_fp32, shared_fp32, routed_fmt, shared_fmt,
                    cache=True):
    """expert_fp32(e) -> (gate, up, down) fp32 arrays; quantised lazily, once."""
    def build(e):
        return expert_from_fp32(routed_fmt, *expert_fp32(e))
    if cache:
        build = functools.lru_cache(maxsize=None)(build)
    sh = expert_from_fp32(shared_fmt, *shared_fp32) if shared_fp32 is not None else None
    return moe.Layer(H=H, E=E, top_k=k, I=I, I_shared=I_sh,
                     router_w=np.asarray(Wr, np.float32),
                     router_b=None if b is None else np.asarray(b, np.float32),
                     expert=build, shared=sh)


def synth_oracle_layer(w, device="cpu", fetch=None):
    """Oracle layer for a synth workload; weights drawn on ``device``."""
    from block_quantized_moe_layer_gb300 import synth
    Wr, b = synth.router(w, device)
    to_np = (lambda t: t.float().cpu().numpy())

    def ex(e):
        return tuple(to_np(t) for t in synth.expert(w, e, device))
    sh = tuple(to_np(t) for t in synth.shared(w, device)) if w.I_shared else None
    return layer_from_fp32(w.H, w.E, w.top_k, w.I, w.I_shared, to_np(Wr),
                           None if b is None else to_np(b), ex, sh, w.routed_fmt, w.shared_fmt)
