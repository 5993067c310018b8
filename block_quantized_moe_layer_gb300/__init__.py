"""Block-quantized MoE layer for MTP verify batches on GB300 (sm_103a).

A thin ctypes binding over the C ABI in ``include/moe_layer.h``: argument
marshalling only.  Every step of the layer runs in the library's CUDA kernels;
there is no CPU fallback, and importing the binding's functions fails loudly
when the library has not been built (``python -m
block_quantized_moe_layer_gb300._build``).  PyTorch provides device memory
and streams.
"""
import ctypes
import os

from ._build import LIB

MOE_OK, MOE_EINVAL, MOE_ENOMEM, MOE_EFORMAT, MOE_ETIMEOUT, MOE_ECUDA = 0, -1, -2, -3, -4, -5
FMT_F32, FMT_BF16, FMT_Q8_0, FMT_Q4KS = 0, 1, 2, 3
ACT_BF16, ACT_F32 = 0, 1

_c = ctypes
EXPORTS = (
    "moe_layer_create", "moe_forward", "moe_get_routing", "moe_layer_status",
    "moe_layer_weight_bytes", "moe_layer_workspace_bytes", "moe_layer_destroy",
    "moe_quantized_bytes", "moe_quantize", "mtp_verify_accept_workspace_bytes",
    "mtp_verify_accept", "mtp_verify_accept_noalloc", "moe_forward_residual", "moe_lm_head_create",
    "moe_lm_head_forward", "moe_lm_head_destroy", "mtp_round_workspace_bytes", "mtp_round", "moe_last_error",
    "moe_layer_timeline", "moe_layer_inject_timeout", "moe_lm_head_status", "moe_forward_f32",
    "mtp_round_hidden", "moe_forward_resnorm",
)

# event names of moe_layer_timeline, in order
TIMELINE = ("entry", "start", "x_records", "router_done", "routing_ready", "first_routed_issue",
            "first_routed_compute", "shared_gate_up_done", "last_gate_up_done", "first_down_issue",
            "queue_exhausted", "last_down_block", "last_combine", "first_exit", "last_exit", "combine_start",
            "combine_ready", "topk_done", "entries_done")


class MoeTensor(_c.Structure):
    _fields_ = [("fmt", _c.c_int32), ("reserved", _c.c_int32), ("rows", _c.c_int64),
                ("cols", _c.c_int64), ("data", _c.c_void_p), ("nbytes", _c.c_size_t)]


class MoeLayerDesc(_c.Structure):
    _fields_ = [("H", _c.c_int32), ("E", _c.c_int32), ("top_k", _c.c_int32), ("I", _c.c_int32),
                ("I_shared", _c.c_int32), ("T_max", _c.c_int32), ("act_dtype", _c.c_int32),
                ("wait_limit_us", _c.c_uint32), ("router_w", MoeTensor), ("router_b", MoeTensor),
                ("gate", _c.POINTER(MoeTensor)), ("up", _c.POINTER(MoeTensor)),
                ("down", _c.POINTER(MoeTensor)), ("sh_gate", MoeTensor), ("sh_up", MoeTensor),
                ("sh_down", MoeTensor), ("expert_begin", _c.c_int32), ("expert_count", _c.c_int32)]


class MoEError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"[{code}] {msg}")
        self.code = code


_lib = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise ImportError(f"CUDA library not built: {LIB} is missing")
        L = _c.CDLL(LIB)
        vp, i32, i64, sz = _c.c_void_p, _c.c_int32, _c.c_int64, _c.c_size_t
        sig = {
            "moe_layer_create": (_c.c_int, [_c.POINTER(MoeLayerDesc), vp, _c.POINTER(vp)]),
            "moe_forward": (_c.c_int, [vp, vp, i32, vp, vp]),
            "moe_get_routing": (_c.c_int, [vp, vp, vp, vp, vp, vp]),
            "moe_layer_status": (_c.c_int, [vp, vp]),
            "moe_layer_weight_bytes": (sz, [vp]),
            "moe_layer_workspace_bytes": (sz, [vp]),
            "moe_layer_destroy": (None, [vp]),
            "moe_quantized_bytes": (sz, [i32, i64, i64]),
            "moe_quantize": (_c.c_int, [i32, vp, i64, i64, vp, vp]),
            "mtp_verify_accept_workspace_bytes": (sz, [i32, i32]),
            "mtp_verify_accept": (_c.c_int, [vp, i32, vp, i32, vp, vp, vp, sz, vp]),
            "mtp_verify_accept_noalloc": (_c.c_int, [vp, i32, vp, i32, vp, vp, vp]),
            "moe_forward_residual": (_c.c_int, [vp, vp, i32, vp, vp]),
            "moe_forward_f32": (_c.c_int, [vp, vp, i32, vp, vp]),
            "moe_lm_head_create": (_c.c_int, [_c.POINTER(MoeTensor), i32, i32, vp, _c.POINTER(vp)]),
            "moe_lm_head_forward": (_c.c_int, [vp, vp, i32, _c.c_float, vp, vp]),
            "moe_lm_head_destroy": (None, [vp]),
            "moe_lm_head_status": (_c.c_int, [vp, vp]),
            "mtp_round_workspace_bytes": (sz, [i32, i32, i32, i32]),
            "mtp_round": (_c.c_int, [_c.POINTER(vp), i32, _c.POINTER(vp), i32, vp, vp, vp, _c.c_float, _c.c_float,
                                     vp, sz, vp, vp, vp, vp, vp, vp, vp]),
            "moe_last_error": (_c.c_char_p, []),
            "moe_layer_timeline": (_c.c_int, [vp, _c.POINTER(i64), i32, vp]),
            "moe_layer_inject_timeout": (_c.c_int, [vp, i32]),
            "mtp_round_hidden": (_c.c_int, [vp, sz, i32, i32, i32, i32, i32, vp, vp]),
            "moe_forward_resnorm": (_c.c_int, [vp, vp, i32, vp, vp, vp, _c.c_float, vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(rc):
    if rc != MOE_OK:
        raise MoEError(rc, lib().moe_last_error().decode())
    return rc


def _require(cond, msg):
    """Argument checks that survive python -O (unlike assert)."""
    if not cond:
        raise MoEError(MOE_EINVAL, msg)


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def quantized_bytes(fmt, rows, cols):
    return lib().moe_quantized_bytes(fmt, rows, cols)


def quantize(fmt, w, out=None, stream=None):
    """fp32 [rows, cols] CUDA tensor -> serialised uint8 CUDA tensor."""
    import torch
    _require(w.is_cuda and w.dtype == torch.float32 and w.is_contiguous() and w.dim() == 2,
             "quantize: w must be a contiguous 2-D fp32 CUDA tensor")
    rows, cols = w.shape
    n = quantized_bytes(fmt, rows, cols)
    if n == 0:
        raise MoEError(MOE_EFORMAT, f"shape {tuple(w.shape)} does not fit format {fmt}")
    if out is None:
        out = torch.empty(n, dtype=torch.uint8, device=w.device)
    _check(lib().moe_quantize(fmt, w.data_ptr(), rows, cols, out.data_ptr(), _stream(stream)))
    return out


def _tensor(fmt, rows, cols, t):
    if t is None:
        return MoeTensor(fmt, 0, rows, cols, None, 0)
    return MoeTensor(fmt, 0, rows, cols, t.data_ptr(), t.numel() * t.element_size())


class Layer:
    """One MoE layer resident on the current CUDA device.

    experts: list of tuples (fmt, gate, up, down) of serialised byte tensors
    (host or device), one per routed expert held: all E, or the n experts
    from ``expert_begin`` on (one shard of an expert-parallel split); shared:
    one such tuple or None.  ``wait_limit_us`` bounds every device-side wait
    (0: the library's default).
    """

    def __init__(self, H, E, top_k, I, I_shared, T_max, act, router_w, router_b, experts, shared,
                 stream=None, expert_begin=0, wait_limit_us=0):
        self.H, self.E, self.top_k, self.I, self.I_shared = H, E, top_k, I, I_shared
        self.T_max, self.act = T_max, act
        n = len(experts)
        _require(n >= 1, "Layer: at least one routed expert must be held")
        self.expert_begin, self.expert_count = expert_begin, n
        gate = (MoeTensor * n)()
        up = (MoeTensor * n)()
        down = (MoeTensor * n)()
        for e, (fmt, g, u, d) in enumerate(experts):
            gate[e] = _tensor(fmt, I, H, g)
            up[e] = _tensor(fmt, I, H, u)
            down[e] = _tensor(fmt, H, I, d)
        desc = MoeLayerDesc()
        desc.H, desc.E, desc.top_k, desc.I, desc.I_shared = H, E, top_k, I, I_shared
        desc.T_max, desc.act_dtype, desc.wait_limit_us = T_max, act, wait_limit_us
        desc.expert_begin, desc.expert_count = expert_begin, (0 if (expert_begin == 0 and n == E) else n)
        desc.router_w = _tensor(FMT_F32, E, H, router_w)
        desc.router_b = _tensor(FMT_F32, 1, E, router_b)
        desc.gate, desc.up, desc.down = gate, up, down
        if shared is not None:
            sfmt, g, u, d = shared
            desc.sh_gate = _tensor(sfmt, I_shared, H, g)
            desc.sh_up = _tensor(sfmt, I_shared, H, u)
            desc.sh_down = _tensor(sfmt, H, I_shared, d)
        h = _c.c_void_p()
        _check(lib().moe_layer_create(_c.byref(desc), _stream(stream), _c.byref(h)))
        self.handle = h

    @property
    def weight_bytes(self):
        return lib().moe_layer_weight_bytes(self.handle)

    @property
    def workspace_bytes(self):
        return lib().moe_layer_workspace_bytes(self.handle)

    def forward(self, x, y=None, stream=None, residual=False, out_f32=False):
        """y = MoE(x), or x + MoE(x) with ``residual``; ``out_f32``: y in fp32
        whatever the act dtype (T <= 8)."""
        import torch
        T = x.shape[0]
        if y is None:
            y = torch.empty(x.shape, dtype=torch.float32, device=x.device) if out_f32 else torch.empty_like(x)
        _require(not (residual and out_f32), "forward: residual and out_f32 do not combine")
        f = lib().moe_forward_f32 if out_f32 else (lib().moe_forward_residual if residual else lib().moe_forward)
        _check(f(self.handle, x.data_ptr() if T else None, T, y.data_ptr() if T else None, _stream(stream)))
        return y

    def forward_resnorm(self, x, h_in, h_out=None, xn=None, eps=1e-6, stream=None):
        """One residual-stream step (``moe_forward_resnorm``): h_out = h_in +
        MoE(x) (fp32), xn = rmsnorm(h_out) (x's dtype).  Returns (h_out, xn)."""
        import torch
        T = x.shape[0]
        if h_out is None:
            h_out = torch.empty(h_in.shape, dtype=torch.float32, device=x.device)
        if xn is None:
            xn = torch.empty_like(x)
        _check(lib().moe_forward_resnorm(self.handle, x.data_ptr() if T else None, T,
                                         h_in.data_ptr() if T else None, h_out.data_ptr() if T else None,
                                         xn.data_ptr() if T else None, eps, _stream(stream)))
        return h_out, xn

    def routing(self, T, stream=None):
        """(ids [T,k] int32, gates [T,k] fp32, offsets [E+1] int32, perm [T*k] int32)."""
        import torch
        dev = torch.device("cuda")
        ids = torch.empty(T, self.top_k, dtype=torch.int32, device=dev)
        gates = torch.empty(T, self.top_k, dtype=torch.float32, device=dev)
        offs = torch.empty(self.E + 1, dtype=torch.int32, device=dev)
        perm = torch.empty(T * self.top_k, dtype=torch.int32, device=dev)
        _check(lib().moe_get_routing(self.handle, ids.data_ptr(), gates.data_ptr(), offs.data_ptr(),
                                     perm.data_ptr(), _stream(stream)))
        return ids, gates, offs, perm

    def timeline(self, stream=None):
        """Phase timeline of the last completed T <= 8 launch: {event: µs
        after the first block passed its dependency wait, or None}."""
        n = len(TIMELINE)
        buf = (_c.c_int64 * n)()
        _check(lib().moe_layer_timeline(self.handle, buf, n, _stream(stream)))
        return {name: (None if buf[i] < 0 and name != "entry" else buf[i] / 1e3)
                for i, name in enumerate(TIMELINE)}

    def inject_timeout(self, site=1):
        """Test hook: the next T <= 8 forward's routing wait runs out (see
        moe_layer_inject_timeout)."""
        _check(lib().moe_layer_inject_timeout(self.handle, site))

    def status(self, stream=None):
        """Raises MoEError(MOE_ETIMEOUT) if a device-side wait gave up."""
        _check(lib().moe_layer_status(self.handle, _stream(stream)))

    def close(self):
        if getattr(self, "handle", None):
            lib().moe_layer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def accept_workspace(k, V, device="cuda"):
    import torch
    n = lib().mtp_verify_accept_workspace_bytes(k, V)
    if n == 0:
        raise MoEError(MOE_EINVAL, f"k={k}, V={V} out of range")
    return torch.zeros((n + 15) // 16 * 16, dtype=torch.uint8, device=device)


def verify_accept(draft_ids, logits, workspace=None, out=None, stream=None):
    """Greedy acceptance; returns a device int32 tensor [n_accepted, next_token]."""
    import torch
    k = draft_ids.numel()
    V = logits.shape[1]
    _require(logits.dim() == 2 and logits.shape[0] == k + 1 and logits.dtype == torch.float32
             and logits.is_contiguous() and logits.is_cuda, "verify_accept: logits must be fp32 [k+1, V] on the GPU")
    _require(k == 0 or (draft_ids.dtype == torch.int32 and draft_ids.is_contiguous() and draft_ids.is_cuda),
             "verify_accept: draft_ids must be contiguous int32 on the GPU")
    if workspace is None:
        workspace = accept_workspace(k, V, logits.device)
    if out is None:
        out = torch.empty(2, dtype=torch.int32, device=logits.device)
    _check(lib().mtp_verify_accept(draft_ids.data_ptr() if k else None, k, logits.data_ptr(), V,
                                   out.data_ptr(), out.data_ptr() + 4, workspace.data_ptr(),
                                   workspace.numel(), _stream(stream)))
    return out


def verify_accept_noalloc(draft_ids, logits, out=None, stream=None):
    """Greedy acceptance through the entry point that uses the library's
    static scratch (no workspace); returns the device int32 tensor
    [n_accepted, next_token]."""
    import torch
    k = draft_ids.numel()
    V = logits.shape[1]
    _require(logits.dim() == 2 and logits.shape[0] == k + 1 and logits.dtype == torch.float32
             and logits.is_contiguous() and logits.is_cuda, "verify_accept: logits must be fp32 [k+1, V] on the GPU")
    _require(k == 0 or (draft_ids.dtype == torch.int32 and draft_ids.is_contiguous() and draft_ids.is_cuda),
             "verify_accept: draft_ids must be contiguous int32 on the GPU")
    if out is None:
        out = torch.empty(2, dtype=torch.int32, device=logits.device)
    _check(lib().mtp_verify_accept_noalloc(draft_ids.data_ptr() if k else None, k, logits.data_ptr(), V,
                                           out.data_ptr(), out.data_ptr() + 4, _stream(stream)))
    return out


class LmHead:
    """Output norm + Q8_0 LM head [V, H] on the current CUDA device; ``w`` is
    the serialised Q8_0 byte tensor (host or device)."""

    def __init__(self, w, V, H, T_max, act, stream=None):
        self.V, self.H, self.T_max, self.act = V, H, T_max, act
        t = _tensor(FMT_Q8_0, V, H, w)
        h = _c.c_void_p()
        _check(lib().moe_lm_head_create(_c.byref(t), T_max, act, _stream(stream), _c.byref(h)))
        self.handle = h

    def forward(self, x, eps=1e-6, out=None, stream=None):
        """fp32 logits [T, V] of rmsnorm(x)."""
        import torch
        T = x.shape[0]
        if out is None:
            out = torch.empty(T, self.V, dtype=torch.float32, device=x.device)
        _check(lib().moe_lm_head_forward(self.handle, x.data_ptr() if T else None, T, eps,
                                         out.data_ptr() if T else None, _stream(stream)))
        return out

    def status(self, stream=None):
        """Raises MoEError(MOE_ETIMEOUT) if a device-side wait gave up."""
        _check(lib().moe_lm_head_status(self.handle, _stream(stream)))

    def close(self):
        if getattr(self, "handle", None):
            lib().moe_lm_head_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def round_workspace(H, k, V, act, device="cuda"):
    import torch
    n = lib().mtp_round_workspace_bytes(H, k, V, act)
    if n == 0:
        raise MoEError(MOE_EINVAL, "mtp_round_workspace_bytes: arguments out of range")
    return torch.zeros(n + 256, dtype=torch.uint8, device=device)


def _aligned(buf, a=256):
    off = (-buf.data_ptr()) % a
    return buf.data_ptr() + off, buf.numel() - off


def mtp_round(layers, heads, lm, x, noise, eps=1e-6, p_min=0.0, workspace=None, head_out=True, stream=None):
    """One MTP draft/verify round (see ``mtp_round`` in moe_layer.h).  Returns
    a dict of device tensors: logits [k+1, V], draft_logits [k, V], drafts
    [k] (-1 past the confidence cut p_min), accept [n, next], head_out
    [k, k, H] (if requested)."""
    import torch
    k = len(heads)
    H, V = lm.H, lm.V
    dev = x.device
    if workspace is None:
        workspace = round_workspace(H, k, V, lm.act, dev)
    wp, wn = _aligned(workspace)
    logits = torch.empty(k + 1, V, dtype=torch.float32, device=dev)
    dlogits = torch.empty(k, V, dtype=torch.float32, device=dev)
    drafts = torch.empty(k, dtype=torch.int32, device=dev)
    acc = torch.empty(2, dtype=torch.int32, device=dev)
    hout = torch.empty(k, k, H, dtype=x.dtype, device=dev) if head_out else None
    tl = (_c.c_void_p * max(1, len(layers)))(*[L.handle.value for L in layers])
    hl = (_c.c_void_p * k)(*[L.handle.value for L in heads])
    _check(lib().mtp_round(tl, len(layers), hl, k, lm.handle, x.data_ptr(), noise.data_ptr(), eps, p_min, wp, wn,
                           logits.data_ptr(), dlogits.data_ptr(), hout.data_ptr() if hout is not None else None,
                           drafts.data_ptr(), acc.data_ptr(), acc.data_ptr() + 4, _stream(stream)))
    return dict(logits=logits, draft_logits=dlogits, drafts=drafts, accept=acc, head_out=hout, workspace=workspace)


def round_hidden(workspace, lm, k, n_target, stream=None):
    """The final residual rows h_n (fp32 [k+1, H]) of the last round run on
    ``workspace`` (``mtp_round_hidden``)."""
    import torch
    wp, wn = _aligned(workspace)
    h = torch.empty(k + 1, lm.H, dtype=torch.float32, device=workspace.device)
    _check(lib().mtp_round_hidden(wp, wn, lm.H, k, lm.V, lm.act, n_target, h.data_ptr(), _stream(stream)))
    return h
