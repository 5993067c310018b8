"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function the header declares, sizes its formats and rejects bad
arguments before touching a device."""
import ctypes
import os
import re

import pytest

import block_quantized_moe_layer_gb300 as pkg

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "moe_layer.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", src, flags=re.M))


@pytest.fixture(scope="module")
def lib():
    from block_quantized_moe_layer_gb300 import _build
    _build.build()
    return pkg.lib()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"moe_layer_create", "moe_forward", "mtp_verify_accept"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert names == set(pkg.EXPORTS)


def test_quantized_sizes(lib):
    assert lib.moe_quantized_bytes(pkg.FMT_Q8_0, 1280, 4096) == 1280 * 128 * 34 == 5_570_560
    assert lib.moe_quantized_bytes(pkg.FMT_Q4KS, 1280, 4096) == 1280 * 16 * 144 == 2_949_120
    assert lib.moe_quantized_bytes(pkg.FMT_Q8_0, 4, 33) == 0
    assert lib.moe_quantized_bytes(pkg.FMT_Q4KS, 4, 128) == 0
    assert lib.moe_quantized_bytes(pkg.FMT_F32, 4, 128) == 0


def test_accept_workspace_sizes(lib):
    assert lib.mtp_verify_accept_workspace_bytes(3, 32768) > 16
    assert lib.mtp_verify_accept_workspace_bytes(16, 10) == 0
    assert lib.mtp_verify_accept_workspace_bytes(3, 0) == 0


def test_bad_arguments_rejected_on_host(lib):
    out = ctypes.c_void_p()
    assert lib.moe_layer_create(None, None, ctypes.byref(out)) == pkg.MOE_EINVAL
    assert lib.moe_forward(None, None, 4, None, None) == pkg.MOE_EINVAL
    assert b"NULL" in lib.moe_last_error()
    d = pkg.MoeLayerDesc()
    d.H, d.E, d.top_k, d.I, d.T_max = 300, 16, 2, 128, 4  # H not a multiple of 256
    assert lib.moe_layer_create(ctypes.byref(d), None, ctypes.byref(out)) == pkg.MOE_EINVAL
    d.H, d.top_k = 256, 17
    assert lib.moe_layer_create(ctypes.byref(d), None, ctypes.byref(out)) == pkg.MOE_EINVAL
    d.top_k, d.T_max = 2, 0
    assert lib.moe_layer_create(ctypes.byref(d), None, ctypes.byref(out)) == pkg.MOE_EINVAL
    assert lib.mtp_verify_accept(None, 3, None, 100, None, None, None, 0, None) == pkg.MOE_EINVAL
    assert lib.mtp_verify_accept(None, 16, None, 100, None, None, None, 0, None) == pkg.MOE_EINVAL
    assert lib.moe_quantize(7, None, 1, 32, None, None) == pkg.MOE_EFORMAT
    assert lib.moe_quantize(pkg.FMT_Q8_0, None, 1, 32, None, None) == pkg.MOE_EINVAL
    assert out.value is None


def test_mtp_entry_points_reject_bad_arguments_on_host(lib):
    # workspace sizing: k outside 1..7, V outside 1..2^24, unknown act dtype
    assert lib.mtp_round_workspace_bytes(4096, 3, 32768, pkg.ACT_BF16) > 0
    assert lib.mtp_round_workspace_bytes(4096, 0, 32768, pkg.ACT_BF16) == 0
    assert lib.mtp_round_workspace_bytes(4096, 8, 32768, pkg.ACT_BF16) == 0
    assert lib.mtp_round_workspace_bytes(4096, 3, 0, pkg.ACT_BF16) == 0
    assert lib.mtp_round_workspace_bytes(4096, 3, 32768, 7) == 0
    # the round: k outside 1..7, then NULL arguments, before any device work
    assert lib.mtp_round(None, 0, None, 0, None, None, None, 1e-6, 0.0, None, 0, None, None, None, None, None,
                         None, None) == pkg.MOE_EINVAL
    assert b"k outside" in lib.moe_last_error()
    assert lib.mtp_round(None, 0, None, 3, None, None, None, 1e-6, 0.0, None, 0, None, None, None, None, None,
                         None, None) == pkg.MOE_EINVAL
    assert b"NULL" in lib.moe_last_error()
    # the LM head: NULL, wrong format, shape and T_max checks
    out = ctypes.c_void_p()
    assert lib.moe_lm_head_create(None, 4, pkg.ACT_BF16, None, ctypes.byref(out)) == pkg.MOE_EINVAL
    t = pkg.MoeTensor()
    t.fmt, t.rows, t.cols = pkg.FMT_Q4KS, 1000, 4096
    assert lib.moe_lm_head_create(ctypes.byref(t), 4, pkg.ACT_BF16, None, ctypes.byref(out)) == pkg.MOE_EFORMAT
    t.fmt, t.cols = pkg.FMT_Q8_0, 4000  # H not a multiple of 512
    assert lib.moe_lm_head_create(ctypes.byref(t), 4, pkg.ACT_BF16, None, ctypes.byref(out)) == pkg.MOE_EINVAL
    t.cols = 4096
    assert lib.moe_lm_head_create(ctypes.byref(t), 9, pkg.ACT_BF16, None, ctypes.byref(out)) == pkg.MOE_EINVAL
    assert lib.moe_lm_head_create(ctypes.byref(t), 4, pkg.ACT_BF16, None, ctypes.byref(out)) == pkg.MOE_EINVAL
    assert b"nbytes" in lib.moe_last_error()  # data NULL
    assert out.value is None
    assert lib.moe_lm_head_forward(None, None, 4, 1e-6, None, None) == pkg.MOE_EINVAL
    assert lib.moe_forward_residual(None, None, 4, None, None) == pkg.MOE_EINVAL


def test_binding_rejects_bad_tensors_before_any_launch():
    import torch
    with pytest.raises(pkg.MoEError):  # logits on the host
        pkg.verify_accept(torch.zeros(3, dtype=torch.int32), torch.zeros(4, 10))
    with pytest.raises(pkg.MoEError):  # [k+1, V] mismatch
        pkg.verify_accept_noalloc(torch.zeros(3, dtype=torch.int32), torch.zeros(3, 10))
    with pytest.raises(pkg.MoEError):  # not a CUDA fp32 matrix
        pkg.quantize(pkg.FMT_Q8_0, torch.zeros(4, 32))
