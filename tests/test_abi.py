"""The C-ABI library builds, loads and exports every symbol bitnet.h declares;
host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

import bitlinear_rmsnorm_token_gb300 as bn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bitnet.h")


@pytest.fixture(scope="module")
def L():
    return bn.lib(build=True)


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"BITNET_API\s+[\w\s\*]*?\b(bitnet_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for want in ("bitnet_pack_i2s", "bitnet_rmsnorm_quant_a8", "bitnet_i2s_gemm", "bitnet_bitlinear_forward"):
        assert want in names
    assert set(bn.EXPORTED_FUNCTIONS) <= set(names)


def test_every_declared_symbol_is_exported(L):
    for name in _declared():
        assert hasattr(L, name), name


def test_packed_bytes(L):
    assert L.bitnet_i2s_packed_bytes(2048, 1024) == 2048 * 1024 // 4 + 4
    assert L.bitnet_i2s_packed_bytes(1, 128) == 36
    assert L.bitnet_i2s_packed_bytes(3, 100) == 0
    assert L.bitnet_i2s_packed_bytes(0, 128) == 0
    assert L.bitnet_i2s_packed_bytes(5, 0) == 0


def test_status_strings(L):
    for code in range(7):
        assert L.bitnet_status_string(code)
    assert b"unknown" in L.bitnet_status_string(99)


# Argument errors are reported before any CUDA call, so these run without a GPU.
FAKE = ctypes.c_void_p(1 << 20)          # 16-byte aligned, never dereferenced
ODD = ctypes.c_void_p((1 << 20) + 4)     # not 16-byte aligned


def test_forward_argument_errors(L):
    f = L.bitnet_bitlinear_forward
    assert f(None, FAKE, FAKE, 1.0, 1, 128, 1, 1e-6, FAKE, None) == bn.ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, 1.0, 0, 128, 1, 1e-6, FAKE, None) == bn.ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, 1.0, 1, 128, 0, 1e-6, FAKE, None) == bn.ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, 1.0, 1, 100, 1, 1e-6, FAKE, None) == bn.ERR_UNSUPPORTED_SHAPE
    assert f(FAKE, FAKE, FAKE, 1.0, 1, 0, 1, 1e-6, FAKE, None) == bn.ERR_UNSUPPORTED_SHAPE
    assert f(FAKE, FAKE, FAKE, 1.0, 1, 65536 + 128, 1, 1e-6, FAKE, None) == bn.ERR_UNSUPPORTED_SHAPE
    assert f(FAKE, FAKE, FAKE, 1.0, 1, 128, 1, 0.0, FAKE, None) == bn.ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, 0.0, 1, 128, 1, 1e-6, FAKE, None) == bn.ERR_INVALID_ARG
    assert f(ODD, FAKE, FAKE, 1.0, 1, 128, 1, 1e-6, FAKE, None) == bn.ERR_MISALIGNED
    assert f(FAKE, FAKE, ODD, 1.0, 1, 128, 1, 1e-6, FAKE, None) == bn.ERR_MISALIGNED


def test_other_entry_point_argument_errors(L):
    assert L.bitnet_pack_i2s(None, 1, 128, FAKE, None, None) == bn.ERR_INVALID_ARG
    assert L.bitnet_pack_i2s(FAKE, 1, 96, FAKE, None, None) == bn.ERR_UNSUPPORTED_SHAPE
    assert L.bitnet_pack_i2s(FAKE, 1, 128, ODD, None, None) == bn.ERR_MISALIGNED
    assert L.bitnet_unpack_i2s(FAKE, 0, 128, FAKE, None) == bn.ERR_INVALID_ARG
    assert L.bitnet_rmsnorm_quant_a8(FAKE, FAKE, 4, 130, 1e-6, FAKE, FAKE, None, None, None) == \
        bn.ERR_UNSUPPORTED_SHAPE
    assert L.bitnet_rmsnorm_quant_a8(FAKE, FAKE, 4, 128, -1.0, FAKE, FAKE, None, None, None) == bn.ERR_INVALID_ARG
    assert L.bitnet_i2s_gemm(FAKE, FAKE, FAKE, 1.0, 4, 128, 4, None, None, None) == bn.ERR_INVALID_ARG
    assert L.bitnet_i2s_gemm(FAKE, FAKE, FAKE, 1.0, 4, 128, 4, ODD, None, None) == bn.ERR_MISALIGNED


def test_group_argument_errors(L):
    P = bn.Projection
    arr = (P * 2)()
    for i in range(2):
        arr[i].x = arr[i].norm_w = arr[i].packed_w = arr[i].y = FAKE.value
        arr[i].w_scale = 1.0
        arr[i].K = 1024
        arr[i].N = 64
    g = L.bitnet_bitlinear_forward_group
    assert g(arr, 0, 1, 1e-6, 0, None) == bn.ERR_INVALID_ARG
    assert g(arr, 17, 1, 1e-6, 0, None) == bn.ERR_INVALID_ARG
    assert g(arr, 2, 1, 1e-6, 8, None) == bn.ERR_INVALID_ARG       # unknown flag
    assert g(arr, 2, 9, 1e-6, 0, None) == bn.ERR_UNSUPPORTED_SHAPE  # grouped path is for M <= 8
    arr[1].K = 1000
    assert g(arr, 2, 1, 1e-6, 0, None) == bn.ERR_UNSUPPORTED_SHAPE
    arr[1].K = 1024
    arr[1].y = ODD.value
    assert g(arr, 2, 1, 1e-6, 0, None) == bn.ERR_MISALIGNED


def test_glu_argument_errors(L):
    f = L.bitnet_bitlinear_forward_glu
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
                  ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
    assert f(FAKE, FAKE, 0, FAKE, FAKE, 1.0, 1, 128, 1, 1e-6, FAKE, None) == bn.ERR_INVALID_ARG  # no activation
    assert f(FAKE, FAKE, 3, FAKE, FAKE, 1.0, 1, 128, 1, 1e-6, FAKE, None) == bn.ERR_INVALID_ARG  # unknown one
    assert f(FAKE, None, 1, FAKE, FAKE, 1.0, 1, 128, 1, 1e-6, FAKE, None) == bn.ERR_INVALID_ARG  # no up
    assert f(FAKE, ODD, 1, FAKE, FAKE, 1.0, 1, 128, 1, 1e-6, FAKE, None) == bn.ERR_MISALIGNED
    assert f(FAKE, FAKE, 2, FAKE, FAKE, 1.0, 1, 100, 1, 1e-6, FAKE, None) == bn.ERR_UNSUPPORTED_SHAPE
    g = L.bitnet_glu
    g.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    assert g(FAKE, FAKE, 1, 6, FAKE, None) == bn.ERR_INVALID_ARG     # not a multiple of 4
    assert g(FAKE, FAKE, 7, 8, FAKE, None) == bn.ERR_INVALID_ARG     # unknown activation
    assert g(FAKE, ODD, 1, 8, FAKE, None) == bn.ERR_MISALIGNED
    q = L.bitnet_glu_rmsnorm_quant_a8
    q.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert q(FAKE, FAKE, 1, FAKE, 4, 4096, 1e-6, FAKE, FAKE, None, None, None) == bn.ERR_UNSUPPORTED_SHAPE


def test_typed_forward_argument_errors(L):
    f = L.bitnet_bitlinear_forward_typed
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_float,
                  ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int,
                  ctypes.c_void_p]
    assert bn.DTYPE_F32 == 0 and bn.DTYPE_F16 == 1 and bn.DTYPE_BF16 == 2  # the header's values
    assert f(None, 2, FAKE, 0, FAKE, 1.0, 1, 128, 1, 1e-6, FAKE, 2, None) == bn.ERR_INVALID_ARG  # no x
    assert f(FAKE, 3, FAKE, 0, FAKE, 1.0, 1, 128, 1, 1e-6, FAKE, 2, None) == bn.ERR_INVALID_ARG  # unknown x type
    assert f(FAKE, 2, FAKE, 2, FAKE, 1.0, 1, 128, 1, 1e-6, FAKE, 2, None) == bn.ERR_INVALID_ARG  # bf16 norm weight
    assert f(FAKE, 2, FAKE, 1, FAKE, 1.0, 1, 128, 1, 1e-6, FAKE, -1, None) == bn.ERR_INVALID_ARG  # unknown y type
    assert f(FAKE, 2, FAKE, 1, FAKE, 1.0, 1, 128, 1, 0.0, FAKE, 1, None) == bn.ERR_INVALID_ARG    # eps = 0
    assert f(FAKE, 2, FAKE, 1, FAKE, 1.0, 1, 100, 1, 1e-6, FAKE, 1, None) == bn.ERR_UNSUPPORTED_SHAPE
    assert f(ODD, 2, FAKE, 1, FAKE, 1.0, 1, 128, 1, 1e-6, FAKE, 1, None) == bn.ERR_MISALIGNED


def test_head_norm_argument_errors(L):
    h = L.bitnet_head_rmsnorm
    h.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float,
                  ctypes.c_void_p, ctypes.c_void_p]
    assert h(None, 1, 256, 128, FAKE, 1e-6, FAKE, None) == bn.ERR_INVALID_ARG
    assert h(FAKE, 0, 256, 128, FAKE, 1e-6, FAKE, None) == bn.ERR_INVALID_ARG
    assert h(FAKE, 1, 256, 128, FAKE, 0.0, FAKE, None) == bn.ERR_INVALID_ARG
    assert h(FAKE, 1, 256, 64, FAKE, 1e-6, FAKE, None) == bn.ERR_UNSUPPORTED_SHAPE   # head_dim not a multiple of 128
    assert h(FAKE, 1, 384, 256, FAKE, 1e-6, FAKE, None) == bn.ERR_UNSUPPORTED_SHAPE  # does not divide N
    assert h(FAKE, 1, 256, 128, ODD, 1e-6, FAKE, None) == bn.ERR_MISALIGNED
    q = L.bitnet_bitlinear_forward_qk
    q.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_int64, ctypes.c_float, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert q(FAKE, FAKE, FAKE, 1.0, 1, 128, 256, 1e-6, 128, None, FAKE, None) == bn.ERR_INVALID_ARG
    assert q(FAKE, FAKE, FAKE, 1.0, 1, 128, 200, 1e-6, 128, FAKE, FAKE, None) == bn.ERR_UNSUPPORTED_SHAPE
    assert q(FAKE, FAKE, FAKE, 1.0, 1, 128, 256, 1e-6, 128, ODD, FAKE, None) == bn.ERR_MISALIGNED
    assert q(None, FAKE, FAKE, 1.0, 1, 128, 256, 1e-6, 128, FAKE, FAKE, None) == bn.ERR_INVALID_ARG


def test_typed_binding_rejects_unsupported_dtypes():
    """The binding checks element types before it touches a device."""
    import torch

    x = torch.zeros((2, 128), dtype=torch.bfloat16)
    packed = torch.zeros(4 * 32 + 4, dtype=torch.uint8)
    with pytest.raises(TypeError):  # bf16 norm weights are not a supported type
        bn.bitlinear_forward_typed(x, torch.zeros(128, dtype=torch.bfloat16), packed, 1.0, 4)
    with pytest.raises(TypeError):  # nor are float64 activations
        bn.bitlinear_forward_typed(x.double(), torch.zeros(128), packed, 1.0, 4)
    with pytest.raises(TypeError):  # nor an int8 output
        bn.bitlinear_forward_typed(x, torch.zeros(128), packed, 1.0, 4, y=torch.zeros((2, 4), dtype=torch.int8))
