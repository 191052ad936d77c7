"""GB300 (sm_103a) W1.58A8 BitLinear: RMSNorm -> per-token int8 absmax quant ->
I2_S ternary matmul -> fp32 rescale, as hand-written CUDA behind a C ABI.

This module is a thin ctypes binding of ``libbitnet_gb300.so`` (include/bitnet.h):
it checks tensor dtypes/devices, passes raw device pointers and the current CUDA
stream, and raises on a non-zero status.  Every step of the projection runs in
the library's kernels; there is no fallback path.  PyTorch only supplies device
memory and streams.
"""
from __future__ import annotations

import ctypes
import os

from . import build_lib

__all__ = [
    "BitnetError", "lib", "packed_bytes", "pack_i2s", "unpack_i2s", "rmsnorm_quant_a8", "i2s_gemm",
    "bitlinear_forward", "bitlinear_forward_group", "last_device_status", "status_string",
    "FLAG_WEIGHTS_STATIC", "MAX_GROUP", "EXPORTED_FUNCTIONS", "bitlinear_forward_noalloc",
    "selftest_bounded_wait", "glu", "glu_rmsnorm_quant_a8", "bitlinear_forward_glu", "ACT_SILU", "ACT_GELU_TANH",
    "bitlinear_forward_typed", "DTYPE_F32", "DTYPE_F16", "DTYPE_BF16", "head_rmsnorm", "bitlinear_forward_qk",
]

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED_SHAPE = 2
ERR_MISALIGNED = 3
ERR_CUDA = 4
ERR_TIMEOUT = 5
ERR_NO_DEVICE = 6
ERR_SCRATCH_LIMIT = 7
NOALLOC_SCRATCH_BYTES = 16 << 20
FLAG_WEIGHTS_STATIC = 1
MAX_GROUP = 16
ACT_SILU = 1
ACT_GELU_TANH = 2
DTYPE_F32 = 0
DTYPE_F16 = 1
DTYPE_BF16 = 2

EXPORTED_FUNCTIONS = (
    "bitnet_i2s_packed_bytes", "bitnet_pack_i2s", "bitnet_unpack_i2s", "bitnet_rmsnorm_quant_a8",
    "bitnet_i2s_gemm", "bitnet_bitlinear_forward", "bitnet_bitlinear_forward_group",
    "bitnet_status_string", "bitnet_last_device_status", "bitnet_bitlinear_forward_noalloc",
    "bitnet_selftest_bounded_wait", "bitnet_glu", "bitnet_glu_rmsnorm_quant_a8", "bitnet_bitlinear_forward_glu",
    "bitnet_bitlinear_forward_typed", "bitnet_head_rmsnorm", "bitnet_bitlinear_forward_qk",
)


class BitnetError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class Projection(ctypes.Structure):
    """Mirror of bitnet_projection."""
    _fields_ = [
        ("x", ctypes.c_void_p), ("norm_w", ctypes.c_void_p), ("packed_w", ctypes.c_void_p),
        ("w_scale", ctypes.c_float), ("K", ctypes.c_int64), ("N", ctypes.c_int64), ("y", ctypes.c_void_p),
    ]


_lib = None


def lib(build: bool = False) -> ctypes.CDLL:
    """The loaded library (built first when `build` is true or it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    path = build_lib.LIB_PATH
    if build or not os.path.exists(path):
        path = build_lib.build()
    L = ctypes.CDLL(path)
    vp, i64, f32, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int32
    L.bitnet_i2s_packed_bytes.restype = ctypes.c_size_t
    L.bitnet_i2s_packed_bytes.argtypes = [i64, i64]
    L.bitnet_pack_i2s.restype = ctypes.c_int
    L.bitnet_pack_i2s.argtypes = [vp, i64, i64, vp, vp, vp]
    L.bitnet_unpack_i2s.restype = ctypes.c_int
    L.bitnet_unpack_i2s.argtypes = [vp, i64, i64, vp, vp]
    L.bitnet_rmsnorm_quant_a8.restype = ctypes.c_int
    L.bitnet_rmsnorm_quant_a8.argtypes = [vp, vp, i64, i64, f32, vp, vp, vp, vp, vp]
    L.bitnet_i2s_gemm.restype = ctypes.c_int
    L.bitnet_i2s_gemm.argtypes = [vp, vp, vp, f32, i64, i64, i64, vp, vp, vp]
    L.bitnet_bitlinear_forward.restype = ctypes.c_int
    L.bitnet_bitlinear_forward.argtypes = [vp, vp, vp, f32, i64, i64, i64, f32, vp, vp]
    L.bitnet_bitlinear_forward_group.restype = ctypes.c_int
    L.bitnet_bitlinear_forward_group.argtypes = [ctypes.POINTER(Projection), i32, i64, f32, ctypes.c_uint32, vp]
    L.bitnet_bitlinear_forward_noalloc.restype = ctypes.c_int
    L.bitnet_bitlinear_forward_noalloc.argtypes = [vp, vp, vp, f32, i64, i64, i64, f32, vp, vp]
    L.bitnet_status_string.restype = ctypes.c_char_p
    L.bitnet_status_string.argtypes = [ctypes.c_int]
    L.bitnet_last_device_status.restype = ctypes.c_int
    L.bitnet_last_device_status.argtypes = [vp]
    L.bitnet_selftest_bounded_wait.restype = ctypes.c_int
    L.bitnet_selftest_bounded_wait.argtypes = [vp]
    L.bitnet_glu.restype = ctypes.c_int
    L.bitnet_glu.argtypes = [vp, vp, ctypes.c_int, i64, vp, vp]
    L.bitnet_glu_rmsnorm_quant_a8.restype = ctypes.c_int
    L.bitnet_glu_rmsnorm_quant_a8.argtypes = [vp, vp, ctypes.c_int, vp, i64, i64, f32, vp, vp, vp, vp, vp]
    L.bitnet_bitlinear_forward_glu.restype = ctypes.c_int
    L.bitnet_bitlinear_forward_glu.argtypes = [vp, vp, ctypes.c_int, vp, vp, f32, i64, i64, i64, f32, vp, vp]
    L.bitnet_head_rmsnorm.restype = ctypes.c_int
    L.bitnet_head_rmsnorm.argtypes = [vp, i64, i64, i64, vp, f32, vp, vp]
    L.bitnet_bitlinear_forward_qk.restype = ctypes.c_int
    L.bitnet_bitlinear_forward_qk.argtypes = [vp, vp, vp, f32, i64, i64, i64, f32, i64, vp, vp, vp]
    L.bitnet_bitlinear_forward_typed.restype = ctypes.c_int
    L.bitnet_bitlinear_forward_typed.argtypes = [vp, ctypes.c_int, vp, ctypes.c_int, vp, f32, i64, i64, i64, f32, vp,
                                                 ctypes.c_int, vp]
    _lib = L
    return L


def status_string(status: int) -> str:
    return lib().bitnet_status_string(int(status)).decode()


def _check(rc: int, where: str) -> None:
    if rc != OK:
        raise BitnetError(rc, where)


def _stream(stream):
    import torch

    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t, dtype, name):
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _opt(t, dtype, name):
    return None if t is None else _dev(t, dtype, name)


def packed_bytes(N: int, K: int) -> int:
    return int(lib().bitnet_i2s_packed_bytes(N, K))


def pack_i2s(w, packed=None, stream=None, return_scale: bool = True):
    """Absmean-ternary quantise and I2_S-pack w[N, K] (fp32, CUDA).

    Returns (packed uint8 tensor, w_scale float) -- or (packed, None) when
    return_scale is False (then the call does not synchronise)."""
    import torch

    N, K = w.shape
    nbytes = packed_bytes(N, K)
    if nbytes == 0:
        raise BitnetError(ERR_UNSUPPORTED_SHAPE, "pack_i2s")
    if packed is None:
        packed = torch.empty(nbytes, dtype=torch.uint8, device=w.device)
    scale = ctypes.c_float(0.0)
    rc = lib().bitnet_pack_i2s(_dev(w, torch.float32, "w"), N, K, _dev(packed, torch.uint8, "packed"),
                               ctypes.byref(scale) if return_scale else None, _stream(stream))
    _check(rc, "bitnet_pack_i2s")
    return packed, (scale.value if return_scale else None)


def unpack_i2s(packed, N: int, K: int, out=None, stream=None):
    import torch

    if out is None:
        out = torch.empty((N, K), dtype=torch.int8, device=packed.device)
    rc = lib().bitnet_unpack_i2s(_dev(packed, torch.uint8, "packed"), N, K, _dev(out, torch.int8, "out"),
                                 _stream(stream))
    _check(rc, "bitnet_unpack_i2s")
    return out


def rmsnorm_quant_a8(x, norm_w, eps: float = 1e-6, codes=None, a_scale=None, rowsum=None, xn_out=None,
                     stream=None):
    """Returns (codes int8 [M,K], a_scale f32 [M], rowsum int32 [M] or None)."""
    import torch

    M, K = x.shape
    if codes is None:
        codes = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if a_scale is None:
        a_scale = torch.empty(M, dtype=torch.float32, device=x.device)
    rc = lib().bitnet_rmsnorm_quant_a8(
        _dev(x, torch.float32, "x"), _dev(norm_w, torch.float32, "norm_w"), M, K, float(eps),
        _dev(codes, torch.int8, "codes"), _dev(a_scale, torch.float32, "a_scale"),
        _opt(rowsum, torch.int32, "rowsum"), _opt(xn_out, torch.float32, "xn_out"), _stream(stream))
    _check(rc, "bitnet_rmsnorm_quant_a8")
    return codes, a_scale, rowsum


def i2s_gemm(codes, a_scale, packed_w, w_scale: float, N: int, y=None, acc_out=None, stream=None):
    import torch

    M, K = codes.shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=codes.device)
    rc = lib().bitnet_i2s_gemm(
        _dev(codes, torch.int8, "codes"), _dev(a_scale, torch.float32, "a_scale"),
        _dev(packed_w, torch.uint8, "packed_w"), float(w_scale), M, K, N, _dev(y, torch.float32, "y"),
        _opt(acc_out, torch.int32, "acc_out"), _stream(stream))
    _check(rc, "bitnet_i2s_gemm")
    return y


def bitlinear_forward(x, norm_w, packed_w, w_scale: float, N: int, eps: float = 1e-6, y=None, stream=None):
    import torch

    M, K = x.shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    rc = lib().bitnet_bitlinear_forward(
        _dev(x, torch.float32, "x"), _dev(norm_w, torch.float32, "norm_w"),
        _dev(packed_w, torch.uint8, "packed_w"), float(w_scale), M, K, N, float(eps),
        _dev(y, torch.float32, "y"), _stream(stream))
    _check(rc, "bitnet_bitlinear_forward")
    return y


def _dtype_code(t, name, allowed):
    import torch

    codes = {torch.float32: DTYPE_F32, torch.float16: DTYPE_F16, torch.bfloat16: DTYPE_BF16}
    if t.dtype not in codes or codes[t.dtype] not in allowed:
        raise TypeError(f"{name}: unsupported dtype {t.dtype}")
    return codes[t.dtype]


def bitlinear_forward_typed(x, norm_w, packed_w, w_scale: float, N: int, eps: float = 1e-6, y=None,
                            y_dtype=None, stream=None):
    """bitlinear_forward with x in float32/float16/bfloat16, norm_w in float32/float16
    and y in float32/float16/bfloat16 (default: x's dtype).  y is the fp32 result of
    the widened inputs, rounded once to y's dtype."""
    import torch

    M, K = x.shape
    if y is None:
        y = torch.empty((M, N), dtype=y_dtype if y_dtype is not None else x.dtype, device=x.device)
    xt = _dtype_code(x, "x", (DTYPE_F32, DTYPE_F16, DTYPE_BF16))
    gt = _dtype_code(norm_w, "norm_w", (DTYPE_F32, DTYPE_F16))
    yt = _dtype_code(y, "y", (DTYPE_F32, DTYPE_F16, DTYPE_BF16))
    rc = lib().bitnet_bitlinear_forward_typed(
        _dev(x, x.dtype, "x"), xt, _dev(norm_w, norm_w.dtype, "norm_w"), gt, _dev(packed_w, torch.uint8, "packed_w"),
        float(w_scale), M, K, N, float(eps), _dev(y, y.dtype, "y"), yt, _stream(stream))
    _check(rc, "bitnet_bitlinear_forward_typed")
    return y


def head_rmsnorm(y, head_dim: int, head_w, eps: float = 1e-6, out=None, stream=None):
    """Per-head RMSNorm of y[M, N] (heads of head_dim consecutive values) times
    head_w[head_dim]; out=y works in place."""
    import torch

    M, N = y.shape
    if out is None:
        out = torch.empty_like(y)
    rc = lib().bitnet_head_rmsnorm(_dev(y, torch.float32, "y"), M, N, int(head_dim),
                                   _dev(head_w, torch.float32, "head_w"), float(eps), _dev(out, torch.float32, "out"),
                                   _stream(stream))
    _check(rc, "bitnet_head_rmsnorm")
    return out


def bitlinear_forward_qk(x, norm_w, packed_w, w_scale: float, N: int, head_dim: int, head_w, eps: float = 1e-6,
                         y=None, stream=None):
    """The q/k projection followed by its head norm."""
    import torch

    M, K = x.shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    rc = lib().bitnet_bitlinear_forward_qk(
        _dev(x, torch.float32, "x"), _dev(norm_w, torch.float32, "norm_w"), _dev(packed_w, torch.uint8, "packed_w"),
        float(w_scale), M, K, N, float(eps), int(head_dim), _dev(head_w, torch.float32, "head_w"),
        _dev(y, torch.float32, "y"), _stream(stream))
    _check(rc, "bitnet_bitlinear_forward_qk")
    return y


def glu(gate, up, act: int, h=None, stream=None):
    """h = act(gate) * up elementwise (the down projection's input)."""
    import torch

    if gate.shape != up.shape:
        raise ValueError("glu: gate and up differ in shape")
    if h is None:
        h = torch.empty_like(gate)
    rc = lib().bitnet_glu(_dev(gate, torch.float32, "gate"), _dev(up, torch.float32, "up"), int(act), gate.numel(),
                          _dev(h, torch.float32, "h"), _stream(stream))
    _check(rc, "bitnet_glu")
    return h


def glu_rmsnorm_quant_a8(gate, up, act: int, norm_w, eps: float = 1e-6, codes=None, a_scale=None, rowsum=None,
                         xn_out=None, stream=None):
    """rmsnorm_quant_a8 of act(gate) * up (K <= 3072).  Returns (codes, a_scale, rowsum)."""
    import torch

    M, K = gate.shape
    if codes is None:
        codes = torch.empty((M, K), dtype=torch.int8, device=gate.device)
    if a_scale is None:
        a_scale = torch.empty(M, dtype=torch.float32, device=gate.device)
    rc = lib().bitnet_glu_rmsnorm_quant_a8(
        _dev(gate, torch.float32, "gate"), _dev(up, torch.float32, "up"), int(act),
        _dev(norm_w, torch.float32, "norm_w"), M, K, float(eps), _dev(codes, torch.int8, "codes"),
        _dev(a_scale, torch.float32, "a_scale"), _opt(rowsum, torch.int32, "rowsum"),
        _opt(xn_out, torch.float32, "xn_out"), _stream(stream))
    _check(rc, "bitnet_glu_rmsnorm_quant_a8")
    return codes, a_scale, rowsum


def bitlinear_forward_glu(gate, up, act: int, norm_w, packed_w, w_scale: float, N: int, eps: float = 1e-6, y=None,
                          stream=None):
    """The down projection: BitLinear(act(gate) * up)."""
    import torch

    M, K = gate.shape
    if up.shape != gate.shape:
        raise ValueError("bitlinear_forward_glu: gate and up differ in shape")
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=gate.device)
    rc = lib().bitnet_bitlinear_forward_glu(
        _dev(gate, torch.float32, "gate"), _dev(up, torch.float32, "up"), int(act),
        _dev(norm_w, torch.float32, "norm_w"), _dev(packed_w, torch.uint8, "packed_w"), float(w_scale), M, K, N,
        float(eps), _dev(y, torch.float32, "y"), _stream(stream))
    _check(rc, "bitnet_bitlinear_forward_glu")
    return y


def bitlinear_forward_noalloc(x, norm_w, packed_w, w_scale: float, N: int, eps: float = 1e-6, y=None,
                              stream=None):
    """bitlinear_forward without any allocation inside the library (the
    temporary data lives in a fixed 16 MiB device array; see bitnet.h).  `y`
    must be supplied by callers that cannot allocate."""
    import torch

    M, K = x.shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    rc = lib().bitnet_bitlinear_forward_noalloc(
        _dev(x, torch.float32, "x"), _dev(norm_w, torch.float32, "norm_w"),
        _dev(packed_w, torch.uint8, "packed_w"), float(w_scale), M, K, N, float(eps),
        _dev(y, torch.float32, "y"), _stream(stream))
    _check(rc, "bitnet_bitlinear_forward_noalloc")
    return y


def make_group(projs):
    """projs: sequence of (x, norm_w, packed_w, w_scale, N, y).  Returns the
    ctypes descriptor array (reusable across calls with the same buffers)."""
    import torch

    arr = (Projection * len(projs))()
    for i, (x, g, pw, ws, N, y) in enumerate(projs):
        arr[i].x = _dev(x, torch.float32, "x").value
        arr[i].norm_w = _dev(g, torch.float32, "norm_w").value
        arr[i].packed_w = _dev(pw, torch.uint8, "packed_w").value
        arr[i].w_scale = float(ws)
        arr[i].K = x.shape[1]
        arr[i].N = int(N)
        arr[i].y = _dev(y, torch.float32, "y").value
    return arr


def bitlinear_forward_group(group, M: int, eps: float = 1e-6, flags: int = 0, stream=None):
    """Run a descriptor array from make_group (or a sequence accepted by it)."""
    if not isinstance(group, ctypes.Array):
        group = make_group(group)
    rc = lib().bitnet_bitlinear_forward_group(group, len(group), int(M), float(eps), int(flags), _stream(stream))
    _check(rc, "bitnet_bitlinear_forward_group")


def last_device_status(stream=None) -> int:
    return int(lib().bitnet_last_device_status(_stream(stream)))


def selftest_bounded_wait(stream=None) -> None:
    """Runs the library's bounded wait against a barrier nothing completes (about
    one second); afterwards last_device_status() reports ERR_TIMEOUT."""
    _check(lib().bitnet_selftest_bounded_wait(_stream(stream)), "bitnet_selftest_bounded_wait")
