"""CPU oracle for the W1.58A8 BitLinear projection -- TEST INFRASTRUCTURE ONLY.

Thin numpy/ctypes wrapper over ``bitnet_oracle.c`` (plain C; OpenMP over
independent rows, and over (row, column) pairs in the contraction).
Only ``tests/``, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline leg use
it; the CUDA library never does.  The C file cites, per function, the passage of
the pages it restates.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bitnet_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libbitnet_oracle.so")
_lib = None

_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i8p = np.ctypeslib.ndpointer(dtype=np.int8, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    lib.oracle_mean_abs.restype = ctypes.c_double
    lib.oracle_mean_abs.argtypes = [_f32p, _i64]
    lib.oracle_weight_scale.restype = ctypes.c_float
    lib.oracle_weight_scale.argtypes = [_f32p, _i64]
    lib.oracle_quantize_ternary.restype = None
    lib.oracle_quantize_ternary.argtypes = [_f32p, _i64, ctypes.c_float, _i8p]
    lib.oracle_encode_i2s.restype = ctypes.c_int
    lib.oracle_encode_i2s.argtypes = [_i8p, _i64, _i64, ctypes.c_float, _u8p]
    lib.oracle_pack_i2s_with_scale.restype = ctypes.c_int
    lib.oracle_pack_i2s_with_scale.argtypes = [_f32p, _i64, _i64, ctypes.c_float, _u8p]
    lib.oracle_pack_i2s.restype = ctypes.c_int
    lib.oracle_pack_i2s.argtypes = [_f32p, _i64, _i64, _u8p, ctypes.POINTER(ctypes.c_float)]
    lib.oracle_unpack_i2s.restype = ctypes.c_int
    lib.oracle_unpack_i2s.argtypes = [_u8p, _i64, _i64, _i8p]
    lib.oracle_count_invalid_codes.restype = ctypes.c_int64
    lib.oracle_count_invalid_codes.argtypes = [_u8p, _i64, _i64]
    lib.oracle_rmsnorm.restype = None
    lib.oracle_rmsnorm.argtypes = [_f32p, _f32p, _i64, _i64, ctypes.c_float, _f32p, ctypes.c_void_p]
    lib.oracle_quant_a8.restype = None
    lib.oracle_quant_a8.argtypes = [_f32p, _i64, _i64, _i8p, _f32p, _i32p]
    lib.oracle_i2s_matmul.restype = ctypes.c_int
    lib.oracle_i2s_matmul.argtypes = [_i8p, _u8p, _i64, _i64, _i64, _i64p]
    lib.oracle_rescale.restype = None
    lib.oracle_rescale.argtypes = [_i64p, _f32p, ctypes.c_float, _i64, _i64, _f32p]
    lib.oracle_bitlinear_forward_rows.restype = ctypes.c_int
    lib.oracle_bitlinear_forward_rows.argtypes = [
        _f32p, _f32p, _u8p, ctypes.c_float, _i64, _i64, _i64, ctypes.c_float,
        ctypes.c_void_p, _i64, _f32p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p]
    lib.oracle_dequant_dot_f64.restype = None
    lib.oracle_dequant_dot_f64.argtypes = [_i8p, _i8p, _f32p, ctypes.c_float, _i64, _i64, _i64, _f64p]
    lib.oracle_activation.restype = ctypes.c_double
    lib.oracle_activation.argtypes = [ctypes.c_double, ctypes.c_int]
    lib.oracle_glu.restype = None
    lib.oracle_glu.argtypes = [_f32p, _f32p, _i64, ctypes.c_int, _f32p]
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_set_num_threads.restype = None
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    _lib = lib
    return lib


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def mean_abs(w) -> float:
    w = _f32(w).ravel()
    return float(_load().oracle_mean_abs(w, w.size))


def weight_scale(w) -> float:
    w = _f32(w).ravel()
    return float(_load().oracle_weight_scale(w, w.size))


def quantize_ternary(w, w_scale: float) -> np.ndarray:
    w = _f32(w)
    q = np.empty(w.shape, dtype=np.int8)
    _load().oracle_quantize_ternary(w.ravel(), w.size, ctypes.c_float(w_scale), q.reshape(-1))
    return q


def encode_i2s(q, w_scale: float) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.int8)
    N, K = q.shape
    out = np.empty(N * K // 4 + 4, dtype=np.uint8)
    rc = _load().oracle_encode_i2s(q, N, K, ctypes.c_float(w_scale), out)
    if rc:
        raise ValueError(f"encode_i2s: bad shape {q.shape}")
    return out


def pack_i2s(w, w_scale: float | None = None):
    """Return (packed bytes, w_scale) for w[N, K]."""
    w = _f32(w)
    N, K = w.shape
    out = np.empty(N * K // 4 + 4, dtype=np.uint8)
    lib = _load()
    if w_scale is None:
        s = ctypes.c_float(0.0)
        rc = lib.oracle_pack_i2s(w, N, K, out, ctypes.byref(s))
        w_scale = s.value
    else:
        rc = lib.oracle_pack_i2s_with_scale(w, N, K, ctypes.c_float(w_scale), out)
    if rc:
        raise ValueError(f"pack_i2s: bad shape {w.shape}")
    return out, float(np.float32(w_scale))


def unpack_i2s(packed, N: int, K: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    q = np.empty((N, K), dtype=np.int8)
    rc = _load().oracle_unpack_i2s(packed, N, K, q)
    if rc:
        raise ValueError("unpack_i2s: bad shape")
    return q


def count_invalid_codes(packed, N: int, K: int) -> int:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    return int(_load().oracle_count_invalid_codes(packed, N, K))


def rmsnorm(x, g, eps: float = 1e-6, return_rstd: bool = False):
    x = _f32(x)
    g = _f32(g)
    M, K = x.shape
    xn = np.empty_like(x)
    rstd = np.empty(M, dtype=np.float32)
    _load().oracle_rmsnorm(x, g, M, K, ctypes.c_float(eps), xn, _ptr(rstd))
    return (xn, rstd) if return_rstd else xn


def quant_a8(xn):
    """Return (codes int8 [M,K], a_scale f32 [M], rowsum int32 [M])."""
    xn = _f32(xn)
    M, K = xn.shape
    q = np.empty((M, K), dtype=np.int8)
    s = np.empty(M, dtype=np.float32)
    rs = np.empty(M, dtype=np.int32)
    _load().oracle_quant_a8(xn, M, K, q, s, rs)
    return q, s, rs


def i2s_matmul(q, packed, N: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.int8)
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    M, K = q.shape
    acc = np.empty((M, N), dtype=np.int64)
    rc = _load().oracle_i2s_matmul(q, packed, M, K, N, acc)
    if rc:
        raise ValueError("i2s_matmul: bad shape")
    return acc


def rescale(acc, a_scale, w_scale: float) -> np.ndarray:
    acc = np.ascontiguousarray(acc, dtype=np.int64)
    a_scale = _f32(a_scale)
    M, N = acc.shape
    y = np.empty((M, N), dtype=np.float32)
    _load().oracle_rescale(acc, a_scale, ctypes.c_float(w_scale), M, N, y)
    return y


def bitlinear_forward(x, g, packed, w_scale: float, N: int, eps: float = 1e-6, rows=None,
                      intermediates: bool = False):
    """y[rows, N] of the whole projection; all rows when rows is None.

    With intermediates=True returns (y, xn, codes, a_scale, acc)."""
    x = _f32(x)
    g = _f32(g)
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    M, K = x.shape
    if rows is None:
        r = None
        n = M
    else:
        r = np.ascontiguousarray(rows, dtype=np.int64)
        n = r.size
    y = np.empty((n, N), dtype=np.float32)
    xn = np.empty((n, K), dtype=np.float32) if intermediates else None
    q = np.empty((n, K), dtype=np.int8) if intermediates else None
    s = np.empty(n, dtype=np.float32) if intermediates else None
    acc = np.empty((n, N), dtype=np.int64) if intermediates else None
    rc = _load().oracle_bitlinear_forward_rows(
        x, g, packed, ctypes.c_float(w_scale), M, K, N, ctypes.c_float(eps), _ptr(r), n, y,
        _ptr(xn), _ptr(q), _ptr(s), _ptr(acc))
    if rc:
        raise ValueError(f"bitlinear_forward: error {rc}")
    return (y, xn, q, s, acc) if intermediates else y


def dequant_dot_f64(q, t, a_scale, w_scale: float) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.int8)
    t = np.ascontiguousarray(t, dtype=np.int8)
    a_scale = _f32(a_scale)
    M, K = q.shape
    N = t.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    _load().oracle_dequant_dot_f64(q, t, a_scale, ctypes.c_float(w_scale), M, K, N, y)
    return y


ACT_SILU = 1
ACT_GELU_TANH = 2


def activation(x: float, act: int) -> float:
    """The gate activation in double (act 1: SiLU, 2: gelu_pytorch_tanh)."""
    return float(_load().oracle_activation(float(x), int(act)))


def glu(gate, up, act: int) -> np.ndarray:
    """h = act(gate) * up: the activation rounded once to float, times up in float."""
    gate = _f32(gate)
    up = _f32(up)
    if gate.shape != up.shape:
        raise ValueError("glu: gate and up differ in shape")
    h = np.empty(gate.shape, dtype=np.float32)
    _load().oracle_glu(gate.reshape(-1), up.reshape(-1), gate.size, int(act), h.reshape(-1))
    return h


def bitlinear_forward_glu(gate, up, act: int, g, packed, w_scale: float, N: int, eps: float = 1e-6,
                          rows=None):
    """The down projection: y = BitLinear(act(gate) * up)."""
    return bitlinear_forward(glu(gate, up, act), g, packed, w_scale, N, eps, rows=rows)


# ----------------------------------------------------------- 16-bit tensors
# The 16-bit activations and outputs of "gguf-gemv" ("Requirements": f32 or
# bf16 activations, the output in the input's type) and the float16 norm
# weights of "BitNet Embeddings GGUF Conversion Implementation" (section 6.1).
# Every fp16 / bf16 value is an fp32 value, so widening is exact; narrowing is
# IEEE 754 rounding to nearest, ties to even, of an fp32 value to a format with
# 11 (fp16) or 8 (bf16) significand bits.

DTYPE_F32, DTYPE_F16, DTYPE_BF16 = 0, 1, 2


def round_bf16(a) -> np.ndarray:
    """fp32 values rounded to bfloat16 (the upper half of an fp32 pattern), to
    nearest with ties to even; returned widened to float32.  Finite inputs only
    (values at or past the largest bfloat16 plus half a unit become infinity)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    # add half a unit of the kept part, plus one when the kept part is odd
    # (a tie then carries into an even pattern), and drop the low 16 bits
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).reshape(np.shape(a))


def round_f16(a) -> np.ndarray:
    """fp32 values rounded to IEEE binary16 (nearest, ties to even; past 65504
    by half a unit or more: infinity), returned widened to float32."""
    with np.errstate(over="ignore"):
        return np.asarray(a, dtype=np.float32).astype(np.float16).astype(np.float32)


def round_to(a, dtype: int) -> np.ndarray:
    if dtype == DTYPE_F32:
        return _f32(a)
    if dtype == DTYPE_F16:
        return round_f16(a)
    if dtype == DTYPE_BF16:
        return round_bf16(a)
    raise ValueError(f"unknown dtype {dtype}")


def bitlinear_forward_typed(x, g, packed, w_scale: float, N: int, eps: float = 1e-6, y_dtype: int = DTYPE_F32,
                            rows=None) -> np.ndarray:
    """The projection with 16-bit tensors: x and g hold the widened 16-bit
    values (exact fp32 values), y is the fp32 projection rounded once to y_dtype
    (returned widened to float32)."""
    return round_to(bitlinear_forward(x, g, packed, w_scale, N, eps, rows=rows), y_dtype)



# ------------------------------------------------------------ QK head norms
# "BitNet Embeddings GGUF Conversion Implementation", section 4.5 ("Attention
# per-projection norms"): after the q / k matmul, RMSNorm with the attention
# eps times attn_q_norm / attn_k_norm, the per-head "QK head norms" of the model
# table: each head's head_dim consecutive outputs are one RMSNorm row.

def head_rmsnorm(y, head_dim: int, w, eps: float = 1e-6) -> np.ndarray:
    """RMSNorm of every (token, head) row of y[M, N] with weight w[head_dim]."""
    y = _f32(y)
    M, N = y.shape
    if N % head_dim:
        raise ValueError("head_rmsnorm: head_dim must divide N")
    return rmsnorm(y.reshape(M * (N // head_dim), head_dim), w, eps).reshape(M, N)


def bitlinear_forward_qk(x, g, packed, w_scale: float, N: int, head_dim: int, head_w, eps: float = 1e-6,
                         rows=None) -> np.ndarray:
    """The q / k projection followed by its head norm (eps shared by both norms)."""
    return head_rmsnorm(bitlinear_forward(x, g, packed, w_scale, N, eps, rows=rows), head_dim, head_w, eps)
