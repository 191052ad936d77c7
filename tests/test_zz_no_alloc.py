"""bitnet_bitlinear_forward_noalloc against bitnet_bitlinear_forward, through the C ABI.

The no-alloc entry point serves callers that may not allocate device memory once
running (a server that reserved all of HBM for its own allocator, a
latency-critical loop).  It keeps its temporary data in one fixed 16 MiB device
array shared by all calls, so calls in a row with different shapes and data must
each give the same y as the allocating entry point (bit for bit: both run the
same kernels on the same integers) and agree with the oracle.  This file is collected
last on purpose; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import bitlinear_rmsnorm_token_gb300 as bn
from bitlinear_rmsnorm_token_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
REL_L2_TOL = 2e-3  # the end-to-end tolerance the parity tests use


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return bn.lib(build=True)


def _case(M, K, N, seed):
    x = torch.from_numpy(wl.gen_x(M, K, seed=seed, outlier_frac=0.01)).cuda()
    g = torch.from_numpy(wl.gen_norm_w(K, seed=seed + 1)).cuda()
    packed, ws = bn.pack_i2s(torch.from_numpy(wl.gen_latent_w(N, K, seed=seed + 2)).cuda())
    return x, g, packed, ws


def _call(fn, x, g, packed, ws, N, y):
    M, K = x.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(p(x), p(g), p(packed), ctypes.c_float(ws), M, K, N, ctypes.c_float(wl.EPS), p(y), stream)


def _assert_rows_match_oracle(oracle_mod, x, g, packed, ws, N, y, rows):
    """Sampled rows against the oracle under the end-to-end row contract."""
    ref = oracle_mod.bitlinear_forward(x[rows].cpu().numpy(), g.cpu().numpy(), packed.cpu().numpy(), ws, N)
    got = y[rows].double().cpu().numpy()
    nrm = np.linalg.norm(ref, axis=1)
    zero = nrm == 0
    assert np.all(got[zero] == 0.0)
    rel = np.linalg.norm(got - ref, axis=1)[~zero] / nrm[~zero]
    assert rel.size == 0 or rel.max() <= REL_L2_TOL


# One shape per route through the fixed array (M, K, N):
ROUTES = {
    "fused decode, no scratch": (4, 1024, 256),
    "norm launch + decode on int8 codes in the array": (2, 18432, 512),
    "norm launch + decode, K = 32768": (2, 32768, 256),
    "9..63 tokens, K split, partial sums in the array": (16, 16384, 1024),
    "9..63 tokens, K = N = 4096": (16, 4096, 4096),
    "tokens-as-M, K split, partial sums in the array": (128, 16384, 1024),
    "tokens-as-M, no split": (1000, 2048, 384),
    "tokens-as-M, ragged": (257, 1024, 130),
    # codes and scales fit (15.6 MiB) but the K split's partial sums would not:
    # the contraction runs unsplit, with the same y
    "tokens-as-M, K split dropped for lack of room": (1000, 8192, 128),
}


@pytest.mark.parametrize("order", ["forward", "reversed"])
def test_noalloc_equals_forward_on_every_route(L, oracle_mod, order):
    """Each route, called one after another so that every call finds the
    previous call's bytes in the shared array: y equal bit for bit to the
    allocating entry point's, and sampled rows within the oracle contract."""
    names = list(ROUTES) if order == "forward" else list(reversed(ROUTES))
    for i, name in enumerate(names):
        M, K, N = ROUTES[name]
        x, g, packed, ws = _case(M, K, N, 100 + i + (50 if order == "reversed" else 0))
        y_ref = torch.empty((M, N), dtype=torch.float32, device="cuda")
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        assert _call(L.bitnet_bitlinear_forward, x, g, packed, ws, N, y_ref) == bn.OK, name
        assert _call(L.bitnet_bitlinear_forward_noalloc, x, g, packed, ws, N, y) == bn.OK, name
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref), name
        rows = np.arange(M) if M <= 16 else np.random.default_rng(M).choice(M, 12, replace=False)
        _assert_rows_match_oracle(oracle_mod, x, g, packed, ws, N, y, rows)
    assert L.bitnet_last_device_status(None) == bn.OK


def test_noalloc_matches_forward_two_calls_in_a_row(L, oracle_mod):
    # both shapes take the tensor-core path, which uses the fixed scratch array;
    # the second, smaller call leaves stale bytes of the first beyond its end
    for (M, K, N, seed) in ((1000, 2048, 384, 11), (257, 1024, 130, 12)):
        x, g, packed, ws = _case(M, K, N, seed)
        y_ref = torch.empty((M, N), dtype=torch.float32, device="cuda")
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        assert _call(L.bitnet_bitlinear_forward, x, g, packed, ws, N, y_ref) == bn.OK
        assert _call(L.bitnet_bitlinear_forward_noalloc, x, g, packed, ws, N, y) == bn.OK
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref)
        _assert_rows_match_oracle(oracle_mod, x, g, packed, ws, N, y, np.arange(0, M, 37))
    assert L.bitnet_last_device_status(None) == bn.OK


def test_noalloc_small_m_and_size_limit(L):
    x, g, packed, ws = _case(4, 1024, 256, 13)  # decode path: no scratch needed
    y_ref = torch.empty((4, 256), dtype=torch.float32, device="cuda")
    y = torch.empty_like(y_ref)
    assert _call(L.bitnet_bitlinear_forward, x, g, packed, ws, 256, y_ref) == bn.OK
    assert _call(L.bitnet_bitlinear_forward_noalloc, x, g, packed, ws, 256, y) == bn.OK
    torch.cuda.synchronize()
    assert torch.equal(y, y_ref)
    # 4096 tokens x 2048 features need 16 MiB + 16 KiB: refused before any launch
    big = ctypes.c_void_p(1 << 20)
    rc = L.bitnet_bitlinear_forward_noalloc(big, big, big, ctypes.c_float(1.0), 4096, 2048, 64,
                                            ctypes.c_float(wl.EPS), big, None)
    assert rc == bn.ERR_SCRATCH_LIMIT
    assert b"16 MiB" in L.bitnet_status_string(rc)
