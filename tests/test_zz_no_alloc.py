"""bitnet_bitlinear_forward_noalloc against bitnet_bitlinear_forward, through the C ABI.

The no-alloc entry point serves callers that may not allocate device memory once
running (a server that reserved all of HBM for its own allocator, a
latency-critical loop).  It keeps its temporary data in one fixed 16 MiB device
array shared by all calls, so two calls in a row with different shapes and data
must each give the same y as the allocating entry point.  This file is collected
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


def _assert_close(y, ref):
    y = y.double().cpu().numpy()
    ref = ref.double().cpu().numpy()
    nrm = np.linalg.norm(ref, axis=1)
    zero = nrm == 0
    assert np.all(y[zero] == 0.0)
    rel = np.linalg.norm(y - ref, axis=1)[~zero] / nrm[~zero]
    assert rel.size == 0 or rel.max() <= REL_L2_TOL


def test_noalloc_matches_forward_two_calls_in_a_row(L):
    # both shapes take the tensor-core path, which uses the fixed scratch array;
    # the second, smaller call leaves stale bytes of the first beyond its end
    for (M, K, N, seed) in ((1000, 2048, 384, 11), (257, 1024, 130, 12)):
        x, g, packed, ws = _case(M, K, N, seed)
        y_ref = torch.empty((M, N), dtype=torch.float32, device="cuda")
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        assert _call(L.bitnet_bitlinear_forward, x, g, packed, ws, N, y_ref) == bn.OK
        assert _call(L.bitnet_bitlinear_forward_noalloc, x, g, packed, ws, N, y) == bn.OK
        torch.cuda.synchronize()
        _assert_close(y, y_ref)
    assert L.bitnet_last_device_status(None) == bn.OK


def test_noalloc_small_m_and_size_limit(L):
    x, g, packed, ws = _case(4, 1024, 256, 13)  # decode path: no scratch needed
    y_ref = torch.empty((4, 256), dtype=torch.float32, device="cuda")
    y = torch.empty_like(y_ref)
    assert _call(L.bitnet_bitlinear_forward, x, g, packed, ws, 256, y_ref) == bn.OK
    assert _call(L.bitnet_bitlinear_forward_noalloc, x, g, packed, ws, 256, y) == bn.OK
    torch.cuda.synchronize()
    _assert_close(y, y_ref)
    # 4096 tokens x 2048 features need 16 MiB + 16 KiB: refused before any launch
    big = ctypes.c_void_p(1 << 20)
    rc = L.bitnet_bitlinear_forward_noalloc(big, big, big, ctypes.c_float(1.0), 4096, 2048, 64,
                                            ctypes.c_float(wl.EPS), big, None)
    assert rc == bn.ERR_SCRATCH_LIMIT
    assert b"16 MiB" in L.bitnet_status_string(rc)
