"""Device-side failure reporting, exercised without a GPU fault.

Every wait inside the library's kernels is bounded: when it runs out, the
kernel records the failure in a per-device error word and returns normally, so
the context stays usable.  The diagnostic entry point waits on a barrier that
nothing completes; the test checks that the status call reports the timeout
once, clears it, and that the same context still computes a correct projection.
"""
import time

import numpy as np
import pytest

import bitlinear_rmsnorm_token_gb300 as bn
from bitlinear_rmsnorm_token_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bn.lib(build=True)


def test_expired_wait_is_reported_and_context_survives(oracle_mod):
    torch.cuda.synchronize()
    assert bn.last_device_status() == bn.OK
    t0 = time.perf_counter()
    bn.selftest_bounded_wait()
    st = bn.last_device_status()  # synchronises the stream
    dt = time.perf_counter() - t0
    assert st == bn.ERR_TIMEOUT, bn.status_string(st)
    assert 0.5 < dt < 30.0, f"the wait should give up after about a second, took {dt:.2f} s"
    assert bn.last_device_status() == bn.OK  # the record was cleared

    M, K, N = 4, 1024, 512
    x = wl.gen_x(M, K, seed=11)
    g = wl.gen_norm_w(K, seed=12)
    w = wl.gen_latent_w(N, K, seed=13)
    packed, ws = bn.pack_i2s(torch.from_numpy(w).cuda())
    y = bn.bitlinear_forward(torch.from_numpy(x).cuda(), torch.from_numpy(g).cuda(), packed, ws, N, wl.EPS)
    torch.cuda.synchronize()
    ref = oracle_mod.bitlinear_forward(x, g, packed.cpu().numpy(), ws, N, wl.EPS)
    assert np.array_equal(y.cpu().numpy(), ref)
    assert bn.last_device_status() == bn.OK
