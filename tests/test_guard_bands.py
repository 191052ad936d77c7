"""Out-of-bounds writes, checked without a sanitizer: every output a caller
hands to the library is placed inside a larger buffer whose bytes before and
after it hold a seeded random pattern.  After the call the bands must be
unchanged (no store outside the output, whatever the tile clipping, split-K
read-back or ragged tail does), every byte of the output itself must have
been written (it starts as random bytes and must equal, bit for bit, the
result of the same call on an exactly sized allocation), and the inputs must
be untouched.

Routes covered (each named in its case id): the fused decode launch (short and
long rows, ragged N), the norm launch + decode launch for rows too long to
fuse, the 9..63-token split-K kernel, the tokens-as-M kernel with its TMA-store
epilogue (clipped rows and columns), its direct-store epilogue (row pitch not a
multiple of 16 bytes) and its split-K read-back, 16-bit y, the fused and the
separate QK head norm, the down projection's routes, the grouped decode launch,
packing, unpacking and the no-alloc entry point.
"""
import numpy as np
import pytest

import bitlinear_rmsnorm_token_gb300 as bn
from bitlinear_rmsnorm_token_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

GUARD = 4096  # bytes of random pattern on each side of an output


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bn.lib(build=True)
    yield
    assert bn.last_device_status() == bn.OK


class Guarded:
    """An output tensor of `shape` and `dtype` with GUARD bytes of random
    pattern before and after it (the output's bytes start random too)."""

    def __init__(self, shape, dtype, seed):
        self.shape = tuple(shape)
        self.dtype = dtype
        esz = torch.empty(0, dtype=dtype).element_size()
        self.nbytes = int(np.prod(self.shape)) * esz
        total = 2 * GUARD + self.nbytes
        total += (-total) % 16
        gen = torch.Generator(device="cpu").manual_seed(seed)
        pattern = torch.randint(0, 256, (total,), dtype=torch.uint8, generator=gen)
        self.raw = pattern.cuda()
        self.snapshot = pattern.clone()
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(self.shape)

    def check(self, what):
        torch.cuda.synchronize()
        now = self.raw.cpu()
        before = now[:GUARD]
        after = now[GUARD + self.nbytes:]
        bad_lo = int((before != self.snapshot[:GUARD]).sum())
        bad_hi = int((after != self.snapshot[GUARD + self.nbytes:]).sum())
        assert bad_lo == 0 and bad_hi == 0, f"{what}: {bad_lo} bytes written before and {bad_hi} after the output"

    def bits(self):
        torch.cuda.synchronize()
        return self.t.contiguous().view(torch.uint8).cpu().numpy()


def same_bits(guarded, exact, what):
    want = exact.contiguous().view(torch.uint8).cpu().numpy()
    got = guarded.bits()
    assert got.shape == want.shape
    nbad = int(np.sum(got != want))
    assert nbad == 0, f"{what}: {nbad} output bytes differ from the exactly sized call (unwritten or wrong)"


class Inputs:
    """Snapshots of input tensors, to check that a call leaves them untouched."""

    def __init__(self, *ts):
        self.ts = ts
        self.copies = [t.clone() for t in ts]

    def check(self, what):
        for i, (t, c) in enumerate(zip(self.ts, self.copies)):
            assert torch.equal(t.reshape(-1).view(torch.uint8), c.reshape(-1).view(torch.uint8)), \
                f"{what}: input {i} was modified"


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def projection(M, K, N, seed):
    x = dev(wl.gen_x(M, K, seed=seed, outlier_frac=0.01))
    g = dev(wl.gen_norm_w(K, seed=seed + 1))
    packed, ws = bn.pack_i2s(dev(wl.gen_latent_w(N, K, seed=seed + 2)))
    return x, g, packed, ws


# --------------------------------------------------------------- forward

FORWARD_ROUTES = [
    ("decode_fused_short_row_N_tail", 1, 1024, 1000),
    ("decode_fused_staged_3_tokens", 3, 2048, 777),
    ("decode_fused_8_tokens", 8, 3072, 100),
    ("decode_fused_long_row", 1, 16384, 333),
    ("decode_fused_long_rows_4_tokens", 4, 8192, 777),
    ("norm_launch_then_decode", 2, 32768, 40),
    ("norm_launch_then_decode_65536", 1, 65536, 300),
    ("split_k_9_to_63_tokens", 12, 4096, 3000),
    ("split_k_9_to_63_tokens_wide", 20, 1024, 16500),
    ("split_k_9_to_63_tokens_ragged", 33, 8192, 130),
    ("tokens_as_m_tma_store_ragged_rows", 300, 1024, 640),
    ("tokens_as_m_tma_store_clipped_cols", 100, 640, 1000),
    ("tokens_as_m_direct_store_odd_pitch", 129, 1024, 385),
    ("tokens_as_m_split_k_readback", 96, 8192, 777),
    ("tokens_as_m_split_k_readback_wide", 200, 8192, 300),
]


@pytest.mark.parametrize("name,M,K,N", FORWARD_ROUTES, ids=[r[0] for r in FORWARD_ROUTES])
def test_forward_guard_bands(name, M, K, N):
    x, g, packed, ws = projection(M, K, N, seed=M + K + N)
    inputs = Inputs(x, g, packed)
    exact = bn.bitlinear_forward(x, g, packed, ws, N, wl.EPS)
    out = Guarded((M, N), torch.float32, seed=M * N)
    bn.bitlinear_forward(x, g, packed, ws, N, wl.EPS, y=out.t)
    out.check(name)
    same_bits(out, exact, name)
    inputs.check(name)


@pytest.mark.parametrize("name,M,K,N", [r for r in FORWARD_ROUTES if r[1] * r[2] * 2 + 4 * r[1] <= 16 << 20],
                         ids=[r[0] for r in FORWARD_ROUTES if r[1] * r[2] * 2 + 4 * r[1] <= 16 << 20])
def test_noalloc_guard_bands(name, M, K, N):
    x, g, packed, ws = projection(M, K, N, seed=3 * M + K + N)
    exact = bn.bitlinear_forward(x, g, packed, ws, N, wl.EPS)
    out = Guarded((M, N), torch.float32, seed=M * N + 1)
    bn.bitlinear_forward_noalloc(x, g, packed, ws, N, wl.EPS, y=out.t)
    out.check(name)
    same_bits(out, exact, name)


TYPED_ROUTES = [
    ("decode_on_fp32_copies", 4, 16384, 600),
    ("split_k_fp32_copy", 16, 16384, 1024),
    ("tokens_as_m_16bit_tma_store", 300, 1024, 640),
    ("tokens_as_m_16bit_direct_store", 200, 3072, 130),
    ("tokens_as_m_16bit_split_k_readback", 128, 16384, 1024),
    ("tokens_as_m_16bit_ragged_cols", 70, 1280, 264),
]


@pytest.mark.parametrize("name,M,K,N", TYPED_ROUTES, ids=[r[0] for r in TYPED_ROUTES])
@pytest.mark.parametrize("ydt", [torch.bfloat16, torch.float16])
def test_typed_guard_bands(name, M, K, N, ydt):
    x, g, packed, ws = projection(M, K, N, seed=M + 2 * K + N)
    xb = x.to(torch.bfloat16)
    gh = g.to(torch.float16)
    inputs = Inputs(xb, gh, packed)
    exact = bn.bitlinear_forward_typed(xb, gh, packed, ws, N, wl.EPS, y_dtype=ydt)
    out = Guarded((M, N), ydt, seed=M * N + 2)
    bn.bitlinear_forward_typed(xb, gh, packed, ws, N, wl.EPS, y=out.t)
    out.check(name)
    same_bits(out, exact, name)
    inputs.check(name)


QK_ROUTES = [
    ("qk_decode", 1, 1024, 2048, 128),
    ("qk_fused_epilogue_128", 300, 1024, 2048, 128),
    ("qk_fused_epilogue_256", 129, 640, 1024, 256),
    ("qk_split_k", 128, 16384, 1024, 128),
]


@pytest.mark.parametrize("name,M,K,N,hd", QK_ROUTES, ids=[r[0] for r in QK_ROUTES])
def test_qk_guard_bands(name, M, K, N, hd):
    x, g, packed, ws = projection(M, K, N, seed=M + K + 5 * N)
    hw = dev(wl.gen_norm_w(hd, seed=hd))
    inputs = Inputs(x, g, packed, hw)
    exact = bn.bitlinear_forward_qk(x, g, packed, ws, N, hd, hw, wl.EPS)
    out = Guarded((M, N), torch.float32, seed=M * N + 3)
    bn.bitlinear_forward_qk(x, g, packed, ws, N, hd, hw, wl.EPS, y=out.t)
    out.check(name)
    same_bits(out, exact, name)
    inputs.check(name)
    # the separate head-norm launch, out of place, on a ragged token count
    y = exact[: M - 1 if M > 1 else 1].contiguous()
    ref = bn.head_rmsnorm(y, hd, hw, wl.EPS)
    hn = Guarded(tuple(y.shape), torch.float32, seed=M + 4)
    bn.head_rmsnorm(y, hd, hw, wl.EPS, out=hn.t)
    hn.check(name + " head_rmsnorm")
    same_bits(hn, ref, name + " head_rmsnorm")


GLU_ROUTES = [
    ("glu_fused_decode", 1, 3072, 1024),
    ("glu_norm_launch_decode", 3, 2048, 640),
    ("glu_through_memory_decode", 2, 8192 + 1024, 300),
    ("glu_tokens_as_m", 300, 2048, 640),
    ("glu_split_k", 128, 16384, 1024),
]


@pytest.mark.parametrize("name,M,K,N", GLU_ROUTES, ids=[r[0] for r in GLU_ROUTES])
def test_glu_guard_bands(name, M, K, N):
    rng = np.random.default_rng(M + K + N)
    gate = dev(rng.normal(0, 2, (M, K)).astype(np.float32))
    up = dev(rng.normal(0, 1, (M, K)).astype(np.float32))
    g = dev(wl.gen_norm_w(K, seed=K))
    packed, ws = bn.pack_i2s(dev(wl.gen_latent_w(N, K, seed=N)))
    inputs = Inputs(gate, up, g, packed)
    exact = bn.bitlinear_forward_glu(gate, up, bn.ACT_SILU, g, packed, ws, N, wl.EPS)
    out = Guarded((M, N), torch.float32, seed=M * N + 5)
    bn.bitlinear_forward_glu(gate, up, bn.ACT_SILU, g, packed, ws, N, wl.EPS, y=out.t)
    out.check(name)
    same_bits(out, exact, name)
    # h itself
    h_exact = bn.glu(gate, up, bn.ACT_GELU_TANH)
    h = Guarded((M, K), torch.float32, seed=M + K)
    bn.glu(gate, up, bn.ACT_GELU_TANH, h=h.t)
    h.check(name + " glu")
    same_bits(h, h_exact, name + " glu")
    inputs.check(name)


# ------------------------------------------------- norm + quant, contraction

@pytest.mark.parametrize("M,K", [(5, 640), (33, 1024), (3, 3072), (7, 4096), (3, 16384), (2, 65536)])
def test_rmsnorm_quant_guard_bands(M, K):
    x, g, _, _ = projection(M, K, 1, seed=M * 17 + K)
    inputs = Inputs(x, g)
    c0, s0, r0 = bn.rmsnorm_quant_a8(x, g, wl.EPS, rowsum=torch.empty(M, dtype=torch.int32, device="cuda"))
    xn0 = torch.empty((M, K), dtype=torch.float32, device="cuda")
    bn.rmsnorm_quant_a8(x, g, wl.EPS, xn_out=xn0)
    codes = Guarded((M, K), torch.int8, seed=1)
    scale = Guarded((M,), torch.float32, seed=2)
    rowsum = Guarded((M,), torch.int32, seed=3)
    xn = Guarded((M, K), torch.float32, seed=4)
    bn.rmsnorm_quant_a8(x, g, wl.EPS, codes=codes.t, a_scale=scale.t, rowsum=rowsum.t, xn_out=xn.t)
    for b, ref, what in ((codes, c0, "codes"), (scale, s0, "a_scale"), (rowsum, r0, "rowsum"), (xn, xn0, "xn")):
        b.check(f"rmsnorm_quant M={M} K={K} {what}")
        same_bits(b, ref, f"rmsnorm_quant M={M} K={K} {what}")
    inputs.check(f"rmsnorm_quant M={M} K={K}")


GEMM_ROUTES = [
    ("decode_acc", 5, 1024, 129),
    ("decode_long_acc", 4, 16384, 2500),
    ("split_k_acc", 33, 8192, 130),
    ("tokens_as_m_acc", 100, 640, 1000),
    ("tokens_as_m_split_k_acc", 200, 8192, 300),
]


@pytest.mark.parametrize("name,M,K,N", GEMM_ROUTES, ids=[r[0] for r in GEMM_ROUTES])
def test_gemm_guard_bands(name, M, K, N):
    rng = np.random.default_rng(M + K + N)
    codes = dev(rng.integers(-128, 128, size=(M, K), dtype=np.int8))
    a_scale = dev(rng.uniform(0.5, 300.0, size=M).astype(np.float32))
    packed, ws = bn.pack_i2s(dev(wl.gen_latent_w(N, K, seed=K + N)))
    inputs = Inputs(codes, a_scale, packed)
    acc0 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    y0 = bn.i2s_gemm(codes, a_scale, packed, ws, N, acc_out=acc0)
    y = Guarded((M, N), torch.float32, seed=7)
    acc = Guarded((M, N), torch.int32, seed=8)
    bn.i2s_gemm(codes, a_scale, packed, ws, N, y=y.t, acc_out=acc.t)
    for b, ref, what in ((y, y0, "y"), (acc, acc0, "acc")):
        b.check(f"{name} {what}")
        same_bits(b, ref, f"{name} {what}")
    # y alone (the vectorised epilogues)
    y1 = Guarded((M, N), torch.float32, seed=9)
    bn.i2s_gemm(codes, a_scale, packed, ws, N, y=y1.t)
    y1.check(f"{name} y without acc")
    same_bits(y1, y0, f"{name} y without acc")
    inputs.check(name)


# ------------------------------------------------------- grouped decode launch

def test_group_guard_bands():
    shapes = [(1024, 2048), (1024, 1000), (3072, 1024), (2048, 333)]
    M = 2
    projs, exact, outs, ins = [], [], [], []
    for i, (K, N) in enumerate(shapes):
        x, g, packed, ws = projection(M, K, N, seed=100 + i)
        exact.append(bn.bitlinear_forward(x, g, packed, ws, N, wl.EPS))
        out = Guarded((M, N), torch.float32, seed=200 + i)
        outs.append(out)
        projs.append((x, g, packed, ws, N, out.t))
        ins.append(Inputs(x, g, packed))
    bn.bitlinear_forward_group(projs, M, wl.EPS)
    for i, (out, ref, inp) in enumerate(zip(outs, exact, ins)):
        out.check(f"group projection {i}")
        same_bits(out, ref, f"group projection {i}")
        inp.check(f"group projection {i}")


# ------------------------------------------------------------ pack / unpack

@pytest.mark.parametrize("N,K", [(3, 256), (130, 3072), (7, 16384)])
def test_pack_unpack_guard_bands(N, K):
    w = dev(wl.gen_latent_w(N, K, seed=N + K))
    inputs = Inputs(w)
    p0, s0 = bn.pack_i2s(w)
    packed = Guarded((bn.packed_bytes(N, K),), torch.uint8, seed=N)
    _, s = bn.pack_i2s(w, packed=packed.t)
    assert s == s0
    packed.check(f"pack N={N} K={K}")
    same_bits(packed, p0, f"pack N={N} K={K}")
    u0 = bn.unpack_i2s(p0, N, K)
    u = Guarded((N, K), torch.int8, seed=K)
    bn.unpack_i2s(p0, N, K, out=u.t)
    u.check(f"unpack N={N} K={K}")
    same_bits(u, u0, f"unpack N={N} K={K}")
    inputs.check(f"pack N={N} K={K}")
