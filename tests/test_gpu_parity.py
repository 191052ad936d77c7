"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Bit-exact: I2_S bytes and scale, unpacked weights, int8 codes / scales / row
sums given the same normalised input, int32 accumulators, and y given the same
codes.  End to end (x -> y) the only freedom is the rounding of the RMSNorm
sum of squares (double in the oracle, a compensated warp reduction on the GPU),
so each row must be within 2e-3 of the oracle row's L2 norm, zero rows exactly
zero, at most 1e-4 of the codes may differ by one, and in practice every row
matches bit for bit (asserted: at most 1 in 1000 rows may differ at all).
"""
import numpy as np
import pytest

import bitlinear_rmsnorm_token_gb300 as bn
from bitlinear_rmsnorm_token_gb300 import workloads as wl

from contract import assert_code_flips_at_ties

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
REL_L2_TOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bn.lib(build=True)
    yield
    assert bn.last_device_status() == bn.OK


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def assert_rows_within_tolerance(y, ref, what=""):
    """The end-to-end row tolerance alone (inputs that differ in the last bits)."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    nrm = np.linalg.norm(ref, axis=1)
    rel = np.linalg.norm(y - ref, axis=1)[nrm > 0] / nrm[nrm > 0]
    assert rel.size == 0 or rel.max() <= REL_L2_TOL, f"{what}: worst row rel-L2 {rel.max():.3e}"


def assert_rows_close(y, ref, what=""):
    """The end-to-end contract, row by row."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    diff = np.linalg.norm(y - ref, axis=1)
    nrm = np.linalg.norm(ref, axis=1)
    zero = nrm == 0
    assert np.all(y[zero] == 0.0), f"{what}: zero rows must stay exactly zero"
    rel = diff[~zero] / nrm[~zero]
    assert rel.size == 0 or rel.max() <= REL_L2_TOL, f"{what}: worst row rel-L2 {rel.max():.3e}"
    inexact = int(np.sum(np.any(y != ref, axis=1)))
    assert inexact <= max(1, y.shape[0] // 1000), f"{what}: {inexact} of {y.shape[0]} rows not bit-identical"


# ------------------------------------------------------------------ packing

@pytest.mark.parametrize("N,K", [(1, 128), (3, 256), (1000, 640), (2048, 1024), (7, 16384), (130, 3072)])
def test_pack_matches_oracle(oracle_mod, N, K):
    w = wl.gen_latent_w(N, K, seed=N * 7 + K)
    packed, s = bn.pack_i2s(dev(w))
    s_ora = oracle_mod.weight_scale(w)
    # the GPU's fixed-order double reduction may round differently in the last
    # place; the scale is then one float ulp away and the codes are compared
    # under the GPU's scale
    assert np.float32(s) == np.float32(s_ora) or abs(np.float32(s) - np.float32(s_ora)) <= np.spacing(np.float32(s))
    ref, _ = oracle_mod.pack_i2s(w, w_scale=s)
    got = host(packed)
    assert np.array_equal(got, ref)
    # deterministic: same bytes again
    packed2, s2 = bn.pack_i2s(dev(w))
    assert s2 == s and np.array_equal(host(packed2), got)


def test_pack_special_tensors(oracle_mod):
    K = 256
    for w in (np.zeros((4, K), np.float32), np.full((4, K), -3.5, np.float32),
              np.tile(np.array([1.5, 0.5, -0.5, -1.5], np.float32), (4, K // 4))):
        packed, s = bn.pack_i2s(dev(w))
        ref, s_ref = oracle_mod.pack_i2s(w)
        assert s == s_ref
        assert np.array_equal(host(packed), ref)


@pytest.mark.parametrize("N,K", [(1, 128), (5, 384), (1024, 1024)])
def test_unpack_matches_oracle(oracle_mod, N, K):
    rng = np.random.default_rng(N + K)
    raw = rng.integers(0, 256, size=N * K // 4, dtype=np.uint8)  # includes invalid code 3
    packed = np.concatenate([raw, np.zeros(4, np.uint8)])
    got = host(bn.unpack_i2s(dev(packed), N, K))
    assert np.array_equal(got, oracle_mod.unpack_i2s(packed, N, K))


# ----------------------------------------------------------- norm + quant

def _x_with_edges(M, K, seed):
    x = wl.gen_x(M, K, seed=seed, outlier_frac=0.01)
    if M >= 3:
        x[1] = 0.0            # zero row -> zero codes
        x[2] = 0.25           # constant row
    return x


@pytest.mark.parametrize("M,K", [(1, 128), (5, 640), (33, 1024), (9, 2048), (4, 1152), (17, 3072), (7, 4096), (2, 5120), (3, 16384), (2, 18432), (2, 65536)])
def test_rmsnorm_quant_matches_oracle(oracle_mod, M, K):
    x = _x_with_edges(M, K, seed=M * 31 + K)
    g = wl.gen_norm_w(K, seed=K)
    codes = torch.empty((M, K), dtype=torch.int8, device="cuda")
    a_scale = torch.empty(M, dtype=torch.float32, device="cuda")
    rowsum = torch.empty(M, dtype=torch.int32, device="cuda")
    xn = torch.empty((M, K), dtype=torch.float32, device="cuda")
    bn.rmsnorm_quant_a8(dev(x), dev(g), wl.EPS, codes, a_scale, rowsum, xn)
    xn_gpu = host(xn)
    # given the same normalised rows, quantisation is bit-exact
    q_o, s_o, rs_o = oracle_mod.quant_a8(xn_gpu)
    assert np.array_equal(host(codes), q_o)
    assert np.array_equal(host(a_scale), s_o)
    assert np.array_equal(host(rowsum), rs_o)
    # the normalised rows themselves: identical unless rstd rounded differently
    xn_o = oracle_mod.rmsnorm(x, g, wl.EPS)
    rows_differ = int(np.sum(np.any(xn_gpu != xn_o, axis=1)))
    assert rows_differ <= max(1, M // 1000)
    # end to end codes: at most 1e-4 differ, by one, and only at rounding ties
    q_e, s_e, _ = oracle_mod.quant_a8(xn_o)
    assert_code_flips_at_ties(host(codes), q_e, xn_o, s_e)
    if M >= 3:
        assert np.all(host(codes)[1] == 0) and host(rowsum)[1] == 0


def _x_extreme_rows(K, seed):
    """Rows that stress the fixed-point sum of squares and the row scale: huge,
    tiny and subnormal magnitudes, two magnitudes 40 decades apart, one
    dominant element over many tiny ones, per-element exponents spread over
    60 binades, a single non-zero element, values near the float maximum."""
    rng = np.random.default_rng(seed)
    b = rng.standard_normal((8, K))
    x = np.empty((8, K), np.float64)
    x[0] = b[0] * 1e30
    x[1] = b[1] * 1e-30
    x[2] = b[2] * 1e-40
    x[3] = b[3] * np.where(np.arange(K) % 2 == 1, 1e20, 1e-20)
    x[4] = b[4] * 1e-7
    x[4, 0] = 3.0
    x[5] = b[5] * np.exp2(rng.integers(-30, 30, K).astype(np.float64))
    x[6] = 0.0
    x[6, K // 2] = -2.5
    x[7] = np.where(rng.random(K) < 0.01, 3.0e38, 1.0) * np.sign(b[7])
    return x.astype(np.float32)


@pytest.mark.parametrize("K", [1024, 65536])
def test_rmsnorm_quant_extreme_rows(oracle_mod, K):
    x = _x_extreme_rows(K, seed=K)
    g = wl.gen_norm_w(K, seed=K + 1)
    M = x.shape[0]
    codes = torch.empty((M, K), dtype=torch.int8, device="cuda")
    a_scale = torch.empty(M, dtype=torch.float32, device="cuda")
    rowsum = torch.empty(M, dtype=torch.int32, device="cuda")
    xn = torch.empty((M, K), dtype=torch.float32, device="cuda")
    bn.rmsnorm_quant_a8(dev(x), dev(g), wl.EPS, codes, a_scale, rowsum, xn)
    xn_gpu = host(xn)
    q_o, s_o, rs_o = oracle_mod.quant_a8(xn_gpu)
    assert np.array_equal(host(codes), q_o)
    assert np.array_equal(host(a_scale), s_o)
    assert np.array_equal(host(rowsum), rs_o)
    xn_o = oracle_mod.rmsnorm(x, g, wl.EPS)
    assert int(np.sum(np.any(xn_gpu != xn_o, axis=1))) <= 1


@pytest.mark.parametrize("K", [1024, 4096])
def test_forward_extreme_rows(oracle_mod, K):
    """The fused decode path (M = 8) and the prefill path on the same rows."""
    x = _x_extreme_rows(K, seed=K + 7)
    g = wl.gen_norm_w(K, seed=K + 8)
    N = 256
    w = wl.gen_latent_w(N, K, seed=K + 9)
    packed, ws = bn.pack_i2s(dev(w))
    ref = oracle_mod.bitlinear_forward(x, g, host(packed), ws, N, wl.EPS)
    y_dec = host(bn.bitlinear_forward(dev(x), dev(g), packed, ws, N, wl.EPS))
    assert_rows_close(y_dec, ref, f"decode K={K}")
    xx = np.tile(x, (4, 1))  # 32 rows: the tensor-core path
    y_tc = host(bn.bitlinear_forward(dev(xx), dev(g), packed, ws, N, wl.EPS))
    assert_rows_close(y_tc, np.tile(ref, (4, 1)), f"prefill K={K}")


# ------------------------------------------------------------ contraction

GEMM_CASES = [
    # decode (dp4a) path
    (1, 128, 1), (1, 1024, 2048), (2, 640, 33), (3, 3072, 200), (5, 1024, 129), (8, 1024, 2048), (8, 8192, 64),
    (1, 16384, 4096), (4, 16384, 2500),
    # split-K 8-bit tensor-core path (9..63 tokens with K >= 4096 or N >= 16384): 128 weight
    # rows x 16/32/48/64 tokens, K split into ranges of I2_S blocks combined by atomic fp32
    # additions, ragged weight tiles (64 tokens: the boundary, taken by the next kernel)
    (16, 16384, 1024), (64, 4096, 4096), (33, 8192, 130), (9, 65536, 256), (12, 4096, 3000),
    (48, 6144, 1000), (20, 1024, 16500), (64, 256, 16384), (44, 4096, 2100), (57, 16384, 700),
    # tensor-core path, tokens as the MMA's M side: 128 tokens x 64/128/256 weights, ragged tails
    (9, 128, 128), (16, 256, 130), (64, 1024, 256), (100, 640, 1000), (40, 2048, 1000), (64, 128, 5000),
    (24, 3072, 2049), (17, 1920, 300), (129, 1024, 384), (300, 3072, 257), (600, 2048, 1024), (1000, 128, 5),
    # the same kernel with K split over CTAs (few output tiles; 64- and 128-wide tiles): exact fp32
    # atomic partial sums, the last range of a tile rescales it; ragged token and weight tails
    (128, 16384, 1024), (128, 4096, 4096), (200, 8192, 300), (65, 2048, 2100), (70, 65536, 256),
    (128, 16384, 2048),
]


@pytest.mark.parametrize("M,K,N", GEMM_CASES)
def test_gemm_matches_oracle(oracle_mod, M, K, N):
    rng = np.random.default_rng(M * 1000 + K + N)
    codes = rng.integers(-128, 128, size=(M, K), dtype=np.int8)
    a_scale = rng.uniform(0.5, 300.0, size=M).astype(np.float32)
    w = wl.gen_latent_w(N, K, seed=K * 3 + N)
    packed, ws = oracle_mod.pack_i2s(w)
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    y = bn.i2s_gemm(dev(codes), dev(a_scale), dev(packed), ws, N, acc_out=acc)
    acc_o = oracle_mod.i2s_matmul(codes, packed, N)
    assert np.array_equal(host(acc).astype(np.int64), acc_o)
    y_o = oracle_mod.rescale(acc_o, a_scale, ws)
    assert np.array_equal(host(y), y_o)
    # without the accumulator output the tensor-core path writes y by TMA
    # stores (N % 4 == 0) that clip the ragged rows and columns of the tiles
    y2 = bn.i2s_gemm(dev(codes), dev(a_scale), dev(packed), ws, N)
    assert np.array_equal(host(y2), y_o)


# Shapes whose tile counts make the tensor-core kernel pick 256-, 128- and
# 64-wide weight tiles with several tiles per CTA and K spanning several packed
# blocks (the ring of packed slots and operand stages wraps across tiles).
MULTI_TILE_CASES = [(4096, 640, 2048), (2048, 640, 2048), (4096, 1024, 2048), (1024, 1152, 4096), (300, 640, 1000)]


@pytest.mark.parametrize("M,K,N", MULTI_TILE_CASES)
def test_gemm_multi_tile_ctas(oracle_mod, M, K, N):
    rng = np.random.default_rng(M + K + N)
    codes = rng.integers(-128, 128, size=(M, K), dtype=np.int8)
    a_scale = rng.uniform(0.5, 300.0, size=M).astype(np.float32)
    w = wl.gen_latent_w(N, K, seed=N + K)
    packed, ws = oracle_mod.pack_i2s(w)
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    cd, sd, pd = dev(codes), dev(a_scale), dev(packed)
    y_acc = bn.i2s_gemm(cd, sd, pd, ws, N, acc_out=acc)   # per-element stores
    y_vec = bn.i2s_gemm(cd, sd, pd, ws, N)                # TMA-store epilogue
    acc_o = oracle_mod.i2s_matmul(codes, packed, N)
    assert np.array_equal(host(acc).astype(np.int64), acc_o)
    y_o = oracle_mod.rescale(acc_o, a_scale, ws)
    assert np.array_equal(host(y_acc), y_o)
    assert np.array_equal(host(y_vec), y_o)


@pytest.mark.parametrize("path_m", [4, 32])
def test_gemm_special_weights(oracle_mod, path_m):
    M, K, N = path_m, 128, 128
    rng = np.random.default_rng(path_m)
    codes = rng.integers(-127, 128, size=(M, K), dtype=np.int8)
    rowsum = codes.astype(np.int64).sum(axis=1)
    a_scale = np.ones(M, np.float32)
    for t, want in ((np.ones((N, K), np.int8), np.repeat(rowsum[:, None], N, 1)),
                    (-np.ones((N, K), np.int8), -np.repeat(rowsum[:, None], N, 1)),
                    (np.zeros((N, K), np.int8), np.zeros((M, N), np.int64)),
                    (np.eye(N, K, dtype=np.int8), codes.astype(np.int64)[:, :N])):
        packed = oracle_mod.encode_i2s(t, 1.0)
        acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
        bn.i2s_gemm(dev(codes), dev(a_scale), dev(packed), 1.0, N, acc_out=acc)
        assert np.array_equal(host(acc).astype(np.int64), want)


@pytest.mark.parametrize("M", [1, 8, 16, 256])
@pytest.mark.parametrize("K", [16384, 65536])
def test_accumulator_exactness_extremes(oracle_mod, M, K):
    """Largest partial sums the fp32 tensor-core accumulator meets: all codes
    +-127 against all +-1 weights (|acc| = 127 K, up to 8,323,072 < 2^24)."""
    N = 128
    codes = np.full((M, K), 127, np.int8)
    codes[1::2, 1::2] = -127
    t = np.ones((N, K), np.int8)
    t[1::2] = -1
    t[2::4, ::2] = -1
    packed = oracle_mod.encode_i2s(t, 1.0)
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    bn.i2s_gemm(dev(codes), dev(np.ones(M, np.float32)), dev(packed), 1.0, N, acc_out=acc)
    want = oracle_mod.i2s_matmul(codes, packed, N)
    assert np.abs(want).max() == 127 * K
    assert np.array_equal(host(acc).astype(np.int64), want)


# ---------------------------------------------------------------- forward

FWD_CASES = [
    # fused decode launch, activations staged in shared memory (M <= 8, 5*M*K + 4*K <= 144 KiB)
    (1, 128, 1), (1, 1024, 2048), (3, 2048, 1024), (8, 1024, 2048), (8, 3072, 100), (1, 10240 - 128, 96),
    # fused decode launch, long rows (K a multiple of 2048 in [4096, 16384]): activations
    # and norm weight in registers, one warp per 8 KB stage of whole rows
    (1, 4096, 4096), (5, 4096, 333), (1, 16384, 4096), (1, 8192, 3000), (4, 8192, 777),
    (3, 16384, 300), (8, 8192, 64), (2, 16384, 4096),
    # fewer weight rows than CTAs, a single row, K = 12288
    (1, 16384, 96), (2, 4096, 150), (4, 4096, 5000), (1, 12288, 1),
    # one token, K = 4096 / 8192 / 16384: the row kernel (CTA pairs sharing the
    # prologue; one row, one row per CTA of a pair, a pair's second CTA with
    # one row or none, partial 32 KB stages, slots reused across laps)
    (1, 4096, 1), (1, 8192, 2), (1, 16384, 3), (1, 4096, 5), (1, 16384, 151), (1, 8192, 1000),
    (1, 4096, 20000),
    # longer rows: row-per-CTA norm launch, then the decode launch streaming its
    # weight ring during it
    (1, 65536, 300), (2, 32768, 40),
    # ring slots reused many times, slot counts not a multiple of the 15 consumer
    # warps (28 slots of 8 KB at K=4096; 6 slots of one 16 KB row at K=65536)
    (1, 4096, 65536), (1, 65536, 4096), (2, 8192, 20000),
    # norm launch + tensor-core launch
    (16, 640, 256), (64, 1024, 2048), (257, 3072, 1024), (1000, 640, 130), (2048, 2048, 384), (40, 8192, 256),
    (128, 8192, 3000), (12, 16384, 1024),
    # norm launch + tensor-core launch with K split over CTAs
    (128, 16384, 1024), (96, 8192, 777)]


@pytest.mark.parametrize("M,K,N", FWD_CASES)
def test_forward_matches_oracle(oracle_mod, M, K, N):
    x = _x_with_edges(M, K, seed=M + K + N)
    g = wl.gen_norm_w(K, seed=N)
    w = wl.gen_latent_w(N, K, seed=M * N + K)
    packed, ws = bn.pack_i2s(dev(w))
    y = bn.bitlinear_forward(dev(x), dev(g), packed, ws, N, wl.EPS)
    ref = oracle_mod.bitlinear_forward(x, g, host(packed), ws, N, wl.EPS)
    assert_rows_close(host(y), ref, f"forward M={M} K={K} N={N}")


# 16-bit x / y and fp16 norm weights: every path (decode launches on fp32
# copies, the split-K kernel with an fp32 y copy, the tokens-as-M kernel
# reading 16-bit x in its norm launch and writing 16-bit y by TMA stores, by
# direct stores when the row pitch is not a multiple of 16 bytes, and by the
# split-K read-back)
TYPED_CASES = [(1, 1024, 2048), (4, 16384, 600), (16, 16384, 1024), (300, 1024, 640), (200, 3072, 130),
               (128, 16384, 1024), (2048, 640, 2048),
               (70, 1280, 256), (70, 3200, 256)]  # norm launch: generic row widths (24 groups, re-read)
TYPED_DTYPES = [("bf16", "f32", "bf16"), ("f16", "f16", "f16"), ("f32", "f16", "bf16"), ("bf16", "f16", "f32")]
_TT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
_OT = {"f32": 0, "f16": 1, "bf16": 2}


@pytest.mark.parametrize("M,K,N", TYPED_CASES)
@pytest.mark.parametrize("xt,gt,yt", TYPED_DTYPES)
def test_forward_typed_matches_oracle(oracle_mod, M, K, N, xt, gt, yt):
    # inputs rounded to their 16-bit types on the host (torch CPU casts); the
    # oracle gets the same values widened, which is exact
    x = torch.from_numpy(_x_with_edges(M, K, seed=M + 3 * K + N)).to(_TT[xt])
    g = torch.from_numpy(wl.gen_norm_w(K, seed=N + 1)).to(_TT[gt])
    packed, ws = bn.pack_i2s(dev(wl.gen_latent_w(N, K, seed=M * N + K + 5)))
    y = bn.bitlinear_forward_typed(x.cuda(), g.cuda(), packed, ws, N, wl.EPS, y_dtype=_TT[yt])
    assert y.dtype == _TT[yt] and y.shape == (M, N)
    ref = oracle_mod.bitlinear_forward_typed(x.float().numpy(), g.float().numpy(), host(packed), ws, N, wl.EPS,
                                             y_dtype=_OT[yt])
    assert_rows_close(host(y.float()), ref, f"typed forward {xt}/{gt}/{yt} M={M} K={K} N={N}")


def test_forward_typed_all_fp32_is_forward():
    M, K, N = 40, 1024, 300
    x = dev(wl.gen_x(M, K, seed=1))
    g = dev(wl.gen_norm_w(K, seed=2))
    packed, ws = bn.pack_i2s(dev(wl.gen_latent_w(N, K, seed=3)))
    assert torch.equal(bn.bitlinear_forward_typed(x, g, packed, ws, N), bn.bitlinear_forward(x, g, packed, ws, N))
    # 16-bit y is the fp32 projection of the same (widened) inputs, rounded once
    yb = bn.bitlinear_forward_typed(x, g, packed, ws, N, y_dtype=torch.bfloat16)
    assert torch.equal(yb, bn.bitlinear_forward(x, g, packed, ws, N).to(torch.bfloat16))


def test_forward_typed_argument_errors():
    x = torch.zeros((2, 128), dtype=torch.bfloat16, device="cuda")
    g = torch.zeros(128, dtype=torch.bfloat16, device="cuda")  # bf16 norm weights: not a supported type
    packed, ws = bn.pack_i2s(torch.ones((4, 128), device="cuda"))
    with pytest.raises(TypeError):
        bn.bitlinear_forward_typed(x, g, packed, ws, 4)
    y = torch.empty((2, 4), dtype=torch.float16, device="cuda")
    rc = bn.lib().bitnet_bitlinear_forward_typed(x.data_ptr(), 2, g.data_ptr(), 7, packed.data_ptr(), ws, 2, 128, 4,
                                                 1e-6, y.data_ptr(), 1, None)
    assert rc == bn.ERR_INVALID_ARG


# QK head norms: per-head RMSNorm of a projection's output (heads of 128 and
# 256 values), standalone (in place and out of place) and chained after the
# projection on every dispatch route
@pytest.mark.parametrize("M,H,hd", [(1, 16, 128), (3, 4, 256), (257, 8, 128), (4096, 1, 256)])
def test_head_rmsnorm_matches_oracle(oracle_mod, M, H, hd):
    y = wl.gen_x(M, H * hd, seed=M + hd, outlier_frac=0.01)
    if M >= 3:
        y[1, :hd] = 0.0       # a zero head stays zero
        y[2, hd:] *= 1e-20    # tiny heads
        y[0, :] *= 1e20       # huge ones
    w = wl.gen_norm_w(hd, seed=hd)
    out = bn.head_rmsnorm(dev(y), hd, dev(w), wl.EPS)
    ref = oracle_mod.head_rmsnorm(y, hd, w, wl.EPS)
    got = host(out)
    # the row arithmetic of the input norm: bit-identical rows except where
    # rstd sits on a rounding boundary (at most 1 row in 1000)
    rows_off = np.sum(np.any(got.reshape(-1, hd) != ref.reshape(-1, hd), axis=1))
    assert rows_off <= max(1, (M * H) // 1000)
    yd = dev(y)
    assert torch.equal(bn.head_rmsnorm(yd, hd, dev(w), wl.EPS, out=yd), out)  # in place


# decode and split-K routes: a second launch; tokens-as-M tiles holding whole
# heads (256- and 128-wide tiles, heads of 128 and 256): fused in the epilogue
QK_CASES = [(1, 1024, 2048, 128), (1, 640, 1024, 256), (5, 3072, 1024, 128), (16, 16384, 1024, 128),
            (300, 1024, 1024, 128), (2048, 640, 256, 256), (128, 16384, 1024, 128), (2048, 640, 640, 128)]


@pytest.mark.parametrize("M,K,N,hd", QK_CASES)
def test_forward_qk_matches_oracle(oracle_mod, M, K, N, hd):
    x = _x_with_edges(M, K, seed=M + K + N + hd)
    g = wl.gen_norm_w(K, seed=N)
    hw = wl.gen_norm_w(hd, seed=hd + 7)
    packed, ws = bn.pack_i2s(dev(wl.gen_latent_w(N, K, seed=M * N + K)))
    y = bn.bitlinear_forward_qk(dev(x), dev(g), packed, ws, N, hd, dev(hw), wl.EPS)
    # chained launch == projection then standalone head norm, bit for bit
    y2 = bn.head_rmsnorm(bn.bitlinear_forward(dev(x), dev(g), packed, ws, N, wl.EPS), hd, dev(hw), wl.EPS)
    assert torch.equal(y, y2)
    ref = oracle_mod.bitlinear_forward_qk(x, g, host(packed), ws, N, hd, hw, wl.EPS)
    assert_rows_close(host(y), ref, f"forward_qk M={M} K={K} N={N} hd={hd}")


@pytest.mark.parametrize("K", [1024, 3072, 16384])
def test_forward_is_composition_of_the_two_calls(K):
    """The row reduction is implemented three ways (registers, global re-read,
    shared memory); all must round identically, so the fused decode launch, the
    norm launch + decode launch and the norm launch + tensor-core launch agree
    bit for bit."""
    M, N = 40, 300
    x = dev(wl.gen_x(M, K, seed=1))
    g = dev(wl.gen_norm_w(K, seed=2))
    packed, ws = bn.pack_i2s(dev(wl.gen_latent_w(N, K, seed=3)))
    y1 = bn.bitlinear_forward(x, g, packed, ws, N)
    codes, a_scale, _ = bn.rmsnorm_quant_a8(x, g)
    y2 = bn.i2s_gemm(codes, a_scale, packed, ws, N)
    assert torch.equal(y1, y2)
    xs = x[:1].contiguous()
    y3 = bn.bitlinear_forward(xs, g, packed, ws, N)       # fused decode launch
    c4, s4, _ = bn.rmsnorm_quant_a8(xs, g)
    assert torch.equal(y3, bn.i2s_gemm(c4, s4, packed, ws, N))
    assert torch.equal(y3, y1[:1])


def test_forward_on_side_stream(oracle_mod):
    M, K, N = 96, 1024, 512
    x = wl.gen_x(M, K, seed=5)
    g = wl.gen_norm_w(K, seed=6)
    w = wl.gen_latent_w(N, K, seed=7)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        xd, gd, wd = dev(x), dev(g), dev(w)
        packed, ws = bn.pack_i2s(wd)
        y = bn.bitlinear_forward(xd, gd, packed, ws, N)
    s.synchronize()
    assert_rows_close(y.cpu().numpy(), oracle_mod.bitlinear_forward(x, g, packed.cpu().numpy(), ws, N), "stream")


# ---------------------------------------------------------- grouped decode

def _qwen3_layer(config, layer, M):
    projs = []
    for i, p in enumerate(wl.QWEN3_0P6B_LAYER):
        x, g, w = wl.gen_projection(config, layer, i, M, p.K, p.N)
        projs.append((p, x, g, w))
    return projs


@pytest.mark.parametrize("M", [1, 2, 8])
def test_group_matches_oracle_and_single_calls(oracle_mod, M):
    layer = _qwen3_layer(1, 0, M)
    items, refs, singles = [], [], []
    for p, x, g, w in layer:
        packed, ws = bn.pack_i2s(dev(w))
        xd, gd = dev(x), dev(g)
        y = torch.empty((M, p.N), dtype=torch.float32, device="cuda")
        items.append((xd, gd, packed, ws, p.N, y))
        refs.append(oracle_mod.bitlinear_forward(x, g, host(packed), ws, p.N))
        singles.append(bn.bitlinear_forward(xd, gd, packed, ws, p.N))
    bn.bitlinear_forward_group(items, M, wl.EPS, flags=bn.FLAG_WEIGHTS_STATIC)
    for (xd, gd, packed, ws, N, y), ref, single in zip(items, refs, singles):
        assert torch.equal(y, single)
        assert_rows_close(host(y), ref, "group")


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("flags", [0, bn.FLAG_WEIGHTS_STATIC])
def test_group_long_rows_matches_oracle(oracle_mod, M, flags):
    """Long-row projections of different widths in one grouped launch, with and
    without early weight streaming."""
    shapes = [(4096, 2048), (16384, 1000), (8192, 3000), (4096, 77)]
    items, refs, singles = [], [], []
    for i, (K, N) in enumerate(shapes):
        x = _x_with_edges(M, K, seed=100 + i)
        g = wl.gen_norm_w(K, seed=200 + i)
        packed, ws = bn.pack_i2s(dev(wl.gen_latent_w(N, K, seed=300 + i)))
        xd, gd = dev(x), dev(g)
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        items.append((xd, gd, packed, ws, N, y))
        refs.append(oracle_mod.bitlinear_forward(x, g, host(packed), ws, N, wl.EPS))
        singles.append(bn.bitlinear_forward(xd, gd, packed, ws, N, wl.EPS))
    bn.bitlinear_forward_group(items, M, wl.EPS, flags=flags)
    for (xd, gd, packed, ws, N, y), ref, single in zip(items, refs, singles):
        assert torch.equal(y, single)
        assert_rows_close(host(y), ref, "group long rows")


def test_group_in_cuda_graph_rotating_layers(oracle_mod):
    """The launch configuration the decode benchmark times: one grouped launch
    per layer, programmatic dependent launch with static weights, replayed from
    a CUDA graph over several distinct layers."""
    L = 4
    layers, descs, refs = [], [], []
    for layer in range(L):
        items, lref = [], []
        for p, x, g, w in _qwen3_layer(1, layer, 1):
            packed, ws = bn.pack_i2s(dev(w))
            y = torch.full((1, p.N), float("nan"), dtype=torch.float32, device="cuda")
            items.append((dev(x), dev(g), packed, ws, p.N, y))
            lref.append(oracle_mod.bitlinear_forward(x, g, host(packed), ws, p.N))
        layers.append(items)
        descs.append(bn.make_group(items))
        refs.append(lref)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for d in descs:  # warm-up outside capture
            bn.bitlinear_forward_group(d, 1, wl.EPS, bn.FLAG_WEIGHTS_STATIC)
    s.synchronize()
    for items in layers:
        for it in items:
            it[5].fill_(float("nan"))
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for d in descs:
            bn.bitlinear_forward_group(d, 1, wl.EPS, bn.FLAG_WEIGHTS_STATIC)
    graph.replay()
    torch.cuda.synchronize()
    for items, lref in zip(layers, refs):
        for it, ref in zip(items, lref):
            assert_rows_close(host(it[5]), ref, "graph")


# ------------------------------------------------------- full-size samples

@pytest.mark.parametrize("which", ["gemma3_gate", "qwen3_down"])
def test_full_size_prefill_sampled_rows(oracle_mod, which):
    """Prefill at the full token count of the layer/stack workloads (M=32768),
    checked on sampled rows (rows are independent)."""
    if which == "gemma3_gate":
        M, K, N, frac = 32768, 640, 2048, 0.01
    else:
        M, K, N, frac = 32768, 3072, 1024, 0.0
    x = wl.gen_x(M, K, seed=K + N, outlier_frac=frac)
    g = wl.gen_norm_w(K, seed=K)
    w = wl.gen_latent_w(N, K, seed=N)
    packed, ws = bn.pack_i2s(dev(w))
    y = bn.bitlinear_forward(dev(x), dev(g), packed, ws, N)
    rows = np.unique(np.concatenate([np.arange(4), np.arange(M - 4, M),
                                     np.random.default_rng(0).choice(M, 56, replace=False)]))
    ref = oracle_mod.bitlinear_forward(x[rows], g, host(packed), ws, N)
    yh = host(y)
    assert_rows_close(yh[rows], ref, which)
    assert np.isfinite(yh).all()


# ------------------------------------------- down projection: act(gate) * up input

def _gate_up(M, K, seed):
    rng = np.random.default_rng(seed)
    gate = rng.normal(0.0, 2.0, (M, K)).astype(np.float32)
    up = rng.normal(0.0, 1.0, (M, K)).astype(np.float32)
    # edge values of the activations: far tails, zero, tiny
    edge = np.array([0.0, -0.0, 1e-30, -1e-30, 30.0, -30.0, 90.0, -90.0, 200.0, -200.0, 4.0, -4.0], np.float32)
    gate[0, : edge.size] = edge
    return gate, up


@pytest.mark.parametrize("act", [bn.ACT_SILU, bn.ACT_GELU_TANH])
def test_glu_matches_oracle(oracle_mod, act):
    """h = act(gate) * up against the oracle (activation in double, rounded once):
    the GPU's x * 1/(1 + expf(-t)) is within a few ulp of it, in relative terms
    except where the result underflows."""
    gate, up = _gate_up(37, 1024, seed=act)
    h = host(bn.glu(dev(gate), dev(up), act))
    ref = oracle_mod.glu(gate, up, act)
    assert np.all(np.isfinite(h))
    tol = 2e-6 * np.abs(ref) + 4e-7 * np.abs(gate) * np.abs(up) + 1e-37
    bad = np.abs(h - ref) > tol
    assert not bad.any(), (gate[bad][:5], h[bad][:5], ref[bad][:5])


@pytest.mark.parametrize("K", [640, 2048, 3072, 1152])
@pytest.mark.parametrize("act", [bn.ACT_SILU, bn.ACT_GELU_TANH])
def test_glu_norm_is_composition(K, act):
    """The norm launch that computes act(gate) * up as it loads the rows gives
    the same bits as bitnet_glu followed by the plain norm launch."""
    M = 21
    gate, up = _gate_up(M, K, seed=K + act)
    g = dev(wl.gen_norm_w(K, seed=K))
    gd, ud = dev(gate), dev(up)
    rs1 = torch.empty(M, dtype=torch.int32, device="cuda")
    xn1 = torch.empty((M, K), dtype=torch.float32, device="cuda")
    c1, s1, _ = bn.glu_rmsnorm_quant_a8(gd, ud, act, g, wl.EPS, rowsum=rs1, xn_out=xn1)
    rs2 = torch.empty(M, dtype=torch.int32, device="cuda")
    xn2 = torch.empty((M, K), dtype=torch.float32, device="cuda")
    c2, s2, _ = bn.rmsnorm_quant_a8(bn.glu(gd, ud, act), g, wl.EPS, rowsum=rs2, xn_out=xn2)
    assert torch.equal(c1, c2) and torch.equal(s1, s2) and torch.equal(rs1, rs2) and torch.equal(xn1, xn2)


GLU_CASES = [
    # fused decode launch (rows in registers): Qwen3 and Gemma3 down projections at M=1, long rows
    (1, 3072, 1024, bn.ACT_SILU), (1, 2048, 640, bn.ACT_GELU_TANH), (1, 8192, 300, bn.ACT_SILU),
    (3, 12288, 200, bn.ACT_GELU_TANH),
    # norm launch with the activation (K <= 3072), then the decode launch on int8 codes
    (2, 3072, 512, bn.ACT_SILU),
    # h written first (K > 3072, not a register-prologue shape), then norm and decode
    (1, 4224, 100, bn.ACT_GELU_TANH),
    # tensor-core paths: split-K (K >= 4096, h through memory) and tokens-as-M (activation in the norm launch)
    (40, 6144, 300, bn.ACT_SILU), (16, 2048, 640, bn.ACT_GELU_TANH), (300, 3072, 257, bn.ACT_SILU),
]


@pytest.mark.parametrize("M,K,N,act", GLU_CASES)
def test_forward_glu_matches_composition_and_oracle(oracle_mod, M, K, N, act):
    gate, up = _gate_up(M, K, seed=M * K + N)
    g = wl.gen_norm_w(K, seed=N + act)
    w = wl.gen_latent_w(N, K, seed=K + N)
    packed, ws = bn.pack_i2s(dev(w))
    gd, ud, gw = dev(gate), dev(up), dev(g)
    y = bn.bitlinear_forward_glu(gd, ud, act, gw, packed, ws, N, wl.EPS)
    h = bn.glu(gd, ud, act)
    assert torch.equal(y, bn.bitlinear_forward(h, gw, packed, ws, N, wl.EPS))
    # the GPU's h through the oracle: the same projection; the oracle's own h (activation
    # rounded from double, a few ulp away): within the row tolerance
    assert_rows_close(host(y), oracle_mod.bitlinear_forward(host(h), g, host(packed), ws, N, wl.EPS),
                      f"glu forward M={M} K={K} N={N} (GPU h)")
    assert_rows_within_tolerance(
        host(y), oracle_mod.bitlinear_forward_glu(gate, up, act, g, host(packed), ws, N, wl.EPS),
        f"glu forward M={M} K={K} N={N}")
