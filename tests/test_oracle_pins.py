"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test ties one oracle function to what the pages or mathematics fix:
hand-worked bytes of the I2_S packing passage, closed forms, library routines
(torch rms_norm in float64, numpy integer matmul) and error bounds.
"""
import math
import os
import struct

import numpy as np
import pytest

from bitlinear_rmsnorm_token_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "i2s_worked_blocks.txt")


def _golden_rows():
    rows = {}
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        name, hx = line.rstrip("\n").split("\t")
        rows[name] = bytes.fromhex(hx)
    return rows


def _pattern(name):
    """The 128 ternary values each worked block describes."""
    v = np.zeros(128, dtype=np.int8)
    if name == "all_plus_one":
        v[:] = 1
    elif name == "all_zero":
        pass
    elif name == "all_minus_one":
        v[:] = -1
    elif name == "quarters":
        v[0:32], v[32:64], v[64:96], v[96:128] = -1, 0, 1, 0
    elif name == "first_plus":
        v[0] = 1
    elif name == "e97_minus":
        v[97] = -1
    elif name == "mod3":
        v[:] = np.arange(128) % 3 - 1
    else:
        raise KeyError(name)
    return v


# ------------------------------------------------------------ packing pins ---

@pytest.mark.parametrize("name", list(_golden_rows().keys()))
def test_worked_block_encode(oracle_mod, name):
    expected = _golden_rows()[name]
    q = _pattern(name).reshape(1, 128)
    out = oracle_mod.encode_i2s(q, 1.0)
    assert bytes(out[:32]) == expected
    assert bytes(out[32:]) == struct.pack("<f", 1.0)


@pytest.mark.parametrize("name", [n for n in _golden_rows() if n != "all_zero"])
def test_worked_block_pack_from_float(oracle_mod, name):
    """Absmean quantisation of c * pattern recovers the pattern (every non-zero
    entry lands at >= 1 after scaling and clamps to +-1) and the same bytes."""
    expected = _golden_rows()[name]
    q = _pattern(name)
    c = 0.37
    w = (q.astype(np.float32) * np.float32(c)).reshape(1, 128)
    packed, s = oracle_mod.pack_i2s(w)
    assert bytes(packed[:32]) == expected
    nnz = int(np.count_nonzero(q))
    assert s == pytest.approx(128.0 / (c * nnz), rel=2 ** -22)
    assert struct.unpack("<f", bytes(packed[32:36]))[0] == s


def test_all_zero_tensor_scale_is_one(oracle_mod):
    packed, s = oracle_mod.pack_i2s(np.zeros((2, 128), np.float32))
    assert s == 1.0
    assert bytes(packed[:64]) == b"\x55" * 64


def test_multi_row_block_order(oracle_mod):
    """Row n, block kb sits at byte offset 32 * (n*K/128 + kb): use distinct
    constant rows/blocks so any misplacement changes the bytes."""
    N, K = 3, 256
    q = np.zeros((N, K), np.int8)
    q[0, :128] = 1
    q[0, 128:] = -1
    q[1, :128] = 0
    q[1, 128:] = 1
    q[2, :] = -1
    out = oracle_mod.encode_i2s(q, 2.0)
    exp = b"\xaa" * 32 + b"\x00" * 32 + b"\x55" * 32 + b"\xaa" * 32 + b"\x00" * 64
    assert bytes(out[:192]) == exp
    assert bytes(out[192:]) == struct.pack("<f", 2.0)


def test_round_half_to_even(oracle_mod):
    """Reading of "round": rint.  mean|w| = 1 so w_scale = 1 and the products
    are exactly +-0.5 / +-1.5: 0.5 -> 0, 1.5 -> 2 -> clamped 1."""
    w = np.array([1.5] * 32 + [0.5] * 32 + [-0.5] * 32 + [-1.5] * 32, np.float32).reshape(1, 128)
    assert oracle_mod.weight_scale(w) == 1.0
    q = oracle_mod.quantize_ternary(w, 1.0)
    assert (q[0, :32] == 1).all() and (q[0, 32:96] == 0).all() and (q[0, 96:] == -1).all()


def test_mean_abs_matches_numpy(oracle_mod):
    w = wl.gen_latent_w(257, 384, seed=11)
    ref = float(np.mean(np.abs(w.astype(np.float64))))
    assert oracle_mod.mean_abs(w) == pytest.approx(ref, rel=1e-13)


def test_gaussian_ternary_statistics(oracle_mod):
    """For w ~ N(0, s), w_scale = 1/E|w| = 1/(s sqrt(2/pi)), so P(q = 0) =
    P(|z| < 0.5 sqrt(2/pi)) = erf(0.5/sqrt(pi)) = 0.3101 and P(+1) = P(-1)."""
    w = wl.gen_latent_w(1024, 1024, seed=5)
    packed, s = oracle_mod.pack_i2s(w)
    q = oracle_mod.unpack_i2s(packed, 1024, 1024)
    p0 = math.erf(0.5 / math.sqrt(math.pi))
    assert abs(p0 - 0.3101) < 1e-4
    frac0 = float(np.mean(q == 0))
    assert abs(frac0 - p0) < 0.003
    assert abs(float(np.mean(q == 1)) - (1 - p0) / 2) < 0.003
    assert abs(float(np.mean(q == -1)) - (1 - p0) / 2) < 0.003
    assert set(np.unique(q).tolist()) <= {-1, 0, 1}
    assert oracle_mod.count_invalid_codes(packed, 1024, 1024) == 0
    # the scale is the reciprocal of the double-precision mean, rounded once
    assert s * oracle_mod.mean_abs(w) == pytest.approx(1.0, abs=2 ** -23)


def test_unpack_inverts_encode(oracle_mod):
    rng = np.random.default_rng(3)
    q = rng.integers(-1, 2, size=(5, 384), dtype=np.int8)
    packed = oracle_mod.encode_i2s(q, 1.5)
    assert np.array_equal(oracle_mod.unpack_i2s(packed, 5, 384), q)


def test_encode_inverts_unpack_on_valid_bytes(oracle_mod):
    """Every byte whose four fields avoid code 3 survives decode + encode."""
    vals = [b for b in range(256) if all(((b >> s) & 3) != 3 for s in (0, 2, 4, 6))]
    assert len(vals) == 81
    stream = np.array((vals * 2)[:160] + [0x55] * 96, np.uint8)  # 256 bytes = 8 blocks
    packed = np.concatenate([stream, np.frombuffer(struct.pack("<f", 1.0), np.uint8)])
    q = oracle_mod.unpack_i2s(packed, 2, 512)
    assert np.array_equal(oracle_mod.encode_i2s(q, 1.0), packed)


def test_invalid_code_count(oracle_mod):
    packed = np.full(32 + 4, 0x55, np.uint8)
    packed[3] = 0xFF  # four fields of code 3
    packed[7] = 0x57  # one
    assert oracle_mod.count_invalid_codes(packed, 1, 128) == 5
    q = oracle_mod.unpack_i2s(packed, 1, 128)
    assert q[0, 3] == 2 and q[0, 32 + 3] == 2 and q[0, 96 + 7] == 2


# ------------------------------------------------------------- RMSNorm pins ---

def _torch_rmsnorm64(x, g, eps):
    import torch

    xt = torch.from_numpy(x.astype(np.float64))
    return (torch.nn.functional.rms_norm(xt, (x.shape[1],), eps=eps) *
            torch.from_numpy(g.astype(np.float64))).numpy()


@pytest.mark.parametrize("K", [128, 640, 1024, 3072])
def test_rmsnorm_matches_torch_f64(oracle_mod, K):
    x = wl.gen_x(9, K, seed=K)
    x[3] = 0.0  # a zero row stays zero (eps keeps rstd finite)
    x[4] *= 1e-3
    g = wl.gen_norm_w(K, seed=K + 1)
    xn = oracle_mod.rmsnorm(x, g, wl.EPS)
    ref = _torch_rmsnorm64(x, g, wl.EPS)
    # three roundings (rstd to float, then two float multiplies), each at most
    # 2^-24 relative
    tol = 3.01 * 2.0 ** -24 * np.abs(ref) + 1e-30
    assert np.all(np.abs(xn - ref) <= tol)
    assert np.all(xn[3] == 0.0)


def test_rmsnorm_eps_placement(oracle_mod):
    """eps is added to the mean square, inside the square root: for a constant
    row x = c with g = 1, xn = c / sqrt(c^2 + eps)."""
    c = 1e-3
    x = np.full((1, 128), c, np.float32)
    g = np.ones(128, np.float32)
    xn = oracle_mod.rmsnorm(x, g, 1e-6)
    want = float(np.float32(c)) / math.sqrt(float(np.float32(c)) ** 2 + float(np.float32(1e-6)))
    assert xn[0, 0] == pytest.approx(want, rel=3e-7)
    assert abs(want - 0.7071) < 1e-3  # c^2 = eps: the eps term halves the mean square


# ---------------------------------------------------------- activation pins ---

def test_quant_a8_invariants(oracle_mod):
    K = 1024
    x = wl.gen_x(6, K, seed=21, outlier_frac=0.01)
    x[2] = 0.0
    x[3] = 0.75
    g = wl.gen_norm_w(K, seed=22)
    xn = oracle_mod.rmsnorm(x, g, wl.EPS)
    xn[3] = oracle_mod.rmsnorm(x[3:4], np.ones(K, np.float32), wl.EPS)[0]
    q, s, rs = oracle_mod.quant_a8(xn)
    assert np.all(np.abs(q.astype(np.int32)) <= 127)
    assert np.array_equal(rs, q.astype(np.int64).sum(axis=1).astype(np.int32))
    for m in range(6):
        amax = float(np.max(np.abs(xn[m])))
        if amax == 0.0:
            assert np.all(q[m] == 0)
            assert s[m] == np.float32(127.0) / np.float32(1e-5)
            continue
        # the largest entry lands on +-127
        k = int(np.argmax(np.abs(xn[m])))
        assert abs(int(q[m, k])) == 127
        # scale is 127 / amax up to one rounding
        assert float(s[m]) * amax == pytest.approx(127.0, rel=2 ** -23)
        # each code is the nearest integer to xn * a_scale
        err = np.abs(xn[m].astype(np.float64) * float(s[m]) - q[m])
        assert float(err.max()) <= 0.5 + 1e-5
    assert np.all(np.abs(q[3]) == 127)  # constant row, unit norm weight


# --------------------------------------------------------- contraction pins ---

def test_matmul_matches_numpy(oracle_mod):
    rng = np.random.default_rng(7)
    M, K, N = 5, 384, 7
    q = rng.integers(-128, 128, size=(M, K), dtype=np.int8)
    t = rng.integers(-1, 2, size=(N, K), dtype=np.int8)
    packed = oracle_mod.encode_i2s(t, 1.0)
    acc = oracle_mod.i2s_matmul(q, packed, N)
    assert np.array_equal(acc, q.astype(np.int64) @ t.astype(np.int64).T)


def test_matmul_special_weights(oracle_mod):
    rng = np.random.default_rng(8)
    M, K = 4, 128
    q = rng.integers(-128, 128, size=(M, K), dtype=np.int8)
    rowsum = q.astype(np.int64).sum(axis=1)
    for val, want in ((1, rowsum), (0, 0 * rowsum), (-1, -rowsum)):
        t = np.full((3, K), val, np.int8)
        acc = oracle_mod.i2s_matmul(q, oracle_mod.encode_i2s(t, 1.0), 3)
        assert np.array_equal(acc, np.repeat(np.asarray(want)[:, None], 3, axis=1))
    eye = np.eye(128, dtype=np.int8)  # one-hot rows pick single features
    acc = oracle_mod.i2s_matmul(q, oracle_mod.encode_i2s(eye, 1.0), 128)
    assert np.array_equal(acc, q.astype(np.int64))


def test_matmul_extreme_sums(oracle_mod):
    """Largest magnitudes the int32 accumulator meets at K = 16384."""
    K = 16384
    q = np.full((2, K), 127, np.int8)
    q[1, 1::2] = -127
    t = np.ones((2, K), np.int8)
    t[1, 1::2] = -1
    acc = oracle_mod.i2s_matmul(q, oracle_mod.encode_i2s(t, 1.0), 2)
    assert acc[0, 0] == 127 * K and acc[1, 1] == 127 * K
    assert acc[0, 1] == 0 and acc[1, 0] == 0


def test_rescale_against_f64(oracle_mod):
    rng = np.random.default_rng(9)
    acc = rng.integers(-2_000_000, 2_000_000, size=(6, 11), dtype=np.int64)
    a_scale = rng.uniform(1.0, 200.0, size=6).astype(np.float32)
    w_scale = np.float32(37.25)
    y = oracle_mod.rescale(acc, a_scale, float(w_scale))
    ref = acc / a_scale.astype(np.float64)[:, None] / float(w_scale)
    # two reciprocals and two products, each rounded once
    assert np.all(np.abs(y - ref) <= 4 * 2.0 ** -24 * np.abs(ref))


def _nearest_f32(r):
    """The float32 nearest to the rational r, ties to the even significand, found
    from the exact value alone (no float32 arithmetic): normal range only."""
    from fractions import Fraction

    if r == 0:
        return 0.0
    a = abs(r)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    assert -126 <= e <= 127
    unit = Fraction(2) ** (e - 23)
    m = round(a / unit)  # Fraction rounding: half to even
    v = m * unit
    return float(v if r > 0 else -v)


def test_rescale_each_operation_rounded_once_in_stated_order(oracle_mod):
    """y = ((float)acc * (1/a_scale)) * (1/w_scale): each of the two reciprocals
    and two products is the float32 nearest to its exact rational value, in that
    order.  The other order gives different bits on these inputs, so a swapped
    order fails here."""
    from fractions import Fraction as F

    rng = np.random.default_rng(19)
    acc = rng.integers(-2_000_000, 2_000_000, size=(8, 16), dtype=np.int64)
    a_scale = rng.uniform(1.0, 200.0, size=8).astype(np.float32)
    w_scale = np.float32(rng.uniform(10.0, 80.0))
    y = oracle_mod.rescale(acc, a_scale, float(w_scale))
    inv_w = F(_nearest_f32(1 / F(float(w_scale))))
    other_order = 0
    for m in range(acc.shape[0]):
        inv_a = F(_nearest_f32(1 / F(float(a_scale[m]))))
        for n in range(acc.shape[1]):
            a = F(int(acc[m, n]))  # |acc| < 2^24: exact in float
            want = _nearest_f32(F(_nearest_f32(a * inv_a)) * inv_w)
            assert float(y[m, n]) == want, (m, n)
            other_order += _nearest_f32(F(_nearest_f32(a * inv_w)) * inv_a) != want
    assert other_order > 0


def _exact_dequant_dot(q, t, a, w):
    """sum_k (q_k / a) * (t_k / w) in exact rationals."""
    from fractions import Fraction as F

    s = sum(int(qk) * int(tk) for qk, tk in zip(q, t))
    return F(s) / (F(float(a)) * F(float(w)))


@pytest.mark.parametrize("M,K,N", [(1, 128, 1), (5, 128, 33), (17, 256, 9), (3, 256, 32)])
def test_forward_matches_f64_dequantised_product(oracle_mod, M, K, N):
    """The brute-force double product of the dequantised codes,
    sum_k (q/a_scale)(t/w_scale), against the exact rationals, and the oracle's
    float y against it: acc is exact in float (|acc| < 2^24), then two
    reciprocals and two products each add at most 2^-24 relative error."""
    x, g, w = wl.gen_projection(0, K, N, M, K, N)
    x[0, :] = 0.0  # a zero row: y must be exactly zero
    if M > 2:
        x[2, :] = 3.0  # a constant row: its codes follow the norm weight, largest +127
    packed, ws = oracle_mod.pack_i2s(w)
    y, xn, q, a_s, acc = oracle_mod.bitlinear_forward(x, g, packed, ws, N, intermediates=True)
    t = oracle_mod.quantize_ternary(w, ws)  # the weights' own ternary values (not unpacked)
    y64 = oracle_mod.dequant_dot_f64(q, t, a_s, ws)
    # double accumulation: at most (K+2) 2^-53 of the sum of |terms| from exact
    sum_abs = (np.abs(q).astype(np.float64) @ np.abs(t).astype(np.float64).T) / a_s.astype(np.float64)[:, None] / float(ws)
    acc_err = 1.01 * (K + 2) * 2.0 ** -53 * sum_abs
    rng = np.random.default_rng(M * N)
    for m, n in [(0, 0), (M - 1, N - 1)] + [tuple(v) for v in zip(rng.integers(0, M, 6), rng.integers(0, N, 6))]:
        exact = _exact_dequant_dot(q[m], t[n], a_s[m], ws)
        assert abs(float(exact) - y64[m, n]) <= acc_err[m, n] + 1e-300
    assert np.all(np.abs(y.astype(np.float64) - y64) <= 4.01 * 2.0 ** -24 * np.abs(y64) + 2 * acc_err)
    assert np.all(y[0] == 0.0)
    if M > 2:
        assert q[2].max() == 127 and q[2].min() > 0


# ------------------------------------------------------------ whole chain ---

@pytest.mark.parametrize("M,K,N", [(3, 128, 5), (4, 640, 33), (2, 1024, 17)])
def test_forward_within_quantisation_bound(oracle_mod, M, K, N):
    """y against the unquantised activations: sum_k t * (q/a_scale - xn) is at
    most sum_k |t| * 0.5 / a_scale, all divided by w_scale."""
    x = wl.gen_x(M, K, seed=M * K, outlier_frac=0.01)
    g = wl.gen_norm_w(K, seed=N)
    w = wl.gen_latent_w(N, K, seed=K + N)
    packed, ws = oracle_mod.pack_i2s(w)
    y, xn, q, a_s, acc = oracle_mod.bitlinear_forward(x, g, packed, ws, N, intermediates=True)
    t = oracle_mod.quantize_ternary(w, ws).astype(np.float64)  # independent of unpack
    xn64 = _torch_rmsnorm64(x, g, wl.EPS)
    ideal = xn64 @ (t / float(ws)).T
    bound = (np.abs(t).sum(axis=1)[None, :] * 0.5 / a_s.astype(np.float64)[:, None]) / float(ws)
    assert np.all(np.abs(y - ideal) <= 1.01 * bound + 1e-5 * np.abs(ideal) + 1e-6)
    # and exactly the integer product of the codes
    assert np.array_equal(acc, q.astype(np.int64) @ t.astype(np.int64).T)


def test_forward_rows_subset(oracle_mod):
    M, K, N = 7, 256, 9
    x, g, w = wl.gen_projection(0, 0, 0, M, K, N)
    packed, ws = oracle_mod.pack_i2s(w)
    full = oracle_mod.bitlinear_forward(x, g, packed, ws, N)
    rows = np.array([6, 0, 3])
    part = oracle_mod.bitlinear_forward(x, g, packed, ws, N, rows=rows)
    assert np.array_equal(part, full[rows])


# ------------------------------------------- down-projection input (act(gate) * up)

def test_activation_silu_pins(oracle_mod):
    """SiLU is x times the logistic function (scipy's expit, a library routine);
    it is 0 at 0, has slope 1/2 there, tends to x for large x and to 0 for very
    negative x, and silu(x) - silu(-x) = x."""
    special = pytest.importorskip("scipy.special")
    act = oracle_mod.ACT_SILU
    xs = np.linspace(-30.0, 30.0, 1201)
    for x in xs:
        ref = x * special.expit(x)
        assert oracle_mod.activation(x, act) == pytest.approx(ref, rel=1e-14, abs=1e-300)
    assert oracle_mod.activation(0.0, act) == 0.0
    assert oracle_mod.activation(1e-8, act) / 1e-8 == pytest.approx(0.5, rel=1e-7)
    assert oracle_mod.activation(40.0, act) == pytest.approx(40.0, rel=1e-15)
    assert 0.0 > oracle_mod.activation(-40.0, act) > -1e-15
    for x in (0.25, 1.0, 3.5, 12.0):
        assert oracle_mod.activation(x, act) - oracle_mod.activation(-x, act) == pytest.approx(x, rel=1e-14)


def test_activation_gelu_tanh_pins(oracle_mod):
    """gelu_pytorch_tanh approximates x * Phi(x) (Phi from scipy's ndtr) to within
    5e-4 everywhere (its largest deviation, ~4.7e-4, is near x = -2.7; a wrong or
    missing cubic term is far outside that); it is 0 at 0 with slope 1/2, tends to
    x for large x, and gelu(x) - gelu(-x) = x (tanh is odd)."""
    special = pytest.importorskip("scipy.special")
    act = oracle_mod.ACT_GELU_TANH
    xs = np.linspace(-8.0, 8.0, 1601)
    dev = [abs(oracle_mod.activation(x, act) - x * special.ndtr(x)) for x in xs]
    assert max(dev) < 5e-4
    assert max(dev) > 4e-4  # the approximation, not the exact GELU
    assert oracle_mod.activation(0.0, act) == 0.0
    assert oracle_mod.activation(1e-8, act) / 1e-8 == pytest.approx(0.5, rel=1e-7)
    assert oracle_mod.activation(12.0, act) == pytest.approx(12.0, rel=1e-15)
    assert abs(oracle_mod.activation(-12.0, act)) < 1e-30
    for x in (0.25, 1.0, 2.7, 6.0):
        assert oracle_mod.activation(x, act) - oracle_mod.activation(-x, act) == pytest.approx(x, rel=1e-14)


@pytest.mark.parametrize("act", [1, 2])
def test_glu_operation_order(oracle_mod, act):
    """h = float(act(gate)) * up: with up = 1 it is the activation rounded once to
    float, with up = 0 it is 0, and otherwise one float multiply of the two."""
    rng = np.random.default_rng(act)
    gate = rng.normal(0, 2, (7, 128)).astype(np.float32)
    up = rng.normal(0, 1, (7, 128)).astype(np.float32)
    a = np.array([[np.float32(oracle_mod.activation(float(v), act)) for v in r] for r in gate], dtype=np.float32)
    assert np.array_equal(oracle_mod.glu(gate, np.ones_like(up), act), a)
    assert not np.any(oracle_mod.glu(gate, np.zeros_like(up), act))
    assert np.array_equal(oracle_mod.glu(gate, up, act), (a * up).astype(np.float32))


def test_glu_forward_is_forward_of_glu(oracle_mod):
    """The down projection is the plain projection applied to h."""
    rng = np.random.default_rng(3)
    M, K, N = 3, 256, 40
    gate = rng.normal(0, 1, (M, K)).astype(np.float32)
    up = rng.normal(0, 1, (M, K)).astype(np.float32)
    g = wl.gen_norm_w(K, seed=4)
    packed, ws = oracle_mod.pack_i2s(wl.gen_latent_w(N, K, seed=5))
    y = oracle_mod.bitlinear_forward_glu(gate, up, 1, g, packed, ws, N)
    assert np.array_equal(y, oracle_mod.bitlinear_forward(oracle_mod.glu(gate, up, 1), g, packed, ws, N))


# --------------------------------------------------------- 16-bit tensors
# Rounding fp32 to bfloat16 / fp16 (IEEE 754, nearest, ties to even) is pinned
# against a brute-force search: of the two representable neighbours of each
# input (its value truncated toward zero in the format, and the next value up
# in magnitude, infinity past the largest finite one), the nearer one, the one
# with an even last significand bit on a tie; distances in fp64 are exact.

def _bf16_neighbours(x):
    u = np.asarray(x, np.float32).view(np.uint32)
    lo = (u & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)
    # the next bfloat16 up in magnitude; past the largest finite, 2^128 stands
    # in for the rounding (it is where infinity takes over)
    step = np.ldexp(1.0, (np.frexp(np.abs(lo))[1] - 8).astype(np.int32))
    hi = lo + np.sign(x.astype(np.float64)) * step
    lo_even = ((u >> 16) & 1) == 0
    return lo, hi, lo_even


def test_bf16_rounding_worked_values(oracle_mod):
    cases = [
        (1.0, 1.0),
        (1.0 + 2.0**-8, 1.0),                      # halfway, 1.0 is even: stays
        (1.0 + 3 * 2.0**-8, 1.0 + 2.0**-6),        # halfway, 1 + 2^-7 is odd: up
        (1.0 + 2.0**-8 + 2.0**-20, 1.0 + 2.0**-7),  # just past halfway: up
        (-(1.0 + 2.0**-8 + 2.0**-20), -(1.0 + 2.0**-7)),
        (1.0 + 2.0**-8 - 2.0**-20, 1.0),           # just below halfway: down
        (3.0e38, 226 * 2.0**120),                   # 225.7 units of 2^120 at this exponent
        (65504.0, 65536.0),
    ]
    x = np.array([c[0] for c in cases], np.float32)
    want = np.array([c[1] for c in cases], np.float32)
    assert np.array_equal(oracle_mod.round_bf16(x), want)
    big = np.array([np.finfo(np.float32).max], np.float32)
    assert np.isinf(oracle_mod.round_bf16(big)[0])  # past the largest bfloat16 by more than half a unit


def test_bf16_rounding_is_nearest_even(oracle_mod):
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 0x7F7FFFFF, size=200000, dtype=np.uint32)
    bits[:1000] = (bits[:1000] & 0xFFFF0000) | 0x8000  # exact ties
    x = bits.view(np.float32) * np.where(rng.random(bits.size) < 0.5, -1, 1).astype(np.float32)
    x = x[np.abs(x) >= np.finfo(np.float32).tiny]  # normal numbers
    lo, hi, lo_even = _bf16_neighbours(x)
    xd = x.astype(np.float64)
    dlo, dhi = np.abs(xd - lo), np.abs(hi - xd)
    want = np.where((dlo < dhi) | ((dlo == dhi) & lo_even), lo, hi)
    want = np.where(np.abs(want) >= 2.0**128, np.sign(want) * np.inf, want)
    got = oracle_mod.round_bf16(x).astype(np.float64)
    assert np.array_equal(got, want)


def test_f16_rounding_is_nearest_even(oracle_mod):
    rng = np.random.default_rng(12)
    x = np.concatenate([rng.normal(0, 300, 50000), rng.uniform(-70000, 70000, 50000),
                        rng.normal(0, 1e-5, 20000)]).astype(np.float32)
    all16 = np.arange(0, 0x7C01, dtype=np.uint16).view(np.float16).astype(np.float64)  # 0 .. +inf, ascending
    mag = np.abs(x.astype(np.float64))
    i = np.clip(np.searchsorted(all16, mag, side="right") - 1, 0, all16.size - 2)
    lo, hi = all16[i], all16[i + 1]
    hi_f = np.where(np.isinf(hi), 65536.0, hi)  # where infinity takes over
    lo_even = (i % 2) == 0
    pick = np.where((mag - lo < hi_f - mag) | ((mag - lo == hi_f - mag) & lo_even), lo, hi)
    want = np.sign(x) * pick
    got = oracle_mod.round_f16(x).astype(np.float64)
    assert np.array_equal(got, want)
    # worked values: 65504 is the largest finite; the halfway point to 65536 rounds to infinity (even)
    v = oracle_mod.round_f16(np.array([65504.0, 65519.0, 65520.0, 1 + 2.0**-11, 1 + 3 * 2.0**-11], np.float32))
    assert v[0] == 65504.0 and v[1] == 65504.0 and np.isinf(v[2]) and v[3] == 1.0 and v[4] == 1 + 2.0**-9


def test_rounding_is_idempotent_and_widening_exact(oracle_mod):
    x = np.random.default_rng(13).normal(0, 10, 10000).astype(np.float32)
    for rnd in (oracle_mod.round_bf16, oracle_mod.round_f16):
        r = rnd(x)
        assert np.array_equal(rnd(r), r)
    # the oracle's rounding agrees with torch's casts (a second implementation)
    import torch
    t = torch.from_numpy(x)
    assert np.array_equal(oracle_mod.round_bf16(x), t.to(torch.bfloat16).float().numpy())
    assert np.array_equal(oracle_mod.round_f16(x), t.to(torch.float16).float().numpy())


def test_typed_forward_rounds_the_fp32_projection(oracle_mod):
    rng = np.random.default_rng(14)
    M, K, N = 3, 256, 50
    x = oracle_mod.round_bf16(rng.normal(0, 1, (M, K)).astype(np.float32))
    g = oracle_mod.round_f16(wl.gen_norm_w(K, seed=2))
    packed, ws = oracle_mod.pack_i2s(wl.gen_latent_w(N, K, seed=3))
    y32 = oracle_mod.bitlinear_forward(x, g, packed, ws, N)
    assert np.array_equal(oracle_mod.bitlinear_forward_typed(x, g, packed, ws, N, y_dtype=oracle_mod.DTYPE_F32), y32)
    yb = oracle_mod.bitlinear_forward_typed(x, g, packed, ws, N, y_dtype=oracle_mod.DTYPE_BF16)
    assert np.array_equal(yb, oracle_mod.round_bf16(y32))
    assert np.all(np.abs(yb - y32) <= np.abs(y32) * 2.0**-8)  # half a unit of 8 significand bits


# ------------------------------------------------------------ QK head norms

@pytest.mark.parametrize("hd", [128, 256])
def test_head_rmsnorm_matches_torch_per_head(oracle_mod, hd):
    M, H = 5, 4
    y = wl.gen_x(M, H * hd, seed=hd)
    y[:, hd:2 * hd] *= 37.0   # heads at different scales
    y[2, 3 * hd:] = 0.0       # a zero head stays zero
    w = wl.gen_norm_w(hd, seed=hd + 1)
    out = oracle_mod.head_rmsnorm(y, hd, w, wl.EPS)
    # torch's rms_norm over the last dimension of [M, H, hd], in float64
    import torch
    ref = torch.nn.functional.rms_norm(torch.from_numpy(y.astype(np.float64)).reshape(M, H, hd), (hd,),
                                       torch.from_numpy(w.astype(np.float64)), eps=wl.EPS).reshape(M, H * hd).numpy()
    tol = 3.01 * 2.0 ** -24 * np.abs(ref) + 1e-30
    assert np.all(np.abs(out - ref) <= tol)
    assert np.all(out[2, 3 * hd:] == 0.0)
    # per head, not per row: the whole-row norm of the same data differs
    whole = oracle_mod.rmsnorm(y, np.tile(w, H), wl.EPS)
    assert not np.allclose(whole, out, rtol=1e-3)


def test_head_rmsnorm_heads_are_independent(oracle_mod):
    hd, H = 128, 3
    y = wl.gen_x(2, H * hd, seed=9)
    w = np.ones(hd, np.float32)
    base = oracle_mod.head_rmsnorm(y, hd, w, wl.EPS)
    y2 = y.copy()
    y2[:, :hd] *= 8.0  # a power of two: the head's rstd scales exactly, its output is unchanged up to eps
    out = oracle_mod.head_rmsnorm(y2, hd, w, wl.EPS)
    assert np.array_equal(out[:, hd:], base[:, hd:])
    assert np.allclose(out[:, :hd], base[:, :hd], rtol=1e-6)
    # unit weights: every head's mean square is 1 up to eps
    ms = (base.astype(np.float64) ** 2).reshape(2, H, hd).mean(axis=2)
    assert np.allclose(ms, 1.0, rtol=1e-5)


def test_forward_qk_is_head_norm_of_forward(oracle_mod):
    M, K, N, hd = 3, 256, 256, 128
    x = wl.gen_x(M, K, seed=1)
    g = wl.gen_norm_w(K, seed=2)
    hw = wl.gen_norm_w(hd, seed=3)
    packed, ws = oracle_mod.pack_i2s(wl.gen_latent_w(N, K, seed=4))
    y = oracle_mod.bitlinear_forward_qk(x, g, packed, ws, N, hd, hw)
    assert np.array_equal(y, oracle_mod.head_rmsnorm(oracle_mod.bitlinear_forward(x, g, packed, ws, N), hd, hw))
