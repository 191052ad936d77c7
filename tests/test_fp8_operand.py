"""The numerical basis of the 8-bit operands of the 9..63-token contraction,
checked from the e4m3 format's definition (no GPU needed).

That contraction multiplies e4m3 weights by e4m3 token values with fp32
accumulation and must reproduce the exact integer sum_k q[m, k] (code - 1):
  - a weight is its 2-bit I2_S code c in {0, 1, 2} taken as an e4m3 byte, which
    must be the value c * 2^-9 (a subnormal, or the smallest normal);
  - a token code q (int8, |q| <= 127) is split as q = 16 hi + lo with
    hi = floor(q / 16) in [-8, 7] and lo = q mod 16 in [0, 15], both of which
    must be exact e4m3 values;
  - each accumulator column holds 2^-9 sum c * plane over up to K = 65536
    terms, which must stay exactly representable in fp32, as must the
    recombined sum 16 D_hi + D_lo and its difference with the code row sum.
The kernel's own results are compared with the oracle bit for bit by the GPU
tests; these tests pin the arithmetic those results rest on.
"""
import numpy as np


def e4m3_value(byte: int) -> float:
    """Value of an e4m3 byte: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
    bits; exponent 0 encodes subnormals (m / 8) * 2^-6; S.1111.111 is NaN and
    the format has no infinities."""
    s = -1.0 if byte & 0x80 else 1.0
    e = (byte >> 3) & 0xF
    m = byte & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_exact(v: float):
    """The byte encoding v exactly, or None."""
    for b in range(256):
        x = e4m3_value(b)
        if x == v and (v != 0.0 or b == 0):
            return b
    return None


def test_small_bytes_are_linear_in_units_of_2_pow_minus_9():
    # the weight operand is the masked 2-bit code itself: byte c must be c * 2^-9
    for b in range(16):
        assert e4m3_value(b) == b * 2.0 ** -9
    assert [e4m3_value(c) for c in (0, 1, 2)] == [0.0, 2.0 ** -9, 2.0 ** -8]
    # beyond 16 the encoding is no longer linear (why codes are shifted down
    # to bits 1:0 before use instead of masked in place)
    assert e4m3_value(0x20) != 0x20 * 2.0 ** -9


def test_token_planes_are_exact_e4m3_integers():
    for v in range(-8, 16):
        b = e4m3_exact(float(v))
        assert b is not None and e4m3_value(b) == v
    # 16 * hi is not needed on the operand side (the planes are recombined in
    # integers), but every plane value must be exact
    for q in range(-127, 128):
        lo = q & 15
        hi = (q - lo) // 16
        assert 16 * hi + lo == q
        assert -8 <= hi <= 7 and 0 <= lo <= 15
        assert e4m3_exact(float(hi)) is not None and e4m3_exact(float(lo)) is not None


def test_accumulator_sums_stay_exact_in_fp32():
    K = 65536
    unit = 2.0 ** -9
    # a column's partial sums are multiples of 2^-9 bounded by 2 * 15 * K units
    # (lo plane; hi is bounded by 2 * 8 * K); fp32 holds every such multiple
    # exactly while the count of units stays below 2^24
    for bound_units in (2 * 8 * K, 2 * 15 * K):
        assert bound_units < 2 ** 24
        top = np.float32(bound_units * unit)
        assert float(top) == bound_units * unit
        assert float(np.float32(top - np.float32(unit))) == (bound_units - 1) * unit
    # recombined in integers: sum c q = 16 sum c hi + sum c lo, at most 2 * 127 K
    # in magnitude, below 2^24, and the result after removing the code row sum,
    # at most 127 K, is exact as an fp32 value too (the split-K partial sums are
    # added in fp32 and the last split subtracts the row sum in fp32)
    assert 2 * 127 * K < 2 ** 24
    rng = np.random.default_rng(7)
    for _ in range(200):
        a = int(rng.integers(-2 * 127 * K, 2 * 127 * K + 1))
        r = int(rng.integers(-127 * K, 127 * K + 1))
        if abs(a - r) > 127 * K:
            continue
        diff = np.float32(np.float32(a) - np.float32(r))
        assert float(np.float32(a)) == a and float(np.float32(r)) == r
        assert float(diff) == a - r


def test_unpacked_columns_follow_the_i2s_layout():
    # the thread converting one row's 32-byte block writes TMEM column 8 s + c
    # from packed word c (bytes 4c .. 4c + 3), slot s: element 32 s + 4c + b for
    # byte b of the word; byte j of an I2_S block holds element 32 s + j in bits
    # (7 - 2s):(6 - 2s).  Check the mapping against an explicit I2_S encoding.
    rng = np.random.default_rng(3)
    t = rng.integers(-1, 2, 128)
    codes = (t + 1).astype(np.uint32)
    block = np.zeros(32, np.uint32)
    for e in range(128):
        s, j = divmod(e, 32)
        block[j] |= codes[e] << (6 - 2 * s)
    words = [int(block[4 * c] | (block[4 * c + 1] << 8) | (block[4 * c + 2] << 16) | (block[4 * c + 3] << 24))
             for c in range(8)]
    for s in range(4):
        for c in range(8):
            col = (words[c] >> (6 - 2 * s)) & 0x03030303
            for b in range(4):
                assert (col >> (8 * b)) & 0xFF == codes[32 * s + 4 * c + b]
