"""Pins of the oracle's block-scaled decoders and of its grouped GEMM on
decoded operands, against things other than the oracle itself:

* a second decoder written with Python integers and Fractions straight from
  the bit-field definitions (sign, exponent, fraction; E8M0 = 2^(e - 127);
  NVFP4 value = code * scale / S_enc, element 2i in the low nibble);
* exact round trips: values built to be exactly representable in MXFP8 come
  back bit for bit through quantize -> decode;
* exact rational arithmetic for the GEMM on tiny inputs whose partial sums are
  all exact in binary64, through a direct per-(row, column) loop that does not
  use the matrix product or the expert search of the oracle;
* planted mistakes (a scale taken from the neighbouring block, swapped
  nibbles, a transposed weight) that the pins must catch.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle


def e4m3_frac(c):
    """E4M3: 1 sign, 4 exponent bits (bias 7), 3 fraction bits; e = 0 subnormal."""
    c = int(c)
    sign = -1 if c & 0x80 else 1
    e, m = (c >> 3) & 0xF, c & 7
    if e == 0xF and m == 7:
        return None                                     # NaN
    if e == 0:
        return sign * Fraction(m, 8) * Fraction(1, 2 ** 6)
    return sign * (1 + Fraction(m, 8)) * (Fraction(2) ** (e - 7))


def e2m1_frac(c):
    """E2M1: 1 sign, 2 exponent bits (bias 1), 1 fraction bit; e = 0 subnormal."""
    c = int(c) & 0xF
    sign = -1 if c & 0x8 else 1
    e, m = (c >> 1) & 3, c & 1
    if e == 0:
        return sign * Fraction(m, 2)
    return sign * (1 + Fraction(m, 2)) * (Fraction(2) ** (e - 1))


def mxfp8_frac(codes, scales):
    rows, cols = codes.shape
    out = [[None] * cols for _ in range(rows)]
    for r in range(rows):
        for c in range(cols):
            s = int(scales[r, c // 32])
            v = e4m3_frac(codes[r, c])
            out[r][c] = None if (v is None or s == 0xFF) else v * Fraction(2) ** (s - 127)
    return out


def nvfp4_frac(packed, scales, s_enc):
    rows, half = packed.shape
    out = [[None] * (2 * half) for _ in range(rows)]
    S = Fraction(float(np.float32(s_enc)))
    for r in range(rows):
        for i in range(half):
            byte = int(packed[r, i])
            for k, code in ((2 * i, byte & 0xF), (2 * i + 1, byte >> 4)):
                out[r][k] = e2m1_frac(code) * e4m3_frac(scales[r, k // 16]) / S
    return out


def test_mxfp8_decode_matches_bit_field_definition():
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 256, (3, 64), dtype=np.uint8)
    codes[codes == 0x7F] = 0x7E
    codes[codes == 0xFF] = 0xFE
    scales = rng.integers(100, 160, (3, 2), dtype=np.uint8)
    scales[1, 0] = 0                                   # 2^-127
    scales[2, 1] = 0xFF                                # NaN block
    got = oracle.mxfp8_decode(codes, scales)
    want = mxfp8_frac(codes, scales)
    for r in range(3):
        for c in range(64):
            if want[r][c] is None:
                assert np.isnan(got[r, c])
            else:
                assert Fraction(float(got[r, c])) == want[r][c], (r, c)


def test_nvfp4_decode_matches_bit_field_definition():
    rng = np.random.default_rng(2)
    packed = rng.integers(0, 256, (2, 32), dtype=np.uint8)
    scales = rng.integers(0, 0x7F, (2, 4), dtype=np.uint8)          # non-negative E4M3 codes, no NaN
    s_enc = np.float32(2688.0) / np.float32(3.7)
    got = oracle.nvfp4_decode(packed, scales, s_enc)
    want = nvfp4_frac(packed, scales, s_enc)
    for r in range(2):
        for c in range(64):
            # one division by S_enc in binary64: within half an ulp of the exact value
            w = want[r][c]
            assert abs(Fraction(float(got[r, c])) - w) <= abs(w) * Fraction(1, 2 ** 53), (r, c)


def test_mxfp8_round_trip_is_exact_for_representable_values():
    """Blocks of E4M3 values times 2^s whose largest magnitude lies in
    [256, 448] (so the encoder picks exactly scale s) decode bit for bit."""
    rng = np.random.default_rng(3)
    finite = np.array([c for c in range(0x7F) if c != 0x7F], dtype=np.uint8)
    rows, cols = 4, 96
    codes = rng.choice(finite, (rows, cols)).astype(np.uint8)
    codes[:, ::32] = rng.integers(0x78, 0x7F, (rows, cols // 32))   # exponent field 15: [256, 448]
    sign = rng.integers(0, 2, (rows, cols)).astype(np.uint8) << 7
    codes = codes | sign
    s = rng.integers(-20, 20, (rows, cols // 32))
    x = oracle.e4m3_value(codes) * np.exp2(np.repeat(s, 32, axis=1).astype(np.float64))
    x_bits = oracle.bf16_rne(x)
    assert np.array_equal(oracle.bf16_to_f64(x_bits), x)               # bf16 holds them exactly
    vals, scales = oracle.mxfp8_quantize(x_bits)
    assert np.array_equal(scales.astype(np.int64), s + 127)
    assert np.array_equal(oracle.mxfp8_decode(vals, scales), x)


def _tiny_problem(kind, seed):
    """Operands whose decoded products and partial sums are exact in binary64."""
    rng = np.random.default_rng(seed)
    E, N, K = 3, 16, 64
    counts = np.array([5, 0, 7])
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(off[-1])
    if kind == "mxfp8":
        # normal E4M3 codes of exponent field 6..9 (values in [0.5, 7.5]), scales 2^-1..2^1
        e = rng.integers(6, 10, (R, K))
        m = rng.integers(0, 8, (R, K))
        xq = ((rng.integers(0, 2, (R, K)) << 7) | (e << 3) | m).astype(np.uint8)
        e = rng.integers(6, 10, (E * N, K))
        m = rng.integers(0, 8, (E * N, K))
        wq = ((rng.integers(0, 2, (E * N, K)) << 7) | (e << 3) | m).astype(np.uint8)
        xs = rng.integers(126, 129, (R, K // 32)).astype(np.uint8)
        ws = rng.integers(126, 129, (E * N, K // 32)).astype(np.uint8)
        Xd = oracle.mxfp8_decode(xq, xs)
        Wd = oracle.mxfp8_decode(wq, ws)
        Xf, Wf = mxfp8_frac(xq, xs), mxfp8_frac(wq, ws)
    else:
        xq = rng.integers(0, 256, (R, K // 2), dtype=np.uint8)
        wq = rng.integers(0, 256, (E * N, K // 2), dtype=np.uint8)
        xs = rng.integers(0x30, 0x41, (R, K // 16)).astype(np.uint8)     # E4M3 0.5 .. 2.25
        ws = rng.integers(0x30, 0x41, (E * N, K // 16)).astype(np.uint8)
        sx, sw = np.float32(0.5), np.float32(4.0)                      # powers of two: exact division
        Xd = oracle.nvfp4_decode(xq, xs, sx)
        Wd = oracle.nvfp4_decode(wq, ws, sw)
        Xf, Wf = nvfp4_frac(xq, xs, sx), nvfp4_frac(wq, ws, sw)
    return E, N, K, off, Xd, Wd.reshape(E, N, K), Xf, Wf


@pytest.mark.parametrize("kind", ["mxfp8", "nvfp4"])
def test_block_scaled_rows_exact_against_rationals(kind):
    E, N, K, off, Xd, Wd, Xf, Wf = _tiny_problem(kind, 11 if kind == "mxfp8" else 12)
    R = int(off[-1])
    rows = np.arange(R)
    Y, Yb, _, _ = oracle.block_scaled_rows(Xd, lambda e: Wd[e], off, rows)
    for r in range(R):
        e = next(x for x in range(E) if off[x] <= r < off[x + 1])      # direct expert lookup
        for n in range(N):
            exact = sum(Xf[r][c] * Wf[e * N + n][c] for c in range(K))
            assert Fraction(float(Y[r, n])) == exact, (r, n)
    assert np.array_equal(Yb, oracle.bf16_rne(Y))


def test_block_scaled_rows_dprob_matches_bf16_path_on_the_same_output():
    """The slots and dots of block-scaled rows are those of the stored bf16
    output, exactly as for bf16 operands (expert_rows with the output's bits as
    X and an identity W reproduces the same Yb, hence the same P and D)."""
    E, N, K, off, Xd, Wd, _, _ = _tiny_problem("mxfp8", 13)
    N = 256
    rng = np.random.default_rng(5)
    Wd = rng.standard_normal((E, N, K))
    R = int(off[-1])
    topk = 2
    T = (R + 1) // 2
    row_src = rng.permutation(T * topk)[:R].astype(np.int32)
    G = oracle.bf16_rne(rng.standard_normal((T, N)))
    Y, Yb, P, D = oracle.block_scaled_rows(Xd, lambda e: Wd[e], off, np.arange(R), G=G, row_src=row_src, topk=topk)
    P2, D2 = oracle.dprob_from_output(G, Yb, row_src, topk)
    assert np.array_equal(P, P2) and np.array_equal(D, D2)
    # slot sums in any order equal the dot within the binary64 bound
    assert np.all(np.abs(P.sum(axis=1) - D) <= 4 * 2.0 ** -52 * np.abs(P).sum(axis=1) + 1e-300)


def test_planted_mistakes_are_caught():
    E, N, K, off, Xd, Wd, Xf, Wf = _tiny_problem("mxfp8", 14)
    R = int(off[-1])
    rows = np.arange(R)
    Y, _, _, _ = oracle.block_scaled_rows(Xd, lambda e: Wd[e], off, rows)
    # a transposed weight slice
    Yt, _, _, _ = oracle.block_scaled_rows(Xd, lambda e: Wd[e][::-1], off, rows)
    assert not np.array_equal(Y, Yt)
    # the scale of the neighbouring block
    rng = np.random.default_rng(7)
    codes = rng.integers(0x38, 0x70, (2, 64), dtype=np.uint8)
    scales = np.array([[120, 130], [125, 128]], dtype=np.uint8)
    good = oracle.mxfp8_decode(codes, scales)
    bad = oracle.mxfp8_decode(codes, scales[:, ::-1])
    assert not np.array_equal(good, bad)
    # swapped nibbles change an NVFP4 decode of unequal codes
    packed = np.array([[0x21, 0x43]], dtype=np.uint8)
    sc = np.array([[0x38]], dtype=np.uint8)
    a = oracle.nvfp4_decode(np.pad(packed, ((0, 0), (0, 6))), sc, np.float32(1))
    b = oracle.nvfp4_decode(np.pad(((packed & 0xF) << 4) | (packed >> 4), ((0, 0), (0, 6))), sc, np.float32(1))
    assert not np.array_equal(a, b)
    assert a[0, 0] == 0.5 and a[0, 1] == 1.0          # element 0 in the low nibble
