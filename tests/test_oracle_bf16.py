"""Pins for the oracle's binary64 -> bfloat16 rounding (round to nearest, ties
to even, IEEE 754 section 4.3.1), which produces the stored expert output the
dprob epilogue reads.

Pinned three ways: hand-built cases whose answer follows from the format
(1+7 significant bits, emin -126, subnormal quantum 2^-133); exhaustive
nearest-neighbour checks with exact rationals; and agreement with torch's
float32 -> bfloat16 conversion on values exactly representable in float32.
"""
from fractions import Fraction
import math

import numpy as np
import pytest

import oracle

U = 2.0 ** -7  # bf16 ulp at 1.0

CASES = [
    (1.0, 0x3F80),
    (1.0 + U, 0x3F81),
    (1.0 + U / 2, 0x3F80),                  # tie, even neighbour below
    (1.0 + 3 * U / 2, 0x3F82),              # tie, even neighbour above
    (1.0 + U / 2 + 2.0 ** -40, 0x3F81),     # just above the tie
    (1.0 + U / 2 - 2.0 ** -40, 0x3F80),     # just below the tie
    (-1.0 - 3 * U / 2, 0xBF82),
    (0.0, 0x0000),
    (-0.0, 0x8000),
    (2.0 ** -133, 0x0001),                  # smallest subnormal
    (2.0 ** -134, 0x0000),                  # tie between 0 and 2^-133 -> even (0)
    (3 * 2.0 ** -134, 0x0002),              # tie between 1 and 2 quanta -> even (2)
    (1.5 * 2.0 ** -134, 0x0001),
    (2.0 ** -126, 0x0080),                  # smallest normal
    (2.0 ** -126 - 2.0 ** -133, 0x007F),    # largest subnormal
    (255.0 * 2.0 ** 120, 0x7F7F),           # largest finite
    (511.0 * 2.0 ** 119 - 2.0 ** 80, 0x7F7F),  # just below the overflow tie
    (511.0 * 2.0 ** 119, 0x7F80),           # overflow tie rounds to even = infinity
    (float("inf"), 0x7F80),
    (float("-inf"), 0xFF80),
    (float("nan"), 0x7FC0),
    (3.0, 0x4040),
    (0.1, 0x3DCD),                          # 0.1 = 1.6 * 2^-4; 1.6*128 = 204.8 -> 205 = 0xCD
]


@pytest.mark.parametrize("x,bits", CASES)
def test_hand_built_cases(x, bits):
    assert int(oracle.bf16_rne(np.array([x]))[0]) == bits


def _bf16_exact(b: int) -> Fraction:
    sign = -1 if b & 0x8000 else 1
    e = (b >> 7) & 0xFF
    m = b & 0x7F
    if e == 0:
        return sign * Fraction(m, 1 << 133)
    return sign * Fraction(128 + m, 128) * Fraction(2) ** (e - 127)


def test_nearest_even_against_exact_neighbours():
    """For random doubles of widely varying magnitude the result is the bf16
    value nearest the exact input, with ties to the even pattern."""
    rng = np.random.default_rng(7)
    xs = rng.standard_normal(3000) * np.exp2(rng.integers(-140, 127, 3000).astype(np.float64))
    # add exact ties between adjacent bf16 values
    for b in rng.integers(1, 0x7F7F, 300):
        mid = (_bf16_exact(int(b)) + _bf16_exact(int(b) + 1)) / 2
        xs = np.append(xs, float(mid))
    out = oracle.bf16_rne(xs)
    for x, b in zip(xs, out):
        b = int(b)
        if not math.isfinite(x) or abs(x) >= 511.0 * 2.0 ** 119:
            continue
        fx = Fraction(x)
        v = _bf16_exact(b)
        mag = b & 0x7FFF
        neighbours = [mag - 1, mag + 1] if mag > 0 else [1]
        for nb in neighbours:
            if nb > 0x7F7F:
                continue
            w = _bf16_exact(nb | (b & 0x8000))
            d_res, d_nb = abs(fx - v), abs(fx - w)
            assert d_res <= d_nb, (x, hex(b), hex(nb))
            if d_res == d_nb:
                assert (mag & 1) == 0, (x, hex(b))


def test_matches_torch_on_float32_representable_values():
    """On values exactly representable in float32, binary64 -> bf16 equals the
    library's float32 -> bf16 conversion (no double rounding can occur)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    f = (rng.standard_normal(20000) * np.exp2(rng.integers(-130, 120, 20000))).astype(np.float32)
    f = f[np.isfinite(f)]
    ours = oracle.bf16_rne(f.astype(np.float64))
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
