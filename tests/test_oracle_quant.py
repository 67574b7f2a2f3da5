"""Pins for the oracle's block-scaled encodings (MXFP8 and NVFP4).

The pages fingerprint the encoded values and scale buffers of MXFP8 and NVFP4
tensors ("NVIDIA fait passer le déterminisme bit à bit de Megatron Core à 2432
GPU ...", section "Méthodologie de débogage du non-déterminisme") and name
E2M1 as the NVFP4 element ("Nemotron 3 Ultra 的 tech report ...", concept
list).  The formats themselves come from their public definitions (FP8 E4M3,
FP4 E2M1, the E8M0 power-of-two scale of the OCP Microscaling v1.0 spec).

Pins:
* code tables against values fixed by the format definitions (largest
  finite, smallest normal and subnormal, one, NaN), all codes round-tripping;
* round to nearest even on hand-built ties and saturation at the largest
  finite value, plus an exhaustive nearest-value search on random inputs;
* MXFP8 on hand-built blocks (power-of-two amax, saturation, all zero, NaN,
  subnormal amax) and the properties amax / X in [256, 512) and the
  dequantisation error bound;
* NVFP4: the block maximum always encodes to +-6, and the dequantisation
  error stays within half an E2M1 step.
"""
import numpy as np
import pytest

import oracle
from bitwise_deterministic_moe_gb300 import synth


def bf16(values):
    return synth.f32_to_bf16_bits(np.asarray(values, dtype=np.float32))


def test_e4m3_table():
    v = oracle.e4m3_value
    assert v(0x7E) == 448.0 and v(0xFE) == -448.0
    assert v(0x08) == 2.0 ** -6 and v(0x07) == 7 / 8 * 2.0 ** -6 and v(0x01) == 2.0 ** -9
    assert v(0x38) == 1.0 and v(0x00) == 0.0 and np.signbit(v(0x80))
    assert np.isnan(v(0x7F)) and np.isnan(v(0xFF))
    pos = v(np.arange(0x7F))
    assert np.all(np.diff(pos) > 0)                       # ascending with the code
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F])
    assert np.array_equal(oracle.e4m3_encode(v(codes)), codes.astype(np.uint8))


def test_e4m3_ties_and_saturation():
    enc = oracle.e4m3_encode
    assert enc(1.0625) == 0x38          # halfway 1 / 1.125 -> even code
    assert enc(1.1875) == 0x3A          # halfway 1.125 / 1.25 -> even code
    assert enc(464.0) == 0x7E and enc(1e6) == 0x7E and enc(-1e6) == 0xFE
    assert enc(2.0 ** -10) == 0x00 and enc(2.0 ** -10 * 1.01) == 0x01
    assert enc(3 * 2.0 ** -10) == 0x02  # halfway subnormals 1 and 2 (x 2^-9) -> even


def _nearest_bruteforce(a, values, codes):
    best = None
    for v, c in zip(values, codes):
        d = abs(a - v)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return best[1]


def test_e4m3_and_e2m1_match_exhaustive_search():
    rng = np.random.default_rng(2)
    xs = np.concatenate([rng.uniform(0, 450, 300), np.exp2(rng.uniform(-12, 9, 300))])
    pv = oracle.e4m3_value(np.arange(0x7F))
    for a in xs:
        assert oracle.e4m3_encode(a) == _nearest_bruteforce(a, pv, range(0x7F))
    fv = oracle.e2m1_value(np.arange(8))
    for a in rng.uniform(0, 6, 300):
        assert oracle.e2m1_encode(a) == _nearest_bruteforce(a, fv, range(8))


def test_e2m1_table_and_ties():
    assert list(oracle.e2m1_value(np.arange(8))) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    enc = oracle.e2m1_encode
    assert [int(enc(x)) for x in (0.25, 0.75, 2.5, 5.0, 7.0, 100.0)] == [0, 2, 4, 6, 7, 7]
    assert int(enc(-1.25)) == 0x8 | 2 and int(enc(-0.0)) == 0x8


def test_mxfp8_hand_blocks():
    row = np.zeros(5 * 32, dtype=np.float32)
    row[0:32] = 0.5
    row[0] = 1.0                               # amax 1 -> s = -8, 1 * 2^8 = 256 = 0x78
    row[32:64] = 1.96875                       # s = -8, 504 saturates to 448
    # row[64:96] all zero
    row[96] = np.nan                           # NaN block
    row[128:160] = np.float32(2.0 ** -130)     # subnormal amax: s clamps at -127
    vals, scales = oracle.mxfp8_quantize(bf16(row)[None, :])
    assert list(scales[0]) == [119, 119, 0, 0xFF, 0]
    assert vals[0, 0] == 0x78 and vals[0, 1] == oracle.e4m3_encode(128.0)
    assert np.all(vals[0, 32:64] == 0x7E)
    assert np.all(vals[0, 64:96] == 0) and np.all(vals[0, 96:128] == 0x7F)
    assert np.all(vals[0, 128:160] == oracle.e4m3_encode(2.0 ** -130 * 2.0 ** 127))


def test_mxfp8_scale_and_error_properties():
    x = synth._normal_bf16(5, 1, (64, 512), 1.0)
    x[3, :32] = synth.f32_to_bf16_bits(np.full(32, 3e-39, np.float32))     # tiny block
    vals, scales = oracle.mxfp8_quantize(x)
    v = oracle.bf16_to_f64(x).reshape(64, 16, 32)
    X = np.exp2(scales.astype(np.float64) - 127)[..., None]
    amax = np.abs(v).max(axis=2, keepdims=True)
    r = amax / X
    normal = scales[..., None] > 0
    assert np.all(((r >= 256) & (r < 512)) | ~normal)
    deq = oracle.e4m3_value(vals).reshape(64, 16, 32) * X
    sat = np.abs(v) / X > 448
    err = np.abs(deq - v)
    ok = (err <= np.maximum(np.abs(v) * 2.0 ** -4, 2.0 ** -10 * X)) | sat
    assert ok.all()
    assert np.all(np.abs(deq[sat]) == 448 * np.broadcast_to(X, sat.shape)[sat])


def test_nvfp4_block_max_and_error():
    x = synth._normal_bf16(6, 1, (32, 256), 0.3)
    packed, scales, s_enc = oracle.nvfp4_quantize(x)
    v = oracle.bf16_to_f64(x).astype(np.float32).astype(np.float64)
    amax_t = np.abs(v).max()
    assert s_enc == np.float32(np.float32(2688.0) / np.float32(amax_t))
    q = np.empty((32, 256), dtype=np.uint8)
    q[:, 0::2] = packed & 0xF
    q[:, 1::2] = packed >> 4
    qv = oracle.e2m1_value(q).reshape(32, 16, 16)
    vb = v.reshape(32, 16, 16)
    imax = np.abs(vb).argmax(axis=2)
    assert np.all(np.abs(np.take_along_axis(qv, imax[..., None], 2)) == 6.0)
    unit = (oracle.e4m3_value(scales) / float(s_enc))[..., None]
    err = np.abs(qv * unit - vb)
    assert np.all(err <= 1.0 * unit * (1 + 1e-6))
    # the zero tensor: S_enc = 1, every scale and element zero
    p0, s0, e0 = oracle.nvfp4_quantize(np.zeros((2, 32), np.uint16))
    assert e0 == 1.0 and not p0.any() and not s0.any()
