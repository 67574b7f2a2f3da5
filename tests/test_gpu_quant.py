"""MXFP8 / NVFP4 encodings on the GPU vs the oracle, byte for byte.

Quantised codes are integer outputs decided by floating point, so both sides
take each decision in the same precision (the scale from the exact exponent
of amax for MXFP8; binary32 steps in a fixed order for NVFP4) and every byte
must match.  The fingerprints of the encoded values and scale buffers -- what
the pages record for MXFP8 and NVFP4 tensors -- must match the oracle's too.
Inputs cover wide dynamic range, all-zero, NaN, infinity and subnormal
blocks, saturation, and the full LatentMoE-shaped X and W (sampled rows).
"""
import numpy as np
import pytest
import torch

import oracle
from bitwise_deterministic_moe_gb300 import api, synth
from tests import gpu_util
from tests.gpu_util import bf16_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gpu_util.ensure_built()


def wide_range(rows, cols, seed):
    """Normal values whose 16-value blocks are scaled by 2^U(-140, 120)."""
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((rows, cols)).astype(np.float32)
    e = rng.integers(-140, 120, (rows, cols // 16)).astype(np.float32)
    v = v * np.repeat(np.exp2(e), 16, axis=1)
    return synth.f32_to_bf16_bits(v)


def special_rows(cols):
    r = np.zeros((6, cols), dtype=np.float32)
    r[0] = 1.96875                       # saturates after scaling
    r[1, :] = 0.0                        # all zero
    r[2, 5] = np.nan
    r[3, 7] = np.inf
    r[3, 40] = -np.inf
    r[4] = np.float32(2.0 ** -133) * np.arange(cols)     # bf16 subnormals
    r[5] = -np.float32(1e-40)
    bits = synth.f32_to_bf16_bits(r)
    bits[2, 5] = 0x7FC0                  # a quiet NaN pattern
    return bits


def host(t):
    return t.cpu().numpy()


@pytest.mark.parametrize("shape,seed", [((64, 512), 1), ((33, 96), 2), ((1, 32), 3), ((300, 2048), 4)])
def test_mxfp8_bytes_and_fingerprints(shape, seed):
    x = wide_range(*shape, seed)
    if shape[1] >= 64:
        sp = special_rows(shape[1])
        x = np.concatenate([x, sp], axis=0)
    vals, scales = api.quantize_mxfp8(bf16_dev(x))
    rv, rs = oracle.mxfp8_quantize(x)
    assert np.array_equal(host(vals), rv)
    assert np.array_equal(host(scales), rs)
    for dev_t, ref in ((vals, rv), (scales, rs)):
        ch, h = api.fingerprint_host(dev_t)
        rch, rh = oracle.fingerprint(ref, oracle.DTYPE_CODES["uint8"])
        assert ch == [int(c) for c in rch] and h == rh


@pytest.mark.parametrize("shape,seed,scale", [((64, 512), 5, 1.0), ((33, 96), 6, 1e-3), ((300, 2048), 7, 30.0)])
def test_nvfp4_bytes_and_fingerprints(shape, seed, scale):
    x = synth._normal_bf16(seed, 1, shape, scale)
    x[0, 0] = synth.f32_to_bf16_bits(np.float32([scale * 1e4]))[0]     # one outlier: tiny block scales
    ws = api.workspace(1, 1, 1)
    packed, scales, s_enc = api.quantize_nvfp4(bf16_dev(x), ws)
    rp, rs, re = oracle.nvfp4_quantize(x)
    assert np.array_equal(host(packed), rp)
    assert np.array_equal(host(scales), rs)
    assert host(s_enc).view(np.uint32)[0] == np.float32(re).view(np.uint32)
    ch, h = api.fingerprint_host(packed)
    rch, rh = oracle.fingerprint(rp, oracle.DTYPE_CODES["uint8"])
    assert ch == [int(c) for c in rch] and h == rh


@pytest.mark.parametrize("shape", [(1, 16), (3, 48), (7, 80)])
def test_nvfp4_signed_zeros_and_odd_block_counts(shape):
    """Odd numbers of 16-value blocks (the encoder handles two per thread),
    negative zeros, and negative values far below their block's maximum, whose
    quotients round to -0: the encoder must keep the sign as IEEE division
    does."""
    rng = np.random.default_rng(sum(shape))
    v = rng.standard_normal(shape).astype(np.float32)
    v[:, 1::5] = -0.0
    v[:, 2::7] = -1e-6 * np.abs(v[:, 2::7])
    v[:, 3::11] = 1e-6 * np.abs(v[:, 3::11])
    x = synth.f32_to_bf16_bits(v)
    ws = api.workspace(1, 1, 1)
    packed, scales, s_enc = api.quantize_nvfp4(bf16_dev(x), ws)
    rp, rs, re = oracle.nvfp4_quantize(x)
    assert np.array_equal(host(scales), rs)
    assert np.array_equal(host(packed), rp)
    assert host(s_enc).view(np.uint32)[0] == np.float32(re).view(np.uint32)
    assert ((rp & 0xF) == 0x8).any() or ((rp >> 4) == 0x8).any()   # the case is exercised


def test_nvfp4_zero_tensor_and_repeat():
    ws = api.workspace(1, 1, 1)
    z = torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda")
    p, s, e = api.quantize_nvfp4(z, ws)
    assert float(e) == 1.0 and not p.any() and not s.any()
    x = bf16_dev(synth._normal_bf16(9, 1, (128, 1024), 1.0))
    ref = [t.clone() for t in api.quantize_nvfp4(x, ws)]
    for _ in range(3):
        got = api.quantize_nvfp4(x, ws)
        assert all(torch.equal(a, b) for a, b in zip(got, ref))


@pytest.mark.parametrize("which", ["X", "W"])
def test_latent_operands_sampled_rows(which):
    """The LatentMoE-shaped operands: X_perm [R, K] and W viewed as [E*N, K]."""
    cfg = synth.CONFIGS["latent"]
    inp = synth.make_inputs(cfg, with_weights=(which == "W"))
    a = inp.X if which == "X" else inp.W.reshape(-1, cfg.K)
    d = bf16_dev(a)
    vals, scales = api.quantize_mxfp8(d)
    ws = api.workspace(1, 1, 1)
    packed, nscales, s_enc = api.quantize_nvfp4(d, ws)
    rows = np.random.default_rng(8).choice(a.shape[0], 256, replace=False)
    rv, rs = oracle.mxfp8_quantize(a[rows])
    idx = torch.from_numpy(rows).cuda()
    assert np.array_equal(host(vals.index_select(0, idx)), rv)
    assert np.array_equal(host(scales.index_select(0, idx)), rs)
    amax = np.abs(oracle.bf16_to_f64(a)).max()
    rp, rns, re = oracle.nvfp4_quantize(a[rows], amax=amax)
    assert host(s_enc).view(np.uint32)[0] == np.float32(re).view(np.uint32)
    assert np.array_equal(host(packed.index_select(0, idx)), rp)
    assert np.array_equal(host(nscales.index_select(0, idx)), rns)


def test_nvfp4_rounding_ties_and_boundaries():
    """Blocks whose scaled values land exactly on E2M1 rounding boundaries
    (0.25, 0.75, 1.25, ... : ties to even) and just beside them: the encoder's
    quotient shortcut must hand these to the exact division and match the
    oracle byte for byte."""
    rows, cols = 64, 512
    rng = np.random.default_rng(21)
    v = np.zeros((rows, cols), dtype=np.float32)
    for r in range(rows):
        for b in range(cols // 16):
            j = int(rng.integers(-20, 20))
            k = rng.integers(0, 25, 16).astype(np.float32)      # multiples of 1/4 up to 6
            k[0] = 24.0                                         # block max = 6 * 2^j
            sign = np.where(rng.random(16) < 0.5, -1.0, 1.0).astype(np.float32)
            nudge = np.float32(1.0) + rng.choice([0.0, 2.0 ** -7, -(2.0 ** -8)], 16).astype(np.float32)
            nudge[0] = 1.0
            v[r, b * 16:(b + 1) * 16] = sign * (k / 4) * np.float32(2.0 ** j) * nudge
    x = synth.f32_to_bf16_bits(v)
    ws = api.workspace(1, 1, 1)
    packed, scales, s_enc = api.quantize_nvfp4(bf16_dev(x), ws)
    rp, rs, re = oracle.nvfp4_quantize(x)
    assert np.array_equal(host(scales), rs)
    assert np.array_equal(host(packed), rp)


def test_block_scale_division_is_correctly_rounded_exhaustively(tmp_path):
    """The NVFP4 encoder divides by the block scale with one reciprocal per
    block and a two-fma correction per element.  For every positive finite
    E4M3 scale and every binary32 significand of dividends of both signs whose
    quotient lies in [2^-3, 2^3) -- where every E2M1 decision is taken -- the
    result must equal the compiler's correctly rounded division bit for bit
    (the check kernel lives in tests/cuda and is built here)."""
    import ctypes
    import os
    import subprocess
    from bitwise_deterministic_moe_gb300 import build as B

    here = os.path.dirname(os.path.abspath(__file__))
    lib = str(tmp_path / "libblock_scale_check.so")
    cmd = [B.nvcc()] + B._flags(["-I", B.CSRC]) + ["-shared", "-o", lib,
                                                     os.path.join(here, "cuda", "block_scale_check.cu")]
    subprocess.run(cmd, check=True, capture_output=True)
    so = ctypes.CDLL(lib)
    mism, first = ctypes.c_ulonglong(), ctypes.c_ulonglong()
    assert so.block_scale_check(ctypes.byref(mism), ctypes.byref(first)) == 0
    assert mism.value == 0, hex(first.value)
