"""Fingerprints taken by the combine (moe_grouped_gemm_dprob_fp) vs the oracle's
chunk fingerprint of the same bytes and vs the standalone GPU fingerprint:
bit-exact (integer work), with the outputs equal to the plain call's."""
import numpy as np
import pytest
import torch

import oracle
from bitwise_deterministic_moe_gb300 import api, synth
from tests import gpu_util
from tests.gpu_util import Problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gpu_util.ensure_built()


def _u64(t):
    return [int(v) & ((1 << 64) - 1) for v in t.cpu().tolist()]


def _check(prob, chunk_bytes):
    out, dprob, slots = prob.run_dprob()
    out2, dprob2, slots2, hs, hd = api.grouped_gemm_dprob_fp(prob.X, prob.W, prob.off, prob.G, prob.src,
                                                             prob.cfg.topk, prob.ws, chunk_bytes=chunk_bytes)
    assert api.read_status(prob.ws) == 0
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(slots.view(torch.int32), slots2.view(torch.int32))
    assert torch.equal(dprob.view(torch.int32), dprob2.view(torch.int32))
    # the oracle's positional chunk hashes of the raw bytes the call left behind
    src_bytes = prob.src.cpu().numpy().view(np.uint8)
    dp_bytes = dprob2.cpu().numpy().reshape(-1).view(np.uint8)
    assert _u64(hs) == [int(v) for v in oracle.fingerprint_chunks(src_bytes, chunk_bytes)]
    assert _u64(hd) == [int(v) for v in oracle.fingerprint_chunks(dp_bytes, chunk_bytes)]
    # and the standalone GPU fingerprint of the same buffers
    assert _u64(hs) == api.fingerprint_host(prob.src, chunk_bytes)[0]
    assert _u64(hd) == api.fingerprint_host(dprob2, chunk_bytes)[0]
    # a second call gives the same hashes: the accumulators were left at zero
    _, _, _, hs2, hd2 = api.grouped_gemm_dprob_fp(prob.X, prob.W, prob.off, prob.G, prob.src, prob.cfg.topk,
                                                  prob.ws, chunk_bytes=chunk_bytes)
    assert _u64(hs2) == _u64(hs) and _u64(hd2) == _u64(hd)
    status_region = prob.ws[:256].cpu().numpy()
    assert not status_region[132:256].any()


SMALL = synth.CONFIGS["small"]   # R = 24,576 rows: 98,304 bytes per buffer


@pytest.mark.parametrize("chunk_bytes", [1 << 20,      # one partial chunk
                                         65536,        # two chunks, the last partial
                                         16384,        # six whole chunks: the most the combine takes
                                         14336,        # seven chunks: a separate fingerprint pass
                                         512])         # 192 chunks: a separate pass
def test_fused_fingerprints_small(chunk_bytes):
    _check(Problem(SMALL), chunk_bytes)


def test_fused_fingerprints_general_combine():
    """R % 4 != 0: the combine's general form, then a separate fingerprint pass."""
    cfg = synth.custom_config("odd", T=301, E=7, topk=3, K=128, N=256, index=321)
    _check(Problem(cfg), 1024)


@pytest.mark.parametrize("name", ["latent", "imbal"])
def test_fused_fingerprints_full_size(name):
    """The benchmark's call: one chunk (LatentMoE) or two (imbalanced) of 1 MiB."""
    _check(Problem(synth.CONFIGS[name]), 1 << 20)


def test_fused_fingerprints_reject_bad_chunk():
    prob = Problem(synth.CONFIGS["tiny"])
    with pytest.raises(api.DmoeError):
        api.grouped_gemm_dprob_fp(prob.X, prob.W, prob.off, prob.G, prob.src, prob.cfg.topk, prob.ws,
                                  chunk_bytes=1000)
