"""Failure detection on the GPU without faulting it: a pipeline wait that is
made to run out (a stage armed but never loaded -- nothing is in flight)
must end the kernel with DMOE_ERR_TIMEOUT in the status word, free its tensor
memory, and leave the context usable: the next call gives the reference bits.
Also: corrupt routing data is reported, never used as an address."""
import numpy as np
import pytest
import torch

from bitwise_deterministic_moe_gb300 import api, synth
from tests import gpu_util
from tests.gpu_util import Problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gpu_util.ensure_built()


def bits(t):
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32).clone()


@pytest.mark.parametrize("kernel", [api.LAUNCH_SINGLE_CTA, api.LAUNCH_CTA_PAIRS], ids=["single", "pairs"])
def test_wait_limit_reports_timeout_and_context_survives(kernel):
    prob = Problem(synth.CONFIGS["small"])
    out, dprob, _ = prob.run_dprob(flags=kernel)
    ref_out, ref_dp = bits(out), bits(dprob)
    assert api.read_status(prob.ws) == 0
    api.grouped_gemm_dprob(prob.X, prob.W, prob.off, prob.G, prob.src, prob.cfg.topk, prob.ws,
                           flags=api.LAUNCH_TEST_STALL | kernel)
    assert api.read_status(prob.ws) == 4          # DMOE_ERR_TIMEOUT
    for _ in range(2):                             # the context and the workspace still work
        out2, dprob2, _ = prob.run_dprob(flags=kernel)
        assert api.read_status(prob.ws) == 0
        assert torch.equal(bits(out2), ref_out)
        assert torch.equal(bits(dprob2), ref_dp)


def test_corrupt_row_src_is_reported_not_followed():
    prob = Problem(synth.CONFIGS["tiny"])
    src = prob.src.clone()
    src[5] = 1 << 30
    src[17] = -7
    api.grouped_gemm_dprob(prob.X, prob.W, prob.off, prob.G, src, prob.cfg.topk, prob.ws)
    assert api.read_status(prob.ws) == 3          # DMOE_ERR_ROUTING
    slots = torch.empty(prob.cfg.S, prob.cfg.R, dtype=torch.float32, device="cuda")
    out, _, _ = prob.run_dprob()
    api.dprob_epilogue(prob.G, out, prob.off, src, prob.cfg.topk, slots=slots)
    dp = torch.zeros(prob.cfg.T, prob.cfg.topk, dtype=torch.float32, device="cuda")
    api.dprob_combine(slots, src, prob.cfg.topk, dprob=dp)
    torch.cuda.synchronize()
    assert api.read_status(prob.ws) == 0


def test_serialized_writers_timeout_then_recover():
    """A stalled stage in the serialized control: the stalled CTA and every
    writer waiting for its turn give up within their limits, the status says
    DMOE_ERR_TIMEOUT, and the next call gives the deterministic bits."""
    prob = Problem(synth.CONFIGS["small"])
    _, ref_dp, _ = prob.run_dprob()
    ref_dp = bits(ref_dp)
    assert api.read_status(prob.ws) == 0
    api.grouped_gemm_dprob_serial(prob.X, prob.W, prob.off, prob.G, prob.src, prob.cfg.topk, prob.ws,
                                  flags=api.LAUNCH_TEST_STALL)
    assert api.read_status(prob.ws) == 4
    _, dp = api.grouped_gemm_dprob_serial(prob.X, prob.W, prob.off, prob.G, prob.src, prob.cfg.topk, prob.ws)
    assert api.read_status(prob.ws) == 0
    assert torch.equal(bits(dp), ref_dp)
