"""moe_grouped_gemm_dprob_noalloc: the variant for callers that cannot
allocate device memory (code hosted by a runtime that only hands over its
input and output buffers, or a loop that must not call cudaMalloc).  It keeps
the slot scratch and the GEMM's tile counters in fixed library-owned device
arrays instead of taking a caller workspace.

Called through the C ABI (ctypes, no binding code) several times in a row on
two different problems -- with the call's own kernel choice, with the CTA-pair
kernel forced, and with two persistent grid sizes one after the other -- and
compared with the existing entry point moe_grouped_gemm_dprob: within the
parity tolerances (bf16 output rel 1e-2 of each row's max-abs, fp32 dprob rel
2e-3 of the max-abs), and in fact bit for bit, since both run the same
kernels.  Calls that follow one another on one stream sharing the fixed tile
counters must each see them at zero, or tiles would be skipped and the bits
would differ.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from bitwise_deterministic_moe_gb300 import api, synth
from tests import gpu_util
from tests.gpu_util import Problem

pytestmark = pytest.mark.gpu

MAX_SLOT_VALUES = 4194304   # DMOE_NOALLOC_MAX_SLOT_VALUES in include/dmoe.h


class Launch(ctypes.Structure):
    """dmoe_launch of include/dmoe.h."""
    _fields_ = [("num_ctas", ctypes.c_int), ("flags", ctypes.c_int)]


def noalloc_fn():
    gpu_util.ensure_built()
    lib = ctypes.CDLL(api.library_path())
    P, I = ctypes.c_void_p, ctypes.c_int
    f = lib.moe_grouped_gemm_dprob_noalloc
    f.argtypes = [P, P, P, I, I, I, I, P, P, P, I, I, P, ctypes.POINTER(Launch), P]
    f.restype = I
    return f


def call_noalloc(f, prob, out, dprob, num_ctas=0, flags=0):
    cfg = prob.cfg
    st = f(prob.X.data_ptr(), prob.W.data_ptr(), prob.off.data_ptr(), cfg.R, cfg.E, cfg.K, cfg.N,
           out.data_ptr(), prob.G.data_ptr(), prob.src.data_ptr(), cfg.T, cfg.topk, dprob.data_ptr(),
           ctypes.byref(Launch(num_ctas, flags)), torch.cuda.current_stream().cuda_stream)
    return st


def compare(out_a, dprob_a, out_b, dprob_b):
    ya = out_a.double().cpu().numpy()
    yb = out_b.double().cpu().numpy()
    rowmax = np.maximum(np.abs(yb).max(axis=1, keepdims=True), 1e-30)
    assert (np.abs(ya - yb) / rowmax).max() <= gpu_util.GEMM_RTOL
    da = dprob_a.double().cpu().numpy()
    db = dprob_b.double().cpu().numpy()
    assert np.abs(da - db).max() <= gpu_util.DPROB_RTOL * max(np.abs(db).max(), 1e-30)
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(dprob_a.view(torch.int32), dprob_b.view(torch.int32))


# (num_ctas, flags) of the calls made one after the other on each problem
CALLS = [(0, 0), (0, api.LAUNCH_CTA_PAIRS), (37, 0), (6, api.LAUNCH_CTA_PAIRS), (0, 0)]


def test_noalloc_matches_existing_entry_point_two_calls():
    f = noalloc_fn()
    problems = [Problem(synth.custom_config("noalloc_a", T=1500, E=24, topk=4, K=192, N=384, index=501)),
                Problem(synth.CONFIGS["small"])]          # S*R = 16 * 24576 fits the array
    for prob in problems:                                  # calls in a row, two problem sizes
        cfg = prob.cfg
        ref_out, ref_dprob, _ = prob.run_dprob()
        assert api.read_status(prob.ws) == 0               # the existing entry point's own check
        ref_out, ref_dprob = ref_out.clone(), ref_dprob.clone()
        for num_ctas, flags in CALLS:
            out = torch.full((cfg.R, cfg.N), float("nan"), dtype=torch.bfloat16, device="cuda")
            dprob = torch.full((cfg.T, cfg.topk), float("nan"), dtype=torch.float32, device="cuda")
            assert call_noalloc(f, prob, out, dprob, num_ctas=num_ctas, flags=flags) == 0
            torch.cuda.synchronize()
            compare(out, dprob, ref_out, ref_dprob)


def test_noalloc_rejects_sizes_beyond_its_array():
    f = noalloc_fn()
    T, k, N = 8192, 64, 2048              # S * R = 16 * 524288 > 4 Mi values
    assert (N // 128) * T * k > MAX_SLOT_VALUES
    # rejected during host-side validation, before any device work
    st = f(16, 16, 16, T * k, 8, 64, N, 16, 16, 16, T, k, 16, None, None)
    assert st == 2                         # DMOE_ERR_UNSUPPORTED
