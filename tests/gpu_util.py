"""Helpers shared by the GPU tests: move seeded inputs to the device and
compare with the oracle using the tolerances fixed for this path
(bf16 GEMM output within rel 1e-2 of each row's max-abs; fp32 dprob and slot
partials within rel 2e-3 of the max-abs reference value)."""
import numpy as np
import torch

import oracle
from bitwise_deterministic_moe_gb300 import api, build, synth

GEMM_RTOL = 1e-2
DPROB_RTOL = 2e-3


def ensure_built():
    build.build()
    api.load()


def bf16_dev(a: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def bf16_host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class Problem:
    """A seeded problem on the device plus its routing."""

    def __init__(self, cfg, inputs=None, dev="cuda"):
        self.cfg = cfg
        self.inp = inputs if inputs is not None else synth.make_inputs(cfg)
        self.ids = torch.from_numpy(self.inp.topk_ids).to(dev)
        self.X = bf16_dev(self.inp.X, dev)
        self.W = bf16_dev(self.inp.W, dev)
        self.G = bf16_dev(self.inp.G, dev)
        self.ws = api.workspace(cfg.T, cfg.topk, cfg.E, dev)
        self.off, self.src = api.permute_indices(self.ids, cfg.E, self.ws)

    def run_dprob(self, num_ctas=0, stream=None, out=None, slots=None, dprob=None, ws=None, flags=0):
        return api.grouped_gemm_dprob(self.X, self.W, self.off, self.G, self.src, self.cfg.topk,
                                      self.ws if ws is None else ws,
                                      out=out, slots=slots, dprob=dprob, num_ctas=num_ctas, stream=stream,
                                      flags=flags)


def check_rows_against_oracle(prob, out, slots, dprob, rows):
    """Element-wise comparison of sampled permuted rows with the oracle.

    expert_out: per row, max_n |Y_gpu - Y_ref| / max_n |Y_ref| <= GEMM_RTOL.
    slots and dprob: the primary bound max |delta| / max |ref| <= DPROB_RTOL over
    the sample, and per element |delta| <= DPROB_RTOL * sum_n |G[t(r),n]| |Yb[r,n]|
    (the sum over the slot's 128 columns for a slot, over all N for dprob), so
    a small entry far below the sample's maximum is held to its own scale.
    """
    cfg, inp = prob.cfg, prob.inp
    off_ref, src_ref = oracle.routing(inp.topk_ids, cfg.E)
    rows = np.asarray(rows, dtype=np.int64)
    Y, Yb, P, D = oracle.expert_rows(inp.X, inp.W, off_ref, rows, G=inp.G, row_src=src_ref, topk=cfg.topk,
                                     want_Y=True, want_Yb=True, want_P=True, want_D=True)
    return compare_rows(out, slots, dprob, rows, Y, Yb, P, D, src_ref, inp.G, cfg.topk)


def compare_rows(out, slots, dprob, rows, Y, Yb, P, D, src_ref, G_bits, topk):
    """The tolerance checks of check_rows_against_oracle for reference values
    (Y binary64, Yb bf16 bits, P, D binary64) computed by the oracle for `rows`."""
    rows = np.asarray(rows, dtype=np.int64)
    idx = torch.from_numpy(rows).to(out.device)
    got_y = oracle.bf16_to_f64(bf16_host_bits(out.index_select(0, idx)))
    rowmax = np.maximum(np.abs(Y).max(axis=1, keepdims=True), 1e-30)
    err_y = np.abs(got_y - Y) / rowmax
    assert err_y.max() <= GEMM_RTOL, f"expert_out rel err {err_y.max():.3e}"
    if slots is None and dprob is None:
        return err_y.max()
    # per-element magnitude scales: |G[t(r), n]| * |Yb[r, n]| summed per slot and per row
    tok = src_ref[rows].astype(np.int64) // topk
    mag = np.abs(oracle.bf16_to_f64(np.asarray(G_bits)[tok])) * np.abs(oracle.bf16_to_f64(Yb))
    slot_mag = mag.reshape(rows.size, -1, 128).sum(axis=2)
    row_mag = mag.sum(axis=1)
    if slots is not None:
        got_p = slots.index_select(1, idx).t().double().cpu().numpy()
        dp = np.abs(got_p - P)
        err_p = dp.max() / max(np.abs(P).max(), 1e-30)
        assert err_p <= DPROB_RTOL, f"slot rel err {err_p:.3e}"
        worst = (dp / np.maximum(slot_mag, 1e-300)).max()
        assert np.all(dp <= DPROB_RTOL * slot_mag), f"slot per-element rel err {worst:.3e}"
    if dprob is not None:
        flat = dprob.reshape(-1)
        src = torch.from_numpy(src_ref[rows].astype(np.int64)).to(out.device)
        got_d = flat.index_select(0, src).double().cpu().numpy()
        dd = np.abs(got_d - D)
        err_d = dd.max() / max(np.abs(D).max(), 1e-30)
        assert err_d <= DPROB_RTOL, f"dprob rel err {err_d:.3e}"
        worst = (dd / np.maximum(row_mag, 1e-300)).max()
        assert np.all(dd <= DPROB_RTOL * row_mag), f"dprob per-element rel err {worst:.3e}"
    return err_y.max()


def sample_rows(off: np.ndarray, n: int, seed: int) -> np.ndarray:
    """Rows at expert boundaries (first/last of each non-empty expert among a
    sample) plus uniform random rows."""
    rng = np.random.default_rng(seed)
    R = int(off[-1])
    if R == 0:
        return np.zeros(0, np.int64)
    picks = set(rng.integers(0, R, n).tolist())
    nonempty = [e for e in range(len(off) - 1) if off[e + 1] > off[e]]
    for e in rng.choice(nonempty, min(len(nonempty), max(1, n // 4)), replace=False):
        picks.add(int(off[e]))
        picks.add(int(off[e + 1]) - 1)
    return np.array(sorted(picks), dtype=np.int64)
