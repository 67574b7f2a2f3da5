"""Pins for the oracle's grouped-GEMM weight gradient.

dW[e, n, c] = sum over expert e's rows r of dY[r, n] * X[r, c]: the gradient of
the FFN-out projection's weight when expert_out = X_e W_e^T.  A weight-gradient
path is one of the workloads whose determinism overhead the pages measure
("Trillion-Parameter Pretraining Goes Bitwise-Deterministic: NVIDIA Cuts the
Determinism Tax to About 2%", section "Synopsis").

Pins, each chosen so that a plausible mistake fails one of them:
* exact rational arithmetic (Python integers) on tiny inputs -- a swapped
  operand (shown by planting it), a wrong expert range or a dropped row fails;
* an independent fp64 matrix product per expert (numpy) within the
  summation bound;
* the adjoint identity <dW_e, W_e> = sum_{r in e} <dY[r], X[r] W_e^T>, which
  ties the wgrad to the forward oracle;
* an expert without rows gets exactly zero.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from bitwise_deterministic_moe_gb300 import synth
from tests.test_oracle_gemm import SCALE, bf16_int


@pytest.fixture(scope="module")
def tiny():
    cfg = synth.CONFIGS["tiny"]
    inp = synth.make_inputs(cfg)
    off, _ = oracle.routing(inp.topk_ids, cfg.E)
    dY = synth._normal_bf16(cfg.seed, 11, (cfg.R, cfg.N), 0.1)
    return cfg, inp, off, dY


def test_wgrad_exact_integers(tiny):
    cfg, inp, off, dY = tiny
    rng = np.random.default_rng(1)
    ent = np.stack([rng.integers(0, cfg.E, 40), rng.integers(0, cfg.N, 40), rng.integers(0, cfg.K, 40)], axis=1)
    got = oracle.wgrad_entries(inp.X, dY, off, ent)
    for (e, n, c), g in zip(ent, got):
        terms = [bf16_int(dY[r, n]) * bf16_int(inp.X[r, c]) for r in range(off[e], off[e + 1])]
        exact = Fraction(sum(terms), 1 << (2 * SCALE))
        bound = Fraction(max(len(terms), 1), 1 << 53) * Fraction(sum(abs(t) for t in terms), 1 << (2 * SCALE))
        assert abs(Fraction(g) - exact) <= bound * Fraction(101, 100), (e, n, c)


def test_wgrad_catches_swapped_operands(tiny):
    """Planted mistake: dY[r, c] * X[r, n] instead of dY[r, n] * X[r, c]."""
    cfg, inp, off, dY = tiny
    e = int(np.argmax(np.diff(off)))
    ent = np.array([[e, n, n + 1] for n in range(0, 64, 8)])
    got = oracle.wgrad_entries(inp.X, dY, off, ent)
    differs = 0
    for (e_, n, c), g in zip(ent, got):
        wrong = sum(bf16_int(dY[r, c]) * bf16_int(inp.X[r, n]) for r in range(off[e_], off[e_ + 1]))
        differs += abs(Fraction(g) - Fraction(wrong, 1 << (2 * SCALE))) > 1e-6
    assert differs > 0


def test_wgrad_matches_fp64_matmul(tiny):
    cfg, inp, off, dY = tiny
    x = oracle.bf16_to_f64(inp.X)
    dy = oracle.bf16_to_f64(dY)
    for e in range(cfg.E):
        got = oracle.wgrad_expert(inp.X, dY, off, e)
        rows = slice(off[e], off[e + 1])
        ref = dy[rows].T @ x[rows]
        mag = np.abs(dy[rows]).T @ np.abs(x[rows])
        assert (np.abs(got - ref) <= 2 * max(1, off[e + 1] - off[e]) * 2.0 ** -53 * mag + 1e-300).all()


def test_wgrad_adjoint_of_forward(tiny):
    """<dW_e, W_e> = sum_{r in e} <dY[r], Y[r]> with Y = X W_e^T before rounding."""
    cfg, inp, off, dY = tiny
    rows = np.arange(cfg.R)
    Y, _, _, _ = oracle.expert_rows(inp.X, inp.W, off, rows, want_Yb=False)
    w = oracle.bf16_to_f64(inp.W)
    dy = oracle.bf16_to_f64(dY)
    x = oracle.bf16_to_f64(inp.X)
    for e in range(cfg.E):
        r0, r1 = off[e], off[e + 1]
        dW = oracle.wgrad_expert(inp.X, dY, off, e)
        lhs = float(np.sum(dW * w[e]))
        rhs = float(np.sum(dy[r0:r1] * Y[r0:r1]))
        mag = float(np.sum((np.abs(dy[r0:r1]).T @ np.abs(x[r0:r1])) * np.abs(w[e])))
        assert abs(lhs - rhs) <= 4 * (cfg.K + cfg.N + (r1 - r0)) * 2.0 ** -53 * mag + 1e-300, e


def test_empty_expert_is_zero():
    cfg = synth.custom_config("holes", T=40, E=6, topk=2, K=16, N=128, index=501)
    inp = synth.make_inputs(cfg)
    ids = inp.topk_ids.copy()
    ids[ids == 3] = 4
    off, _ = oracle.routing(ids, cfg.E)
    assert off[4] == off[3]
    dY = synth._normal_bf16(cfg.seed, 11, (cfg.R, cfg.N), 0.1)
    assert np.all(oracle.wgrad_expert(inp.X, dY, off, 3) == 0.0)
