"""Pins for the oracle's dispatch gather, row inverse and token combine.

The steps either side of the grouped GEMM: each token's hidden state is copied
to every permuted row it was routed to, and each token's output is the sum of
its expert outputs weighted by the routing probabilities.  dprob is the
derivative of that combine with respect to the probabilities ("Trillion-
Parameter Pretraining Goes Bitwise-Deterministic: NVIDIA Cuts the Determinism
Tax to About 2%", section "Interpretation"), and routing maps and dispatch
outputs are order-sensitive data ("NVIDIA fait passer le déterminisme bit à
bit de Megatron Core à 2432 GPU ...", section "Méthodologie de débogage du
non-déterminisme").

Pins, chosen so that a plausible mistake fails one of them:
* brute-force Python loops for the inverse and the gather;
* a closed form: identity experts with power-of-two weights that sum to one
  give back every token's hidden state exactly, bit for bit -- a wrong row,
  token or weight index fails;
* exact rational arithmetic for the combine on tiny inputs;
* the adjoint identity <y[t], G[t]> = sum_j prob[t,j] * dprob[t,j], which ties
  the combine to the dprob oracle -- reading rows through row_src instead of
  its inverse fails it (checked by planting exactly that mistake);
* permuting the token order permutes the combined rows, bitwise.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from bitwise_deterministic_moe_gb300 import synth


@pytest.fixture(scope="module")
def tiny():
    cfg = synth.CONFIGS["tiny"]
    inp = synth.make_inputs(cfg)
    off, row_src = oracle.routing(inp.topk_ids, cfg.E)
    hidden = synth.hidden_states(cfg)
    return cfg, inp, off, row_src, hidden


def test_inverse_rows_brute(tiny):
    cfg, inp, off, row_src, hidden = tiny
    row_of = oracle.inverse_rows(row_src)
    for f in range(cfg.R):
        r = int(row_of[f])
        assert 0 <= r < cfg.R and int(row_src[r]) == f
    with pytest.raises(ValueError):
        oracle.inverse_rows(np.array([0, 0, 2], dtype=np.int32))


def test_dispatch_brute(tiny):
    cfg, inp, off, row_src, hidden = tiny
    Xp = oracle.dispatch(hidden, row_src, cfg.topk)
    assert Xp.shape == (cfg.R, cfg.N) and Xp.dtype == np.uint16
    for r in range(0, cfg.R, 3):
        t = int(row_src[r]) // cfg.topk
        assert list(Xp[r]) == list(hidden[t])
    # every routed (token, choice) lands in exactly one row of its expert
    eid = inp.topk_ids.reshape(-1)
    for f in range(0, cfg.R, 5):
        r = int(oracle.inverse_rows(row_src)[f])
        assert off[eid[f]] <= r < off[eid[f] + 1]


def test_identity_experts_give_back_hidden(tiny):
    """Closed form: expert_out = X_perm and weights 1/2, 1/4, ..., summing to
    one; every partial sum is exact in binary64, so y = hidden bit for bit."""
    cfg, inp, off, row_src, hidden = tiny
    Xp = oracle.dispatch(hidden, row_src, cfg.topk)
    p = synth.dyadic_probs(cfg.T, cfg.topk)
    y, yb = oracle.token_combine(Xp, p, row_src)
    assert np.array_equal(y, oracle.bf16_to_f64(hidden))
    assert np.array_equal(yb, hidden)


def test_identity_roundtrip_uneven_topk():
    """Same closed form with topk = 5 (weights 1/2, 1/4, 1/8, 1/16, 1/16) and a
    ragged token count."""
    cfg = synth.custom_config("t5", T=37, E=11, topk=5, K=16, N=136, index=7)
    inp = synth.make_inputs(cfg, with_weights=False)
    _, row_src = oracle.routing(inp.topk_ids, cfg.E)
    hidden = synth.hidden_states(cfg)
    p = synth.dyadic_probs(cfg.T, cfg.topk)
    _, yb = oracle.token_combine(oracle.dispatch(hidden, row_src, cfg.topk), p, row_src)
    assert np.array_equal(yb, hidden)


def test_combine_exact_rational(tiny):
    cfg, inp, off, row_src, hidden = tiny
    # stored expert outputs: any bf16 rows will do; use X_perm-shaped draws of width N
    eo = synth._normal_bf16(cfg.seed, 9, (cfg.R, cfg.N), 0.1)
    tokens = np.array([0, 1, 77, 128, cfg.T - 1])
    y, _ = oracle.token_combine(eo, inp.probs, row_src, tokens)
    row_of = oracle.inverse_rows(row_src).reshape(cfg.T, cfg.topk)
    vals = oracle.bf16_to_f64(eo)
    for i, t in enumerate(tokens):
        for n in range(0, cfg.N, 11):
            terms = [Fraction(float(inp.probs[t, j])) * Fraction(float(vals[row_of[t, j], n]))
                     for j in range(cfg.topk)]
            exact = sum(terms)
            bound = Fraction(cfg.topk, 1 << 53) * sum(abs(x) for x in terms) * Fraction(101, 100)
            assert abs(Fraction(y[i, n]) - exact) <= bound, (t, n)


def _adjoint_gaps(eo, probs, G, row_src, topk, tokens):
    """|<y[t],G[t]> - sum_j p[t,j] D[t,j]| and its rounding bound, per token."""
    y, _ = oracle.token_combine(eo, probs, row_src, tokens)
    _, D = oracle.dprob_from_output(G, eo, row_src, topk)
    dprob = oracle.combine(D, row_src, probs.shape[0], topk)
    g = oracle.bf16_to_f64(G)
    vals = oracle.bf16_to_f64(eo)
    row_of = oracle.inverse_rows(row_src).reshape(probs.shape[0], topk)
    N = eo.shape[1]
    out = []
    for i, t in enumerate(tokens):
        lhs = math.fsum((y[i] * g[t]).tolist())
        rhs = math.fsum([float(probs[t, j]) * dprob[t, j] for j in range(topk)])
        mag = sum(float(abs(probs[t, j])) * float(np.abs(g[t] * vals[row_of[t, j]]).sum()) for j in range(topk))
        out.append((abs(lhs - rhs), 2.0 * (topk + N + 2) * 2.0 ** -53 * mag))
    return out


def test_combine_adjoint_identity(tiny):
    cfg, inp, off, row_src, hidden = tiny
    eo = synth._normal_bf16(cfg.seed, 9, (cfg.R, cfg.N), 0.1)
    for gap, bound in _adjoint_gaps(eo, inp.probs, inp.G, row_src, cfg.topk, np.arange(0, cfg.T, 5)):
        assert gap <= bound


def test_adjoint_catches_wrong_direction(tiny, monkeypatch):
    """Planted mistake: indexing rows by row_src instead of its inverse."""
    cfg, inp, off, row_src, hidden = tiny
    assert not np.array_equal(oracle.inverse_rows(row_src), row_src)
    eo = synth._normal_bf16(cfg.seed, 9, (cfg.R, cfg.N), 0.1)
    real = oracle.inverse_rows
    monkeypatch.setattr(oracle, "inverse_rows", lambda rs: np.asarray(rs, dtype=np.int32).copy())
    y_bad, _ = oracle.token_combine(eo, inp.probs, row_src, np.arange(0, cfg.T, 5))
    monkeypatch.setattr(oracle, "inverse_rows", real)
    y_ok, _ = oracle.token_combine(eo, inp.probs, row_src, np.arange(0, cfg.T, 5))
    assert not np.allclose(y_bad, y_ok)
    gaps = _adjoint_gaps(eo, inp.probs, inp.G, row_src, cfg.topk, np.arange(0, cfg.T, 5))
    g = oracle.bf16_to_f64(inp.G)
    bad = 0
    for i, t in enumerate(np.arange(0, cfg.T, 5)):
        lhs = math.fsum((y_bad[i] * g[t]).tolist())
        ok_lhs = math.fsum((y_ok[i] * g[t]).tolist())
        if abs(lhs - ok_lhs) > gaps[i][1] * 4:
            bad += 1
    assert bad > 0


def test_combine_token_permutation_bitwise(tiny):
    """Permuting the tokens (routing, weights and their expert-output rows with
    them) permutes the combined rows, bit for bit."""
    cfg, inp, off, row_src, hidden = tiny
    eo = synth._normal_bf16(cfg.seed, 9, (cfg.R, cfg.N), 0.1)
    y, yb = oracle.token_combine(eo, inp.probs, row_src)
    pi = np.random.default_rng(5).permutation(cfg.T)
    ids2 = inp.topk_ids[pi]
    probs2 = inp.probs[pi]
    _, row_src2 = oracle.routing(ids2, cfg.E)
    row_of = oracle.inverse_rows(row_src).reshape(cfg.T, cfg.topk)
    row_of2 = oracle.inverse_rows(row_src2).reshape(cfg.T, cfg.topk)
    eo2 = np.empty_like(eo)
    for t2 in range(cfg.T):
        for j in range(cfg.topk):
            eo2[row_of2[t2, j]] = eo[row_of[pi[t2], j]]
    y2, yb2 = oracle.token_combine(eo2, probs2, row_src2)
    assert np.array_equal(y2, y[pi]) and np.array_equal(yb2, yb[pi])
