"""Pins for the oracle's grouped GEMM, private-slot partials and dprob.

What the pages fix ("Trillion-Parameter Pretraining Goes Bitwise-Deterministic:
NVIDIA Cuts the Determinism Tax to About 2%", section "Interpretation"): the
grouped GEMM's epilogue produces dprob[token] as a sum of per-N-tile
contributions; each N-tile writes a private slot and the slots are combined in
a fixed order.  So the slot sum must equal the full per-row dot product, and
dprob is the derivative of the loss sum_{t,j} prob[t,j] <expert_out[t,j],
grad_out[t]> with respect to prob.

Pins, each chosen so that a plausible mistake fails one of them:
* exact rational arithmetic (Python integers) for the GEMM and the dots on
  tiny inputs -- a transposed operand, a wrong expert or a dropped term fails;
* the binary64 result is within the textbook summation bound of the exact one;
* finite differences of the loss give dprob -- a wrong token index fails;
* a direct per-(token, choice) loop that never uses the permutation;
* slot partials summed in any order equal the full dot;
* relabelling experts and permuting tokens leaves dprob unchanged, bitwise.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from bitwise_deterministic_moe_gb300 import synth

SCALE = 133   # every bf16 value times 2^133 is an integer


def bf16_int(b):
    """bf16 pattern -> integer v such that value = v / 2^133 (exact)."""
    b = int(b)
    sign = -1 if b & 0x8000 else 1
    e = (b >> 7) & 0xFF
    m = b & 0x7F
    assert e != 0xFF
    if e == 0:
        return sign * m
    return sign * ((128 + m) << (e - 1))


@pytest.fixture(scope="module")
def tiny():
    cfg = synth.CONFIGS["tiny"]
    inp = synth.make_inputs(cfg)
    off, row_src = oracle.routing(inp.topk_ids, cfg.E)
    return cfg, inp, off, row_src


def expert_of(off, r):
    return int(np.searchsorted(off, r, side="right") - 1)


def test_gemm_exact_integers(tiny):
    cfg, inp, off, row_src = tiny
    rows = np.array([0, 1, 63, 64, 200, 255, 256, 400, cfg.R - 1], dtype=np.int64)
    Y, Yb, _, _ = oracle.expert_rows(inp.X, inp.W, off, rows)
    for i, r in enumerate(rows):
        e = expert_of(off, r)
        x = [bf16_int(v) for v in inp.X[r]]
        for n in range(0, cfg.N, 7):
            w = [bf16_int(v) for v in inp.W[e, n]]
            exact = sum(a * b for a, b in zip(x, w))                  # scaled by 2^266
            absum = sum(abs(a * b) for a, b in zip(x, w))
            err = abs(Fraction(Y[i, n]) - Fraction(exact, 1 << (2 * SCALE)))
            bound = Fraction(cfg.K, 1 << 53) * Fraction(absum, 1 << (2 * SCALE)) * 1.01
            assert err <= bound, (r, n)


def test_gemm_catches_transposed_weight(tiny):
    """Planted mistake: reading W[e, c, n] instead of W[e, n, c] is detected."""
    cfg, inp, off, row_src = tiny
    r = 5
    e = expert_of(off, r)
    Y, _, _, _ = oracle.expert_rows(inp.X, inp.W, off, np.array([r]))
    x = [bf16_int(v) for v in inp.X[r]]
    wrong = [sum(a * bf16_int(inp.W[e, c, n]) for c, a in enumerate(x)) for n in range(4)]
    assert any(abs(Fraction(Y[0, n]) - Fraction(wrong[n], 1 << 266)) > 1e-6 for n in range(4))


def test_dots_exact_integers(tiny):
    """P and D from the stored bf16 output against exact integer dots."""
    cfg, inp, off, row_src = tiny
    rows = np.arange(0, cfg.R, 37, dtype=np.int64)
    _, Yb, P, D = oracle.expert_rows(inp.X, inp.W, off, rows, G=inp.G, row_src=row_src,
                                     topk=cfg.topk, want_P=True, want_D=True)
    for i, r in enumerate(rows):
        t = int(row_src[r]) // cfg.topk
        g = [bf16_int(v) for v in inp.G[t]]
        y = [bf16_int(v) for v in Yb[i]]
        terms = [a * b for a, b in zip(g, y)]
        exact = Fraction(sum(terms), 1 << 266)
        bound = Fraction(cfg.N, 1 << 53) * Fraction(sum(abs(v) for v in terms), 1 << 266) * 1.01
        assert abs(Fraction(D[i]) - exact) <= bound
        for s in range(cfg.S):
            seg = terms[s * 128:(s + 1) * 128]
            ex = Fraction(sum(seg), 1 << 266)
            bd = Fraction(128, 1 << 53) * Fraction(sum(abs(v) for v in seg), 1 << 266) * 1.01
            assert abs(Fraction(P[i, s]) - ex) <= bd


def _rne_fraction(q: Fraction) -> int:
    """Exact bf16 rounding of a rational (normal range only), as a pattern."""
    if q == 0:
        return 0
    sign = 0x8000 if q < 0 else 0
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    quantum = Fraction(2) ** (e - 7)
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    r = fl + 1 if rem > Fraction(1, 2) else fl if rem < Fraction(1, 2) else (fl if fl % 2 == 0 else fl + 1)
    if r == 256:
        r, e = 128, e + 1
    return sign | ((e + 127) << 7) | (r - 128)


def test_stored_output_is_rounded_exact_value(tiny):
    cfg, inp, off, row_src = tiny
    rows = np.array([3, 77, 300], dtype=np.int64)
    Y, Yb, _, _ = oracle.expert_rows(inp.X, inp.W, off, rows)
    for i, r in enumerate(rows):
        e = expert_of(off, r)
        x = [bf16_int(v) for v in inp.X[r]]
        for n in range(cfg.N):
            w = [bf16_int(v) for v in inp.W[e, n]]
            exact = Fraction(sum(a * b for a, b in zip(x, w)), 1 << 266)
            want = _rne_fraction(exact)
            if int(Yb[i, n]) != want:
                # allowed only when binary64 rounding moved the value across a tie
                lo, hi = sorted([int(Yb[i, n]) & 0x7FFF, want & 0x7FFF])
                assert hi - lo == 1
                assert abs(Fraction(Y[i, n]) - exact) > 0


def loss(inp, off, row_src, Yb_all, p):
    """L(p) = sum_t < sum_j p[t,j] * expert_out[t,j], grad_out[t] >  (binary64)."""
    cfg = inp.cfg
    inv = np.empty(cfg.R, dtype=np.int64)
    inv[row_src] = np.arange(cfg.R)
    yb = oracle.bf16_to_f64(Yb_all)                     # [R, N] in permuted order
    g = oracle.bf16_to_f64(inp.G)                        # [T, N]
    y_tok = yb[inv].reshape(cfg.T, cfg.topk, cfg.N)     # token order
    mix = np.einsum("tj,tjn->tn", p, y_tok)
    return float(np.sum(mix * g)), float(np.sum(np.abs(p)[:, :, None] * np.abs(y_tok) * np.abs(g)[:, None, :]))


def test_dprob_finite_difference(tiny):
    cfg, inp, off, row_src = tiny
    ref = oracle.full(inp)
    p = inp.probs.astype(np.float64)
    h = 2.0 ** -10
    rng = np.random.default_rng(3)
    for _ in range(24):
        t = int(rng.integers(cfg.T))
        j = int(rng.integers(cfg.topk))
        pp, pm = p.copy(), p.copy()
        pp[t, j] += h
        pm[t, j] -= h
        lp, mag = loss(inp, off, row_src, ref["Yb"], pp)
        lm, _ = loss(inp, off, row_src, ref["Yb"], pm)
        fd = (lp - lm) / (2 * h)
        bound = 4 * 2.0 ** -53 * mag / h * 4
        assert abs(fd - ref["dprob"][t, j]) <= bound + 1e-300, (t, j)


def test_finite_difference_catches_wrong_token(tiny):
    """Planted mistake: dprob taken with the neighbouring token's gradient."""
    cfg, inp, off, row_src = tiny
    ref = oracle.full(inp)
    g_shift = np.roll(inp.G, 1, axis=0)
    _, D_bad = oracle.dprob_from_output(g_shift, ref["Yb"], row_src, cfg.topk)
    bad = oracle.combine(D_bad, row_src, cfg.T, cfg.topk)
    p = inp.probs.astype(np.float64)
    h = 2.0 ** -10
    t, j = 10, 1
    pp, pm = p.copy(), p.copy()
    pp[t, j] += h
    pm[t, j] -= h
    fd = (loss(inp, off, row_src, ref["Yb"], pp)[0] - loss(inp, off, row_src, ref["Yb"], pm)[0]) / (2 * h)
    assert abs(fd - bad[t, j]) > 1e-6
    assert abs(fd - ref["dprob"][t, j]) < 1e-9


def test_direct_loop_without_permutation(tiny):
    """dprob[t,j] from a direct loop over (t, j) and the expert id in topk_ids
    equals the permuted computation bit for bit (same terms, same order)."""
    cfg, inp, off, row_src = tiny
    ref = oracle.full(inp)
    inv = np.empty(cfg.R, dtype=np.int64)
    inv[row_src] = np.arange(cfg.R)
    g = oracle.bf16_to_f64(inp.G)
    for t in range(0, cfg.T, 17):
        for j in range(cfg.topk):
            e = int(inp.topk_ids[t, j])
            x = oracle.bf16_to_f64(inp.X[inv[t * cfg.topk + j]])
            w = oracle.bf16_to_f64(inp.W[e])
            y = np.zeros(cfg.N)
            for c in range(cfg.K):            # ascending reduction index, like the definition
                y = y + x[c] * w[:, c]
            yb = oracle.bf16_to_f64(oracle.bf16_rne(y))
            d = 0.0
            for n in range(cfg.N):
                d += g[t, n] * yb[n]
            assert d == ref["dprob"][t, j], (t, j)


def test_slot_sum_any_order_equals_full_dot(tiny):
    cfg, inp, off, row_src = tiny
    ref = oracle.full(inp)
    P, D = ref["P"], ref["D"]
    g = oracle.bf16_to_f64(inp.G)
    yb = oracle.bf16_to_f64(ref["Yb"])
    mag = np.abs(g[row_src // cfg.topk]) * np.abs(yb)
    rng = np.random.default_rng(9)
    for _ in range(5):
        order = rng.permutation(P.shape[1])
        s = np.zeros(cfg.R)
        for k in order:
            s = s + P[:, k]
        bound = (cfg.S + 128) * 2.0 ** -52 * mag.sum(axis=1)
        assert np.all(np.abs(s - D) <= bound)


def test_relabel_and_token_permutation_invariance():
    cfg = synth.custom_config("perm", T=96, E=6, topk=3, K=64, N=256, index=201)
    inp = synth.make_inputs(cfg)
    off, row_src = oracle.routing(inp.topk_ids, cfg.E)
    base = oracle.full(inp)["dprob"]
    inv = np.empty(cfg.R, dtype=np.int64)
    inv[row_src] = np.arange(cfg.R)
    X_tok = inp.X[inv].reshape(cfg.T, cfg.topk, cfg.K)     # X row of each (t, j)

    rng = np.random.default_rng(4)
    # 1) expert relabelling: W'[pi(e)] = W[e], ids' = pi(ids)
    pi = rng.permutation(cfg.E)
    W2 = np.empty_like(inp.W)
    W2[pi] = inp.W
    ids2 = pi[inp.topk_ids].astype(np.int32)
    off2, src2 = oracle.routing(ids2, cfg.E)
    X2 = X_tok.reshape(cfg.R, cfg.K)[src2]
    inp2 = synth.MoEInputs(cfg, ids2, X2, W2, inp.G, inp.probs)
    np.testing.assert_array_equal(oracle.full(inp2)["dprob"], base)

    # 2) token permutation
    tp = rng.permutation(cfg.T)
    ids3 = inp.topk_ids[tp]
    off3, src3 = oracle.routing(ids3, cfg.E)
    X3 = X_tok[tp].reshape(cfg.R, cfg.K)[src3]
    inp3 = synth.MoEInputs(cfg, ids3, X3, inp.W, inp.G[tp], inp.probs[tp])
    np.testing.assert_array_equal(oracle.full(inp3)["dprob"], base[tp])


def test_empty_expert_and_ragged_rows():
    """Experts with no rows are skipped; every row is covered exactly once."""
    cfg = synth.custom_config("ragged", T=50, E=7, topk=2, K=32, N=384, index=202)
    inp = synth.make_inputs(cfg)
    ids = inp.topk_ids.copy()
    ids[ids == 3] = 4          # expert 3 now empty; duplicates allowed
    off, row_src = oracle.routing(ids, cfg.E)
    assert off[4] == off[3]
    inp2 = synth.MoEInputs(cfg, ids, inp.X, inp.W, inp.G, inp.probs)
    ref = oracle.full(inp2)
    assert np.all(np.isfinite(ref["dprob"]))
    with pytest.raises(ValueError):
        oracle.expert_rows(inp.X, inp.W, off, np.array([cfg.R]))
