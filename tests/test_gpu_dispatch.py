"""Dispatch gather, routing inverse and token combine on the GPU vs the oracle.

Integer and copy work is compared bit for bit (row_of, x_perm); the combine's
bf16 output element by element within the bf16 output bar (rel 1e-2 of each
row's max-abs) and a per-element bound from its arithmetic: one bf16 rounding
(half an ulp, 2^-9 relative) plus an fp32 multiply-add chain over topk terms.
Shapes span ragged rows (vectors per row not a multiple of 32), several
chunks of in-flight loads, every warps-per-token variant, topk from 1 to the
limit, and the full LatentMoE-shaped size.
"""
import numpy as np
import pytest
import torch

import oracle
from bitwise_deterministic_moe_gb300 import api, synth
from tests import gpu_util
from tests.gpu_util import Problem, bf16_dev, bf16_host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gpu_util.ensure_built()


def routed(cfg, dev="cuda"):
    """topk_ids from the seeded generator, routed on the GPU with the inverse map."""
    inp = synth.make_inputs(cfg, with_weights=False)
    ids = torch.from_numpy(inp.topk_ids).to(dev)
    ws = api.workspace(cfg.T, cfg.topk, cfg.E, dev)
    off, src, row_of = api.permute_indices(ids, cfg.E, ws, with_row_of=True)
    return inp, ws, off, src, row_of


def combine_bound(eo_bits, probs, row_of_ref, tokens):
    """Per-element error bound of the GPU combine against the binary64 oracle."""
    vals = oracle.bf16_to_f64(eo_bits)
    T, topk = probs.shape
    ro = row_of_ref.reshape(T, topk)
    mag = np.zeros((len(tokens), eo_bits.shape[1]))
    for j in range(topk):
        mag += np.abs(probs[tokens, j].astype(np.float64))[:, None] * np.abs(vals[ro[tokens, j]])
    return mag


def check_combine(y_dev, eo_bits, probs, src_ref, tokens):
    y_ref, yb_ref = oracle.token_combine(eo_bits, probs, src_ref, tokens)
    idx = torch.from_numpy(np.asarray(tokens, dtype=np.int64)).to(y_dev.device)
    got = oracle.bf16_to_f64(bf16_host_bits(y_dev.index_select(0, idx)))
    rowmax = np.maximum(np.abs(y_ref).max(axis=1, keepdims=True), 1e-30)
    assert (np.abs(got - y_ref) / rowmax).max() <= gpu_util.GEMM_RTOL
    topk = probs.shape[1]
    mag = combine_bound(eo_bits, probs, oracle.inverse_rows(src_ref), np.asarray(tokens))
    bound = 2.0 ** -8 * np.abs(y_ref) + 2.0 * (topk + 1) * 2.0 ** -24 * mag + 1e-38
    assert (np.abs(got - y_ref) <= bound).all()
    return float((got != oracle.bf16_to_f64(yb_ref)).mean())


GATHER_SHAPES = [
    (synth.custom_config("g8", T=33, E=3, topk=2, K=16, N=8, index=401), "H = 8: one vector per row"),
    (synth.custom_config("g136", T=129, E=7, topk=3, K=16, N=136, index=402), "17 vectors: ragged lanes"),
    (synth.custom_config("g2048", T=300, E=16, topk=6, K=16, N=2048, index=403), "one full chunk per lane"),
    (synth.custom_config("g4104", T=70, E=5, topk=4, K=16, N=4104, index=404), "513 vectors: chunk tail"),
    (synth.custom_config("g65536", T=20, E=3, topk=2, K=16, N=65536, index=405), "H at the limit: 32 chunks"),
]


@pytest.mark.parametrize("cfg,why", GATHER_SHAPES, ids=[c.name for c, _ in GATHER_SHAPES])
def test_row_of_and_gather_bit_exact(cfg, why):
    inp, ws, off, src, row_of = routed(cfg)
    off_ref, src_ref = oracle.routing(inp.topk_ids, cfg.E)
    assert np.array_equal(row_of.cpu().numpy(), oracle.inverse_rows(src_ref))
    hidden = synth.hidden_states(cfg)
    xp = api.dispatch_gather(bf16_dev(hidden), src, cfg.topk, ws)
    assert api.read_status(ws) == 0
    assert np.array_equal(bf16_host_bits(xp), oracle.dispatch(hidden, src_ref, cfg.topk))


COMBINE_SHAPES = [
    synth.custom_config("c8", T=37, E=5, topk=1, K=16, N=8, index=411),          # 1 warp per token
    synth.custom_config("c136", T=130, E=9, topk=5, K=16, N=136, index=412),     # 17 vectors, 1 warp
    synth.custom_config("c520", T=91, E=12, topk=9, K=16, N=520, index=413),     # 65 vectors, 4 warps
    synth.custom_config("c384", T=64, E=8, topk=3, K=16, N=384, index=414),      # 48 vectors, 2 warps
    synth.custom_config("c2056", T=50, E=40, topk=22, K=16, N=2056, index=415),  # 257 vectors, 8 warps + tail
    synth.custom_config("c64", T=20, E=70, topk=64, K=16, N=256, index=416),     # topk at the limit
    synth.custom_config("c65536", T=16, E=6, topk=3, K=16, N=65536, index=417),  # N at the limit
]


@pytest.mark.parametrize("cfg", COMBINE_SHAPES, ids=[c.name for c in COMBINE_SHAPES])
def test_combine_parity(cfg):
    inp, ws, off, src, row_of = routed(cfg)
    _, src_ref = oracle.routing(inp.topk_ids, cfg.E)
    eo = synth._normal_bf16(cfg.seed, 9, (cfg.R, cfg.N), 0.1)
    y = api.token_combine(bf16_dev(eo), torch.from_numpy(inp.probs).cuda(), row_of, ws)
    assert api.read_status(ws) == 0
    check_combine(y, eo, inp.probs, src_ref, np.arange(cfg.T))


@pytest.mark.parametrize("topk", [1, 2, 5, 9, 22, 64])
def test_identity_experts_give_back_hidden(topk):
    """Gather, identity experts, combine with weights 1/2, 1/4, ... summing to
    one: the fp32 chain stays within 2^-18 of the bf16 input, so the bf16
    result is the token's hidden state bit for bit."""
    cfg = synth.custom_config(f"id{topk}", T=97, E=max(topk, 8) + 3, topk=topk, K=16, N=264, index=420 + topk)
    inp, ws, off, src, row_of = routed(cfg)
    hidden = synth.hidden_states(cfg)
    h = bf16_dev(hidden)
    xp = api.dispatch_gather(h, src, topk, ws)
    p = torch.from_numpy(synth.dyadic_probs(cfg.T, topk)).cuda()
    y = api.token_combine(xp, p, row_of, ws)
    assert api.read_status(ws) == 0
    assert torch.equal(y.view(torch.int16), h.view(torch.int16))


def test_combine_after_gemm_matches_dprob_adjoint():
    """On the GEMM's own output: the combine matches the oracle, and
    <y[t], G[t]> agrees with sum_j prob[t, j] * dprob[t, j] from the fused
    epilogue (two GPU outputs tied by the adjoint identity)."""
    cfg = synth.CONFIGS["small"]
    prob = Problem(cfg)
    out, dprob, _ = prob.run_dprob()
    _, _, row_of = api.permute_indices(prob.ids, cfg.E, prob.ws, with_row_of=True)
    probs = torch.from_numpy(prob.inp.probs).cuda()
    y = api.token_combine(out, probs, row_of, prob.ws)
    assert api.read_status(prob.ws) == 0
    _, src_ref = oracle.routing(prob.inp.topk_ids, cfg.E)
    eo_bits = bf16_host_bits(out)
    tokens = np.random.default_rng(3).choice(cfg.T, 96, replace=False)
    check_combine(y, eo_bits, prob.inp.probs, src_ref, tokens)
    # adjoint: y is rounded to bf16, so compare in its own precision
    yv = y.float().double()
    g = prob.G.float().double()
    lhs = (yv * g).sum(dim=1)
    rhs = (probs.double() * dprob.double()).sum(dim=1)
    scale = (probs.double().abs() * dprob.double().abs()).sum(dim=1) + (yv.abs() * g.abs()).sum(dim=1)
    assert ((lhs - rhs).abs() <= 1e-2 * scale + 1e-30).all()


def test_deterministic_across_runs_and_streams():
    cfg = synth.custom_config("det", T=2048, E=64, topk=8, K=16, N=2048, routing="zipf", index=430)
    inp, ws, off, src, row_of = routed(cfg)
    eo = bf16_dev(synth._normal_bf16(cfg.seed, 9, (cfg.R, cfg.N), 0.1))
    hidden = bf16_dev(synth.hidden_states(cfg))
    probs = torch.from_numpy(inp.probs).cuda()
    y0 = api.token_combine(eo, probs, row_of)
    x0 = api.dispatch_gather(hidden, src, cfg.topk)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    ys = [torch.empty_like(y0) for _ in streams]
    xs = [torch.empty_like(x0) for _ in streams]
    for it in range(10):
        for s, yo, xo in zip(streams, ys, xs):
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                api.token_combine(eo, probs, row_of, out=yo)
                api.dispatch_gather(hidden, src, cfg.topk, out=xo)
        torch.cuda.synchronize()
        for yo, xo in zip(ys, xs):
            assert torch.equal(yo.view(torch.int16), y0.view(torch.int16))
            assert torch.equal(xo.view(torch.int16), x0.view(torch.int16))


def test_bad_indices_reported():
    cfg = synth.custom_config("bad", T=64, E=4, topk=2, K=16, N=256, index=431)
    inp, ws, off, src, row_of = routed(cfg)
    eo = bf16_dev(synth._normal_bf16(cfg.seed, 9, (cfg.R, cfg.N), 0.1))
    probs = torch.from_numpy(inp.probs).cuda()
    bad_of = row_of.clone()
    bad_of[7] = cfg.R + 5
    api.token_combine(eo, probs, bad_of, ws)
    assert api.read_status(ws) == 3
    bad_src = src.clone()
    bad_src[3] = -1
    api.dispatch_gather(bf16_dev(synth.hidden_states(cfg)), bad_src, cfg.topk, ws)
    assert api.read_status(ws) == 3
    # the good inputs still work afterwards
    api.token_combine(eo, probs, row_of, ws)
    assert api.read_status(ws) == 0


def test_no_tokens():
    dev = "cuda"
    hidden = torch.empty(0, 16, dtype=torch.bfloat16, device=dev)
    src = torch.empty(0, dtype=torch.int32, device=dev)
    assert api.dispatch_gather(hidden, src, 4).shape == (0, 16)
    eo = torch.empty(0, 16, dtype=torch.bfloat16, device=dev)
    probs = torch.empty(0, 4, dtype=torch.float32, device=dev)
    assert api.token_combine(eo, probs, src).shape == (0, 16)


def test_latent_full_size():
    """The LatentMoE-shaped routing (8192 tokens, top-22 of 512, 2048 wide):
    the whole x_perm bit for bit, the combine on sampled tokens."""
    cfg = synth.CONFIGS["latent"]
    inp, ws, off, src, row_of = routed(cfg)
    _, src_ref = oracle.routing(inp.topk_ids, cfg.E)
    assert np.array_equal(src.cpu().numpy(), src_ref)
    assert np.array_equal(row_of.cpu().numpy(), oracle.inverse_rows(src_ref))
    hidden = synth.hidden_states(cfg)
    xp = api.dispatch_gather(bf16_dev(hidden), src, cfg.topk, ws)
    assert api.read_status(ws) == 0
    assert np.array_equal(bf16_host_bits(xp), oracle.dispatch(hidden, src_ref, cfg.topk))
    del xp
    eo = synth._normal_bf16(cfg.seed, 9, (cfg.R, cfg.N), 0.1)
    y = api.token_combine(bf16_dev(eo), torch.from_numpy(inp.probs).cuda(), row_of, ws)
    assert api.read_status(ws) == 0
    tokens = np.concatenate([[0, 1, cfg.T - 1], np.random.default_rng(4).choice(cfg.T, 61, replace=False)])
    check_combine(y, eo, inp.probs, src_ref, tokens)
