"""Block-scaled grouped GEMM (MXFP8 / NVFP4 operands) with the private-slot
dprob epilogue, on the GPU vs the oracle.

Both sides start from the same seeded bf16 operands: the GPU encodes them
with its own encoders (dmoe_quantize_mxfp8 / _nvfp4) and runs the
block-scaled GEMM; the oracle encodes them with its own encoders, decodes the
codes to binary64 and runs its grouped GEMM.  The encodings must agree byte
for byte; expert_out within rel 1e-2 of each row's max-abs; slots and dprob
within rel 2e-3 of the sample's max-abs and, per element, of the element's own
sum |G| |Yb|.  Results are bitwise identical across grids and streams."""
import numpy as np
import pytest
import torch

import oracle
from bitwise_deterministic_moe_gb300 import api, synth
from tests import gpu_util
from tests.gpu_util import Problem

pytestmark = pytest.mark.gpu

KINDS = ["mxfp8", "nvfp4"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    gpu_util.ensure_built()


def amax_bits(bits):
    """max |x| of a bf16 bit array (finite values: larger magnitude = larger pattern)."""
    m = int((np.asarray(bits, dtype=np.uint16) & np.uint16(0x7FFF)).max()) if np.asarray(bits).size else 0
    return float(oracle.bf16_to_f64(np.array([m], dtype=np.uint16))[0])


class Encoded:
    """One problem's operands encoded on the GPU (the path under test)."""

    def __init__(self, prob, kind):
        cfg = prob.cfg
        self.kind = kind
        X2 = prob.X
        W2 = prob.W.view(cfg.E * cfg.N, cfg.K)
        if kind == "mxfp8":
            self.xq, self.xs = api.quantize_mxfp8(X2)
            self.wq, self.ws = api.quantize_mxfp8(W2)
            self.xg = self.wg = None
        else:
            self.xq, self.xs, self.xg = api.quantize_nvfp4(X2, prob.ws)
            self.wq, self.ws, self.wg = api.quantize_nvfp4(W2, prob.ws)
        kb = cfg.K if kind == "mxfp8" else cfg.K // 2
        self.wq3 = self.wq.view(cfg.E, cfg.N, kb)

    def run(self, prob, grad=True, num_ctas=0, stream=None, out=None, slots=None, dprob=None, flags=0):
        cfg = prob.cfg
        G = prob.G if grad else None
        src = prob.src if grad else None
        if self.kind == "mxfp8":
            return api.grouped_gemm_dprob_mxfp8(self.xq, self.xs, self.wq3, self.ws, prob.off, G, src, cfg.topk,
                                                prob.ws, out=out, slots=slots, dprob=dprob, num_ctas=num_ctas,
                                                stream=stream, flags=flags)
        return api.grouped_gemm_dprob_nvfp4(self.xq, self.xs, self.xg, self.wq3, self.ws, self.wg, prob.off, G, src,
                                            cfg.topk, prob.ws, out=out, slots=slots, dprob=dprob, num_ctas=num_ctas,
                                            stream=stream)


def oracle_rows(prob, kind, rows, check_codes=None):
    """The oracle's encode -> decode -> binary64 grouped GEMM for `rows`
    (and the slot partials / dots of its stored bf16 output)."""
    cfg, inp = prob.cfg, prob.inp
    off, src = oracle.routing(inp.topk_ids, cfg.E)
    rows = np.asarray(rows, dtype=np.int64)
    experts = np.unique(np.searchsorted(off, rows, side="right") - 1)
    Xr = np.asarray(inp.X)[rows]
    Wb = np.asarray(inp.W)
    if kind == "mxfp8":
        xq, xs = oracle.mxfp8_quantize(Xr)
        Xd_rows = oracle.mxfp8_decode(xq, xs)
        wenc = {int(e): oracle.mxfp8_quantize(Wb[e]) for e in experts}
        dec = lambda e: oracle.mxfp8_decode(*wenc[e])
    else:
        xq, xs, sx = oracle.nvfp4_quantize(Xr, amax=amax_bits(inp.X))
        Xd_rows = oracle.nvfp4_decode(xq, xs, sx)
        aw = amax_bits(inp.W)
        wenc = {int(e): oracle.nvfp4_quantize(Wb[e], amax=aw) for e in experts}
        dec = lambda e: oracle.nvfp4_decode(*wenc[e])
    if check_codes is not None:
        # the two encoders agree byte for byte on these rows and experts
        enc = check_codes
        idx = torch.from_numpy(rows).to(enc.xq.device)
        assert np.array_equal(enc.xq.index_select(0, idx).cpu().numpy(), xq)
        assert np.array_equal(enc.xs.index_select(0, idx).cpu().numpy(), xs)
        for e in experts[:4]:
            e = int(e)
            assert np.array_equal(enc.wq3[e].cpu().numpy(), wenc[e][0])
            assert np.array_equal(enc.ws[e * cfg.N:(e + 1) * cfg.N].cpu().numpy(), wenc[e][1])
    # X decoded only for the requested rows (row i of Xd_rows is permuted row rows[i])
    n = rows.size
    Y = np.empty((n, cfg.N))
    for e in experts:
        sel = np.where((rows >= off[e]) & (rows < off[e + 1]))[0]
        Y[sel] = Xd_rows[sel] @ dec(int(e)).T
    Yb = oracle.bf16_rne(Y)
    P, D = oracle.dprob_from_output(inp.G, Yb, src[rows].astype(np.int32), cfg.topk, rows=np.arange(n))
    return Y, Yb, P, D, src


SHAPES = [
    synth.custom_config("bs_small", T=300, E=6, topk=2, K=512, N=256, index=401),
    synth.custom_config("bs_ragged", T=500, E=12, topk=3, K=1024, N=384, index=402),
    synth.custom_config("bs_manyexp", T=400, E=64, topk=4, K=512, N=256, index=403),
    synth.custom_config("bs_zipf", T=600, E=16, topk=4, K=512, N=512, routing="zipf", index=404),
    synth.custom_config("bs_n128", T=300, E=5, topk=2, K=512, N=128, index=406),     # one slot, one n-tile
]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("cfg", SHAPES, ids=[c.name for c in SHAPES])
def test_block_scaled_full_parity(cfg, kind):
    prob = Problem(cfg)
    enc = Encoded(prob, kind)
    out, dprob, slots = enc.run(prob)
    assert api.read_status(prob.ws) == 0
    rows = np.arange(cfg.R)
    Y, Yb, P, D, src = oracle_rows(prob, kind, rows, check_codes=enc)
    gpu_util.compare_rows(out, slots, dprob, rows, Y, Yb, P, D, src, prob.inp.G, cfg.topk)


@pytest.mark.parametrize("kind", KINDS)
def test_block_scaled_empty_and_hot_experts(kind):
    cfg = synth.custom_config("bs_holes", T=700, E=40, topk=4, K=512, N=256, index=405)
    inp = synth.make_inputs(cfg)
    ids = inp.topk_ids.copy()
    ids[ids % 5 == 0] = 1           # experts 0,5,10,... empty; expert 1 hot
    prob = Problem(cfg, synth.MoEInputs(cfg, ids, inp.X, inp.W, inp.G, inp.probs))
    enc = Encoded(prob, kind)
    out, dprob, slots = enc.run(prob)
    assert api.read_status(prob.ws) == 0
    rows = np.arange(cfg.R)
    Y, Yb, P, D, src = oracle_rows(prob, kind, rows)
    gpu_util.compare_rows(out, slots, dprob, rows, Y, Yb, P, D, src, prob.inp.G, cfg.topk)


@pytest.mark.parametrize("kind", KINDS)
def test_block_scaled_forward_only_and_repeatability(kind):
    """grad_out omitted: the same expert_out bits; and bitwise identical
    results across persistent grid sizes and two concurrent streams."""
    cfg = SHAPES[1]
    prob = Problem(cfg)
    enc = Encoded(prob, kind)
    out, dprob, slots = enc.run(prob)
    ref = (out.clone(), dprob.clone(), slots.clone())
    out_f, d_f, s_f = enc.run(prob, grad=False)
    assert d_f is None and s_f is None
    assert torch.equal(out_f.view(torch.int16), ref[0].view(torch.int16))
    for num_ctas in (37, 5, 1):
        o, d, s = enc.run(prob, num_ctas=num_ctas)
        assert torch.equal(o.view(torch.int16), ref[0].view(torch.int16))
        assert torch.equal(d.view(torch.int32), ref[1].view(torch.int32))
        assert torch.equal(s.view(torch.int32), ref[2].view(torch.int32))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    wss = [api.workspace(cfg.T, cfg.topk, cfg.E) for _ in streams]
    outs = []
    torch.cuda.synchronize()
    for st, ws in zip(streams, wss):
        with torch.cuda.stream(st):
            prob_ws, prob.ws = prob.ws, ws
            outs.append(enc.run(prob, stream=st))
            prob.ws = prob_ws
    torch.cuda.synchronize()
    for o, d, s in outs:
        assert torch.equal(o.view(torch.int16), ref[0].view(torch.int16))
        assert torch.equal(d.view(torch.int32), ref[1].view(torch.int32))
    for ws in wss:
        assert api.read_status(ws) == 0
    assert api.read_status(prob.ws) == 0


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("name", ["latent", "stress"])
def test_block_scaled_latent_sampled_rows(kind, name):
    """Full-size workloads -- LatentMoE-shaped (T=8192, E=512, top-22,
    K=1024, N=2048) and the stress size (T=32768, K=2048) -- on rows of
    twelve experts (the hottest, the lightest non-empty and ten others) that
    the oracle computes one by one."""
    cfg = synth.CONFIGS[name]
    prob = Problem(cfg)
    enc = Encoded(prob, kind)
    out, dprob, slots = enc.run(prob)
    assert api.read_status(prob.ws) == 0
    off = prob.off.cpu().numpy().astype(np.int64)
    counts = np.diff(off)
    nonempty = np.where(counts > 0)[0]
    rng = np.random.default_rng(cfg.seed)
    pick = {int(nonempty[np.argmax(counts[nonempty])]), int(nonempty[np.argmin(counts[nonempty])])}
    pick |= set(int(e) for e in rng.choice(nonempty, 10, replace=False))
    rows = []
    for e in sorted(pick):
        rows += [int(off[e]), int(off[e + 1]) - 1] + [int(r) for r in rng.integers(off[e], off[e + 1], 2)]
    rows = np.array(sorted(set(rows)), dtype=np.int64)
    Y, Yb, P, D, src = oracle_rows(prob, kind, rows, check_codes=enc)
    gpu_util.compare_rows(out, slots, dprob, rows, Y, Yb, P, D, src, prob.inp.G, cfg.topk)


def test_block_scaled_rejects_unsupported_shapes():
    cfg = SHAPES[0]
    prob = Problem(cfg)
    enc = Encoded(prob, "mxfp8")
    # K % 512 != 0 for MXFP8: a K of 256 is refused before any device work
    x = torch.zeros(cfg.R, 256, dtype=torch.uint8, device="cuda")
    xs = torch.zeros(cfg.R, 8, dtype=torch.uint8, device="cuda")
    w = torch.zeros(cfg.E, cfg.N, 256, dtype=torch.uint8, device="cuda")
    wsc = torch.zeros(cfg.E * cfg.N, 8, dtype=torch.uint8, device="cuda")
    with pytest.raises(api.DmoeError) as ei:
        api.grouped_gemm_dprob_mxfp8(x, xs, w, wsc, prob.off, prob.G, prob.src, cfg.topk, prob.ws)
    assert ei.value.status == 2
    del enc


@pytest.mark.parametrize("kind", KINDS)
def test_block_scaled_dprob_is_the_combine_of_its_slots(kind):
    """dprob of the block-scaled call is bit for bit the fixed-order combine
    of the slots it returns, written afresh on every call (NaN-filled
    buffers) and for every grid size."""
    cfg = SHAPES[1]
    prob = Problem(cfg)
    enc = Encoded(prob, kind)
    nan = lambda: torch.full((cfg.T, cfg.topk), float("nan"), device="cuda")
    out, dprob, slots = enc.run(prob, dprob=nan())
    assert api.read_status(prob.ws) == 0
    ref = api.dprob_combine(slots, prob.src, cfg.topk, dprob=nan())
    assert not torch.isnan(ref).any()
    assert torch.equal(dprob.view(torch.int32), ref.view(torch.int32))
    for num_ctas in (0, 9, 1):
        _, d, _ = enc.run(prob, num_ctas=num_ctas, dprob=nan())
        assert api.read_status(prob.ws) == 0
        assert torch.equal(d.view(torch.int32), ref.view(torch.int32))


def test_nvfp4_single_stage_k256():
    """NVFP4 at its smallest K (256: one 128-byte stage per row, one 16-byte
    scale unit), ragged experts, every row against the oracle."""
    cfg = synth.custom_config("bs_k256", T=400, E=7, topk=3, K=256, N=256, index=407)
    prob = Problem(cfg)
    enc = Encoded(prob, "nvfp4")
    out, dprob, slots = enc.run(prob)
    assert api.read_status(prob.ws) == 0
    rows = np.arange(cfg.R)
    Y, Yb, P, D, src = oracle_rows(prob, "nvfp4", rows, check_codes=enc)
    gpu_util.compare_rows(out, slots, dprob, rows, Y, Yb, P, D, src, prob.inp.G, cfg.topk)


@pytest.mark.parametrize("name", ["bs_small", "bs_zipf", "latent"])
def test_mxfp8_two_slot_tiles_equal_one_slot_tiles(name):
    """MXFP8 with N % 256 == 0 runs 128 x 256 tiles (the two slots' MMAs
    share the A operand); forcing 128 x 128 tiles gives the same bits:
    expert_out, slots and dprob, forward and dprob calls, two grid sizes."""
    cfg = synth.CONFIGS[name] if name in synth.CONFIGS else next(c for c in SHAPES if c.name == name)
    assert cfg.N % 256 == 0
    prob = Problem(cfg)
    enc = Encoded(prob, "mxfp8")
    wide = enc.run(prob)
    wide = tuple(t.clone() for t in wide)
    narrow = enc.run(prob, flags=api.LAUNCH_NARROW_TILES)
    for a, b in zip(wide, narrow):
        assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a.view(torch.int16),
                           b.view(torch.int32) if b.dtype == torch.float32 else b.view(torch.int16))
    fw = enc.run(prob, grad=False)[0].clone()
    fn = enc.run(prob, grad=False, flags=api.LAUNCH_NARROW_TILES)[0]
    assert torch.equal(fw.view(torch.int16), fn.view(torch.int16))
    assert torch.equal(fw.view(torch.int16), wide[0].view(torch.int16))
    o, d, s_ = enc.run(prob, num_ctas=37)
    assert torch.equal(o.view(torch.int16), wide[0].view(torch.int16))
    assert torch.equal(d.view(torch.int32), wide[1].view(torch.int32))
    assert api.read_status(prob.ws) == 0
