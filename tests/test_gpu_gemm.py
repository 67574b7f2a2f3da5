"""Grouped GEMM + private-slot dprob on the GPU vs the oracle, element by
element, on shapes that span several tiles, ragged expert tails, empty
experts, K tails and half-width N tiles; plus sampled rows at the full
LatentMoE-shaped size in the benchmark's launch configuration."""
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


SHAPES = [
    synth.CONFIGS["tiny"],
    synth.custom_config("ragged", T=600, E=12, topk=3, K=320, N=384, index=301),   # K tail, N % 256 == 128
    synth.custom_config("wide", T=300, E=5, topk=2, K=72, N=1024, index=302),      # K < one stage
    synth.custom_config("manyexp", T=700, E=1024, topk=8, K=128, N=256, index=303),  # many small experts
    synth.custom_config("zipf", T=1024, E=64, topk=6, K=256, N=512, routing="zipf", index=304),
    synth.custom_config("n128", T=400, E=6, topk=2, K=192, N=128, index=306),       # one slot, half N-tile only
]

# large dimensions (index arithmetic past 2^31 bytes of W, deep K, wide N), sampled rows
LARGE = [
    synth.custom_config("wideN", T=96, E=4, topk=2, K=128, N=8192, index=307),
    synth.custom_config("deepK", T=160, E=8, topk=3, K=8192, N=256, index=308),
    synth.custom_config("bigW", T=256, E=1024, topk=2, K=4096, N=512, index=309),  # W = 4 GiB
    # the documented extremes: K = 8 (one 8-column slice, the rest of the box
    # zero-filled), K = 65536 (1024 k-blocks), N = 65536 (256 n-tiles, 512 slots)
    synth.custom_config("k8", T=200, E=3, topk=2, K=8, N=256, index=311),
    synth.custom_config("k64k", T=40, E=2, topk=1, K=65536, N=128, index=312),
    synth.custom_config("n64k", T=24, E=2, topk=2, K=64, N=65536, index=313),
]


KERNELS = [api.LAUNCH_SINGLE_CTA, api.LAUNCH_CTA_PAIRS]
KERNEL_IDS = ["single", "pairs"]


@pytest.mark.parametrize("flags", KERNELS, ids=KERNEL_IDS)
@pytest.mark.parametrize("cfg", SHAPES, ids=[c.name for c in SHAPES])
def test_full_parity_small_shapes(cfg, flags):
    prob = Problem(cfg)
    out, dprob, slots = prob.run_dprob(flags=flags)
    assert api.read_status(prob.ws) == 0
    rows = np.arange(cfg.R)
    gpu_util.check_rows_against_oracle(prob, out, slots, dprob, rows)


def fuzz_shapes(n, seed=2024):
    """Seeded random shapes inside the supported envelope: T 50-900 tokens,
    1-96 experts, top-1 to top-8, K a multiple of 8 up to 1024, N a multiple
    of 128 up to 1024, uniform or Zipf routing."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(rng.integers(1, 97))
        topk = int(rng.integers(1, min(8, E) + 1))
        T = int(rng.integers(50, 901))
        K = 8 * int(rng.integers(1, 129))
        N = 128 * int(rng.integers(1, 9))
        routing = "zipf" if rng.random() < 0.5 else "uniform"
        out.append(synth.custom_config(f"fuzz{i}", T=T, E=E, topk=topk, K=K, N=N, routing=routing, index=320 + i))
    return out


FUZZ = fuzz_shapes(8)


@pytest.mark.parametrize("flags", KERNELS, ids=KERNEL_IDS)
@pytest.mark.parametrize("cfg", FUZZ, ids=[f"{c.name}-T{c.T}-E{c.E}-k{c.topk}-K{c.K}-N{c.N}" for c in FUZZ])
def test_fuzz_shapes_full_parity(cfg, flags):
    prob = Problem(cfg)
    out, dprob, slots = prob.run_dprob(flags=flags)
    assert api.read_status(prob.ws) == 0
    gpu_util.check_rows_against_oracle(prob, out, slots, dprob, np.arange(cfg.R))


@pytest.mark.parametrize("flags", KERNELS, ids=KERNEL_IDS)
@pytest.mark.parametrize("cfg", SHAPES[:2], ids=[c.name for c in SHAPES[:2]])
def test_fwd_equals_dprob_output_and_unfused_epilogue(cfg, flags):
    prob = Problem(cfg)
    out, dprob, slots = prob.run_dprob(flags=flags)
    out2 = api.grouped_gemm_fwd(prob.X, prob.W, prob.off, prob.ws, flags=flags)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    slots2 = api.dprob_epilogue(prob.G, out, prob.off, prob.src, cfg.topk)
    assert torch.equal(slots.view(torch.int32), slots2.view(torch.int32))      # fused == unfused, bitwise
    dprob2 = api.dprob_combine(slots2, prob.src, cfg.topk)
    assert torch.equal(dprob.view(torch.int32), dprob2.view(torch.int32))


def test_unfused_epilogue_on_oracle_output():
    """The unfused epilogue + combine on the ORACLE's bf16 output vs oracle dots."""
    cfg = SHAPES[1]
    inp = synth.make_inputs(cfg)
    ref = oracle.full(inp)
    ws = api.workspace(cfg.T, cfg.topk, cfg.E)
    off = torch.from_numpy(ref["off"]).cuda()
    src = torch.from_numpy(ref["row_src"]).cuda()
    Yb = gpu_util.bf16_dev(ref["Yb"])
    G = gpu_util.bf16_dev(inp.G)
    slots = api.dprob_epilogue(G, Yb, off, src, cfg.topk)
    dprob = api.dprob_combine(slots, src, cfg.topk)
    P = ref["P"]
    got_p = slots.t().double().cpu().numpy()
    assert np.abs(got_p - P).max() <= 2e-3 * np.abs(P).max()
    D = ref["dprob"]
    assert np.abs(dprob.double().cpu().numpy() - D).max() <= 2e-3 * np.abs(D).max()


@pytest.mark.parametrize("flags", KERNELS, ids=KERNEL_IDS)
def test_atomic_control_close_to_deterministic(flags):
    cfg = SHAPES[4]
    prob = Problem(cfg)
    out, dprob, _ = prob.run_dprob(flags=flags)
    out_a, dprob_a = api.grouped_gemm_dprob_atomic(prob.X, prob.W, prob.off, prob.G, prob.src, cfg.topk, prob.ws,
                                                   flags=flags)
    assert torch.equal(out.view(torch.int16), out_a.view(torch.int16))
    scale = dprob.abs().max().item()
    assert (dprob - dprob_a).abs().max().item() <= 1e-5 * scale
    rows = np.arange(0, cfg.R, 7)
    gpu_util.check_rows_against_oracle(prob, out_a, None, dprob_a, rows)


@pytest.mark.parametrize("flags", KERNELS, ids=KERNEL_IDS)
def test_empty_experts_and_hot_expert(flags):
    cfg = synth.custom_config("holes", T=900, E=40, topk=4, K=192, N=256, index=305)
    inp = synth.make_inputs(cfg)
    ids = inp.topk_ids.copy()
    ids[ids % 5 == 0] = 1           # experts 0,5,10,... empty; expert 1 hot (duplicates allowed)
    inp2 = synth.MoEInputs(cfg, ids, inp.X, inp.W, inp.G, inp.probs)
    prob = Problem(cfg, inp2)
    out, dprob, slots = prob.run_dprob(flags=flags)
    assert api.read_status(prob.ws) == 0
    gpu_util.check_rows_against_oracle(prob, out, slots, dprob, np.arange(cfg.R))


@pytest.mark.parametrize("flags", KERNELS, ids=KERNEL_IDS)
def test_bad_offsets_set_routing_status(flags):
    cfg = SHAPES[0]
    prob = Problem(cfg)
    bad = prob.off.clone()
    bad[3] = bad[4] + 1            # not monotone
    api.grouped_gemm_fwd(prob.X, prob.W, bad, prob.ws, flags=flags)
    assert api.read_status(prob.ws) == 3
    bad = prob.off.clone()
    bad[-1] -= 1                   # does not end at R
    api.grouped_gemm_fwd(prob.X, prob.W, bad, prob.ws, flags=flags)
    assert api.read_status(prob.ws) == 3
    assert api.read_status(prob.ws) == 0   # cleared by the read


def test_zero_rows():
    ws = api.workspace(0, 2, 4)
    X = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.randn(4, 256, 64, device="cuda").to(torch.bfloat16)
    off = torch.zeros(5, dtype=torch.int32, device="cuda")
    out = api.grouped_gemm_fwd(X, W, off, ws)
    torch.cuda.synchronize()
    assert out.shape == (0, 256)


@pytest.mark.parametrize("name", ["small", "latent", "imbal", "stress"])
def test_full_size_sampled_rows(name):
    """Full size, in the benchmark's launch configuration (flags 0) and with
    each kernel forced, on sampled rows the oracle computes one by one, with
    the per-element bound on slots and dprob."""
    cfg = synth.CONFIGS[name]
    prob = Problem(cfg)
    off = prob.off.cpu().numpy()
    rows = gpu_util.sample_rows(off, 96, seed=cfg.seed)
    for flags in [0] + KERNELS:
        out, dprob, slots = prob.run_dprob(flags=flags)
        assert api.read_status(prob.ws) == 0
        gpu_util.check_rows_against_oracle(prob, out, slots, dprob, rows)
        del out, dprob, slots


@pytest.mark.parametrize("name", ["tiny", "small", "latent", "imbal"])
def test_single_and_pair_kernels_bitwise_equal(name):
    """The two kernels give the same bits, so the automatic choice between
    them never changes a result."""
    prob = Problem(synth.CONFIGS[name])
    o1, d1, s1 = prob.run_dprob(flags=api.LAUNCH_SINGLE_CTA)
    o1, d1, s1 = o1.clone(), d1.clone(), s1.clone()
    o2, d2, s2 = prob.run_dprob(flags=api.LAUNCH_CTA_PAIRS)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(s1.view(torch.int32), s2.view(torch.int32))
    assert torch.equal(d1.view(torch.int32), d2.view(torch.int32))
    assert api.read_status(prob.ws) == 0


@pytest.mark.parametrize("name", ["latent", "imbal"])
def test_unfused_epilogue_full_size_bitwise(name):
    """The separate epilogue and combine launches give the fused call's slots
    and dprob bit for bit at full size (every row, every slot)."""
    prob = Problem(synth.CONFIGS[name])
    out, dprob, slots = prob.run_dprob()
    slots2 = api.dprob_epilogue(prob.G, out, prob.off, prob.src, prob.cfg.topk)
    dprob2 = api.dprob_combine(slots2, prob.src, prob.cfg.topk)
    assert api.read_status(prob.ws) == 0
    assert torch.equal(slots.view(torch.int32), slots2.view(torch.int32))
    assert torch.equal(dprob.view(torch.int32), dprob2.view(torch.int32))


@pytest.mark.parametrize("num_ctas", [0, 37, 1])
@pytest.mark.parametrize("cfg", SHAPES, ids=[c.name for c in SHAPES])
def test_serialized_writers_bitwise_equal_to_slots(cfg, num_ctas):
    """The serialized-writer control adds the slots into dprob in ascending
    order as they come, so it must give the fixed-order combine's bits (and the
    same expert_out) for any grid, including a single CTA that holds every
    turn itself."""
    prob = Problem(cfg)
    out, dprob, _ = prob.run_dprob(flags=api.LAUNCH_SINGLE_CTA)
    out, dprob = out.clone(), dprob.clone()
    out_s, dprob_s = api.grouped_gemm_dprob_serial(prob.X, prob.W, prob.off, prob.G, prob.src, cfg.topk, prob.ws,
                                                   num_ctas=num_ctas)
    assert api.read_status(prob.ws) == 0
    assert torch.equal(out.view(torch.int16), out_s.view(torch.int16))
    assert torch.equal(dprob.view(torch.int32), dprob_s.view(torch.int32))


@pytest.mark.parametrize("name", ["latent", "imbal"])
def test_serialized_writers_full_size(name):
    prob = Problem(synth.CONFIGS[name])
    _, dprob, _ = prob.run_dprob()
    dprob = dprob.clone()
    for _ in range(2):
        _, dprob_s = api.grouped_gemm_dprob_serial(prob.X, prob.W, prob.off, prob.G, prob.src, prob.cfg.topk,
                                                   prob.ws)
        assert api.read_status(prob.ws) == 0
        assert torch.equal(dprob.view(torch.int32), dprob_s.view(torch.int32))


@pytest.mark.parametrize("flags", KERNELS, ids=KERNEL_IDS)
@pytest.mark.parametrize("cfg", LARGE, ids=[c.name for c in LARGE])
def test_large_dimensions(cfg, flags):
    prob = Problem(cfg)
    out, dprob, slots = prob.run_dprob(flags=flags)
    assert api.read_status(prob.ws) == 0
    off = prob.off.cpu().numpy()
    gpu_util.check_rows_against_oracle(prob, out, slots, dprob, gpu_util.sample_rows(off, 48, seed=cfg.seed))


@pytest.mark.parametrize("R,S", [(4096, 16), (4097, 16), (1803, 2), (2048, 5), (1000, 1)])
@pytest.mark.parametrize("aligned", [True, False], ids=["aligned", "offset_views"])
def test_combine_vector_and_general_forms(R, S, aligned):
    """The fixed-order combine is defined as an fp32 left-to-right sum over
    ascending slots, scattered through row_src.  Both kernel forms (four rows
    per thread with 16-byte loads when R % 4 == 0 and the buffers are 16-byte
    aligned; one row per thread otherwise, here forced by R % 4 != 0 or by
    views that start 4 bytes into their buffers) must give exactly those bits."""
    g = torch.Generator().manual_seed(R * 31 + S)
    sl_h = (torch.randn(S, R, generator=g) * torch.exp(torch.randn(S, R, generator=g) * 3)).float()
    src_h = torch.randperm(R, generator=g).to(torch.int32)
    if aligned:
        sl = sl_h.cuda()
        src = src_h.cuda()
    else:
        sl_buf = torch.empty(S * R + 1, dtype=torch.float32, device="cuda")
        sl = sl_buf[1:].view(S, R)
        sl.copy_(sl_h)
        src_buf = torch.empty(R + 1, dtype=torch.int32, device="cuda")
        src = src_buf[1:]
        src.copy_(src_h)
    dprob = api.dprob_combine(sl, src, 1)
    torch.cuda.synchronize()
    a = sl_h.numpy()
    acc = a[0].copy()
    for s in range(1, S):
        acc = (acc + a[s]).astype(np.float32)      # IEEE fp32 addition, round to nearest even
    want = np.empty(R, np.float32)
    want[src_h.numpy()] = acc
    got = dprob.reshape(-1).cpu().numpy()
    assert np.array_equal(got.view(np.int32), want.view(np.int32))


@pytest.mark.parametrize("name", ["latent", "imbal"])
def test_l2_reserve_changes_timing_only(name):
    """With grad_out's persisting-L2 set-aside in place (the setting the
    benchmark makes), the call's expert_out, slots and dprob equal the ones
    without it bit for bit; the set-aside is clamped to half of L2 and 0
    releases it."""
    prob = Problem(synth.CONFIGS[name])
    assert api.reserve_l2_persisting(0) == 0
    o1, d1, s1 = prob.run_dprob()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    want = min(prob.cfg.T * prob.cfg.N * 2, l2 // 2)
    slack = 4 << 20                        # the runtime rounds to its own granularity
    got = api.reserve_l2_persisting(prob.cfg.T * prob.cfg.N * 2)
    try:
        assert abs(got - want) <= slack
        assert api.reserve_l2_persisting(1 << 40) <= l2 // 2 + slack
        api.reserve_l2_persisting(got)
        o2, d2, s2 = prob.run_dprob()
        assert api.read_status(prob.ws) == 0
    finally:
        assert api.reserve_l2_persisting(0) == 0
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(s1.view(torch.int32), s2.view(torch.int32))
    assert torch.equal(d1.view(torch.int32), d2.view(torch.int32))
