"""Checks on the seeded input generator (not on the method): shapes, seeds and
the routing skew the workloads are meant to have.  The MaxVio bound E/topk =
512/22 = 23.27 is the one printed on "Nemotron 3 Ultra 的 tech report: 550B 的
hybrid MoE 怎么训练、怎么 scale?" ("两次 divergence" table notes), which holds
only for MaxVio = max load / mean load."""
import numpy as np
import pytest

from bitwise_deterministic_moe_gb300 import synth


def test_maxvio_bound_printed_on_page():
    assert round(512 / 22, 2) == 23.27


@pytest.mark.parametrize("name", ["tiny", "small", "latent", "imbal"])
def test_routing_is_distinct_and_in_range(name):
    cfg = synth.CONFIGS[name]
    ids = synth.routing(cfg, np.random.default_rng(cfg.seed))
    assert ids.shape == (cfg.T, cfg.topk) and ids.dtype == np.int32
    assert ids.min() >= 0 and ids.max() < cfg.E
    s = np.sort(ids, axis=1)
    assert np.all(s[:, 1:] != s[:, :-1])
    mv = synth.maxvio(ids, cfg.E)
    assert 1.0 <= mv <= cfg.E / cfg.topk + 1e-9


def test_imbalanced_config_hits_maxvio_12():
    cfg = synth.CONFIGS["imbal"]
    ids = synth.routing(cfg, np.random.default_rng(cfg.seed))
    loads = synth.expert_loads(ids, cfg.E)
    assert abs(synth.maxvio(ids, cfg.E) - 12.0) < 1e-9
    assert int((loads == 0).sum()) == 26


def test_zipf_config_is_skewed():
    cfg = synth.CONFIGS["latent"]
    ids = synth.routing(cfg, np.random.default_rng(cfg.seed))
    assert synth.maxvio(ids, cfg.E) > 12.0


def test_inputs_are_seeded_and_bf16():
    cfg = synth.CONFIGS["tiny"]
    a = synth.make_inputs(cfg)
    b = synth.make_inputs(cfg)
    for x, y in [(a.X, b.X), (a.W, b.W), (a.G, b.G), (a.topk_ids, b.topk_ids)]:
        np.testing.assert_array_equal(x, y)
    assert a.X.dtype == np.uint16 and a.X.shape == (cfg.R, cfg.K)
    assert a.W.shape == (cfg.E, cfg.N, cfg.K) and a.G.shape == (cfg.T, cfg.N)
    v = synth.bf16_bits_to_f32(a.X)
    assert abs(float(v.std()) * np.sqrt(cfg.K) - 1.0) < 0.05
