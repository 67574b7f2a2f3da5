"""GPU routing indices vs the oracle: bit-exact (integer work)."""
import numpy as np
import pytest
import torch

import oracle
from bitwise_deterministic_moe_gb300 import api, synth
from tests import gpu_util

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gpu_util.ensure_built()


def run(ids_np, E):
    T, k = ids_np.shape
    ws = api.workspace(T, k, E)
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).cuda()
    off, src = api.permute_indices(ids, E, ws)
    st = api.read_status(ws)
    return off.cpu().numpy(), src.cpu().numpy(), st


@pytest.mark.parametrize("name", ["tiny", "small", "latent", "imbal", "stress"])
def test_configs_bit_exact(name):
    cfg = synth.CONFIGS[name]
    ids = synth.routing(cfg, np.random.default_rng(cfg.seed))
    off, src, st = run(ids, cfg.E)
    assert st == 0
    roff, rsrc = oracle.routing(ids, cfg.E)
    np.testing.assert_array_equal(off, roff)
    np.testing.assert_array_equal(src, rsrc)


@pytest.mark.parametrize("T,E,k,seed", [(1, 1, 1, 0), (3, 1024, 5, 1), (1000, 7, 3, 2), (4097, 33, 1, 3),
                                        (2049, 1024, 2, 4), (50, 3, 8, 5)])
def test_edge_shapes_bit_exact(T, E, k, seed):
    ids = np.random.default_rng(seed).integers(0, E, (T, k)).astype(np.int32)   # duplicates allowed
    off, src, st = run(ids, E)
    assert st == 0
    roff, rsrc = oracle.routing(ids, E)
    np.testing.assert_array_equal(off, roff)
    np.testing.assert_array_equal(src, rsrc)


def test_all_to_one_expert_and_empty():
    ids = np.full((3000, 2), 5, np.int32)
    off, src, st = run(ids, 9)
    roff, rsrc = oracle.routing(ids, 9)
    np.testing.assert_array_equal(off, roff)
    np.testing.assert_array_equal(src, rsrc)
    off, src, st = run(np.zeros((0, 4), np.int32), 6)
    assert st == 0 and off.tolist() == [0] * 7 and src.size == 0


def test_out_of_range_id_sets_routing_status():
    ids = np.zeros((100, 2), np.int32)
    ids[17, 1] = 8
    _, _, st = run(ids, 8)
    assert st == 3
    ids[17, 1] = -2
    _, _, st = run(ids, 8)
    assert st == 3


def test_repeated_calls_share_one_workspace():
    """The grid barrier words live in the workspace: calls of different sizes
    (different grids) back to back on one workspace stay consistent."""
    E = 64
    ws = api.workspace(20000, 6, E)
    rng = np.random.default_rng(11)
    for it in range(24):
        T = int(rng.integers(1, 20000))
        ids_np = rng.integers(0, E, (T, 6)).astype(np.int32)
        ids = torch.from_numpy(ids_np).cuda()
        off, src, row_of = api.permute_indices(ids, E, ws, with_row_of=True)
        roff, rsrc = oracle.routing(ids_np, E)
        np.testing.assert_array_equal(off.cpu().numpy(), roff)
        np.testing.assert_array_equal(src.cpu().numpy(), rsrc)
        np.testing.assert_array_equal(row_of.cpu().numpy(), oracle.inverse_rows(rsrc))
    assert api.read_status(ws) == 0
