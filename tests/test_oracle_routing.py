"""Pins for the oracle's deterministic routing permutation.

The order is fixed because routing maps are order-sensitive ("NVIDIA fait
passer le déterminisme bit à bit de Megatron Core à 2432 GPU ...", section
"Méthodologie de débogage du non-déterminisme"): experts ascending, and inside
an expert the flat routing index t*topk + j ascending.  Pinned against a
pure-Python double loop (brute force) and against the invariants that define
such a permutation.
"""
import numpy as np
import pytest

import oracle
from bitwise_deterministic_moe_gb300 import synth


def brute_force(topk_ids, E):
    flat = [int(v) for v in np.asarray(topk_ids).reshape(-1)]
    row_src, off = [], [0]
    for e in range(E):
        for i, v in enumerate(flat):
            if v == e:
                row_src.append(i)
        off.append(len(row_src))
    return np.array(off, dtype=np.int32), np.array(row_src, dtype=np.int32)


def check_invariants(topk_ids, E, off, row_src):
    eid = np.asarray(topk_ids).reshape(-1)
    R = eid.size
    assert off[0] == 0 and off[-1] == R
    assert np.all(np.diff(off) >= 0)
    assert sorted(row_src.tolist()) == list(range(R))          # a permutation
    for e in range(E):
        seg = row_src[off[e]:off[e + 1]]
        assert np.all(eid[seg] == e)
        assert np.all(np.diff(seg) > 0)                         # stable: ascending flat index


@pytest.mark.parametrize("name", ["tiny"])
def test_matches_brute_force_on_config(name):
    cfg = synth.CONFIGS[name]
    ids = synth.routing(cfg, np.random.default_rng(cfg.seed))
    off, row_src = oracle.routing(ids, cfg.E)
    boff, bsrc = brute_force(ids, cfg.E)
    np.testing.assert_array_equal(off, boff)
    np.testing.assert_array_equal(row_src, bsrc)
    check_invariants(ids, cfg.E, off, row_src)


@pytest.mark.parametrize("T,E,k,seed", [(1, 1, 1, 0), (7, 3, 2, 1), (33, 16, 4, 2), (100, 5, 5, 3), (257, 64, 6, 4)])
def test_random_shapes(T, E, k, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, (T, k)).astype(np.int32)      # duplicates allowed
    off, row_src = oracle.routing(ids, E)
    boff, bsrc = brute_force(ids, E)
    np.testing.assert_array_equal(off, boff)
    np.testing.assert_array_equal(row_src, bsrc)
    check_invariants(ids, E, off, row_src)


def test_empty_and_degenerate():
    off, row_src = oracle.routing(np.zeros((0, 4), np.int32), 8)
    assert off.tolist() == [0] * 9 and row_src.size == 0
    ids = np.full((5, 2), 3, np.int32)                      # everything to one expert
    off, row_src = oracle.routing(ids, 4)
    assert off.tolist() == [0, 0, 0, 0, 10, 10][:5]
    assert row_src.tolist() == list(range(10))


def test_out_of_range_ids_rejected():
    with pytest.raises(ValueError):
        oracle.routing(np.array([[0, 4]], np.int32), 4)
    with pytest.raises(ValueError):
        oracle.routing(np.array([[-1, 0]], np.int32), 4)


def test_planted_mistake_is_caught():
    """An unstable order inside an expert (a plausible bug) breaks the invariants."""
    rng = np.random.default_rng(5)
    ids = rng.integers(0, 4, (50, 3)).astype(np.int32)
    off, row_src = oracle.routing(ids, 4)
    bad = row_src.copy()
    bad[off[1]:off[2]] = bad[off[1]:off[2]][::-1]
    with pytest.raises(AssertionError):
        check_invariants(ids, 4, off, bad)
