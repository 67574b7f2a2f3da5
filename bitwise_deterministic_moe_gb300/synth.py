"""Seeded synthetic inputs for the routed-token grouped GEMM.

This module only draws random inputs; it holds none of the method's
arithmetic (no GEMM, no dot products, no hashing).  The GPU path and the CPU
oracle both take their inputs from here, so they see identical bytes.

Workload shapes follow the LatentMoE layer described on "Nemotron 3 Ultra 的
tech report: 550B 的 hybrid MoE 怎么训练、怎么 scale?" (concept list,
"LatentMoE": experts compute in a 2048-wide latent, 512 experts, top-22) and
the expert-imbalance figure in its "两次 divergence" table (MaxVio ~12 of a
512/22 bound).  Everything is host numpy (PCG64), seed = 1234 + config index.

Routing and logits come from one sequential Generator (routing first).  The
operands X_perm, W and grad_out are N(0,1)/sqrt(K) drawn in float32 from
independently seeded blocks (so they can be filled by several threads) and
rounded to bfloat16 (round-to-nearest-even on the float32 bit pattern); bf16
tensors are returned as uint16 bit patterns.
"""
from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import math
import os

import numpy as np


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int          # tokens
    E: int          # experts
    topk: int       # experts chosen per token
    K: int          # FFN intermediate (reduction) dim
    N: int          # latent (output) dim
    routing: str    # "uniform" | "zipf" | "maxvio"
    zipf_s: float = 1.1
    maxvio: float = 12.0
    zero_frac: float = 0.05
    index: int = 0

    @property
    def R(self) -> int:
        return self.T * self.topk

    @property
    def seed(self) -> int:
        return 1234 + self.index

    @property
    def S(self) -> int:
        """Number of 128-column private dprob slots per row."""
        return (self.N + 127) // 128


CONFIGS = {
    "tiny": MoEConfig("tiny", T=256, E=8, topk=2, K=128, N=256, routing="uniform", index=0),
    "small": MoEConfig("small", T=4096, E=64, topk=6, K=1024, N=2048, routing="uniform", index=1),
    "latent": MoEConfig("latent", T=8192, E=512, topk=22, K=1024, N=2048, routing="zipf", index=2),
    "imbal": MoEConfig("imbal", T=16384, E=512, topk=22, K=1024, N=2048, routing="maxvio", index=3),
    "stress": MoEConfig("stress", T=32768, E=512, topk=22, K=2048, N=2048, routing="zipf", index=4),
}


def custom_config(name, T, E, topk, K, N, routing="uniform", index=100, **kw) -> MoEConfig:
    """Extra parity shapes (ragged tails, odd sizes) that are not bench lines."""
    return MoEConfig(name, T=T, E=E, topk=topk, K=K, N=N, routing=routing, index=index, **kw)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest-even) and return the uint16 bit patterns.

    Input preparation only: finite inputs are assumed (normal draws)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


_BLOCK = 1 << 22   # elements per independently seeded block


def _normal_bf16(seed: int, tag: int, shape, scale: float) -> np.ndarray:
    """N(0,1)*scale drawn in float32 and rounded to bf16 bits.

    Block b of 2^22 elements is drawn from its own PCG64 stream seeded by
    SeedSequence(seed, spawn_key=(tag, b)), so the bytes do not depend on how
    many threads fill the blocks."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    nblocks = (n + _BLOCK - 1) // _BLOCK

    def fill(b):
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(tag, b))))
        m = min(_BLOCK, n - b * _BLOCK)
        v = g.standard_normal(m, dtype=np.float32)
        v *= np.float32(scale)
        out[b * _BLOCK:b * _BLOCK + m] = f32_to_bf16_bits(v)

    workers = min(nblocks, max(1, len(os.sched_getaffinity(0)))) if nblocks else 1
    if workers <= 1:
        for b in range(nblocks):
            fill(b)
    else:
        with cf.ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(nblocks)))
    return out.reshape(shape)


def _route_uniform(rng, T, E, k):
    keys = rng.random((T, E))
    ids = np.argpartition(keys, k - 1, axis=1)[:, :k]
    # order the k choices by key so that column j has a definite meaning
    order = np.argsort(np.take_along_axis(keys, ids, axis=1), axis=1, kind="stable")
    return np.take_along_axis(ids, order, axis=1).astype(np.int32)


def _route_zipf(rng, T, E, k, s):
    """Zipf(s) expert popularity, k distinct experts per token.

    Plackett-Luce sampling without replacement via Gumbel-top-k: key =
    log(rank^-s) + Gumbel.  Ranks go to experts through a seeded permutation
    so that the hot experts are not ids 0, 1, ..."""
    rank_of = rng.permutation(E) + 1
    logw = -s * np.log(rank_of.astype(np.float64))
    ids = np.empty((T, k), dtype=np.int32)
    step = 4096
    for t0 in range(0, T, step):
        t1 = min(T, t0 + step)
        g = rng.gumbel(size=(t1 - t0, E))
        key = logw[None, :] + g
        part = np.argpartition(-key, k - 1, axis=1)[:, :k]
        order = np.argsort(-np.take_along_axis(key, part, axis=1), axis=1, kind="stable")
        ids[t0:t1] = np.take_along_axis(part, order, axis=1)
    return ids


def _route_maxvio(rng, T, E, k, maxvio, zero_frac):
    """One hot expert with exactly maxvio x mean load, ~zero_frac of experts idle,
    every other choice uniform without replacement over the remaining experts."""
    perm = rng.permutation(E)
    hot = int(perm[0])
    n_zero = int(round(zero_frac * E))
    rest = perm[1 + n_zero:]
    mean = T * k / E
    n_hot = int(round(maxvio * mean))
    if n_hot > T:
        raise ValueError("maxvio too large for T")
    hot_tokens = np.zeros(T, dtype=bool)
    hot_tokens[rng.choice(T, size=n_hot, replace=False)] = True
    ids = np.empty((T, k), dtype=np.int32)
    keys = rng.random((T, rest.size))
    pick = np.argpartition(keys, k - 1, axis=1)[:, :k]
    order = np.argsort(np.take_along_axis(keys, pick, axis=1), axis=1, kind="stable")
    pick = np.take_along_axis(pick, order, axis=1)
    ids[:] = rest[pick]
    # hot tokens: the hot expert takes column 0, the other k-1 stay distinct
    ids[hot_tokens, 1:] = ids[hot_tokens, :k - 1]
    ids[hot_tokens, 0] = hot
    return ids


def routing(cfg: MoEConfig, rng: np.random.Generator) -> np.ndarray:
    if cfg.routing == "uniform":
        return _route_uniform(rng, cfg.T, cfg.E, cfg.topk)
    if cfg.routing == "zipf":
        return _route_zipf(rng, cfg.T, cfg.E, cfg.topk, cfg.zipf_s)
    if cfg.routing == "maxvio":
        return _route_maxvio(rng, cfg.T, cfg.E, cfg.topk, cfg.maxvio, cfg.zero_frac)
    raise ValueError(cfg.routing)


@dataclasses.dataclass
class MoEInputs:
    cfg: MoEConfig
    topk_ids: np.ndarray   # int32 [T, topk]
    X: np.ndarray          # uint16 (bf16 bits) [R, K], rows already in expert-permuted order
    W: np.ndarray          # uint16 (bf16 bits) [E, N, K]
    G: np.ndarray          # uint16 (bf16 bits) [T, N]  (grad_out)
    probs: np.ndarray      # float32 [T, topk] (finite-difference loss only)


def make_inputs(cfg: MoEConfig, with_weights: bool = True) -> MoEInputs:
    rng = np.random.default_rng(cfg.seed)
    ids = routing(cfg, rng)
    scale = 1.0 / math.sqrt(cfg.K)
    X = _normal_bf16(cfg.seed, 1, (cfg.R, cfg.K), scale)
    W = _normal_bf16(cfg.seed, 2, (cfg.E, cfg.N, cfg.K), scale) if with_weights else None
    G = _normal_bf16(cfg.seed, 3, (cfg.T, cfg.N), scale)
    logits = rng.standard_normal((cfg.T, cfg.topk), dtype=np.float32)
    z = np.exp(logits - logits.max(axis=1, keepdims=True))
    probs = (z / z.sum(axis=1, keepdims=True)).astype(np.float32)
    return MoEInputs(cfg, ids, X, W, G, probs)


def expert_loads(topk_ids: np.ndarray, E: int) -> np.ndarray:
    return np.bincount(topk_ids.reshape(-1), minlength=E)


def maxvio(topk_ids: np.ndarray, E: int) -> float:
    """Max expert load over mean load (the imbalance measure whose bound is E/topk)."""
    loads = expert_loads(topk_ids, E)
    return float(loads.max() / loads.mean())


def hidden_states(cfg: MoEConfig) -> np.ndarray:
    """Token hidden states in the latent dim, bf16 bits [T, N], N(0,1).

    Input of the dispatch gather that forms the expert rows; drawn from its
    own seeded blocks (tag 4), so it leaves every other input's bytes as they
    are."""
    return _normal_bf16(cfg.seed, 4, (cfg.T, cfg.N), 1.0)


def dyadic_probs(T: int, topk: int) -> np.ndarray:
    """Routing weights that are powers of two summing to exactly 1 per token
    (1/2, 1/4, ..., with the last two equal), float32 [T, topk]."""
    p = np.empty(topk, dtype=np.float64)
    for j in range(topk):
        p[j] = 2.0 ** -(j + 1)
    if topk > 1:
        p[-1] = p[-2]
    else:
        p[0] = 1.0
    return np.broadcast_to(p.astype(np.float32), (T, topk)).copy()
