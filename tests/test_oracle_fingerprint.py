"""Pins for the oracle's chunk-wise tensor fingerprint.

The pages ("NVIDIA fait passer le déterminisme bit à bit de Megatron Core à
2432 GPU ...", section "Méthodologie de débogage du non-déterminisme")
fingerprint tensors on the GPU with torch.hash_tensor, record shape, dtype and
element count, and hash order-sensitive data chunk by chunk.  The positional
mode is the library's own definition (see the oracle's header); it is pinned by the
published vectors of its two mixing functions, by a second, independent
pure-Python implementation, and by the properties a chunk fingerprint must
have.  The xor mode is pinned against the library routine torch.hash_tensor.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hash_vectors.txt")


def golden_vectors():
    out = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        kind, a, b = line.split()
        out.append((kind, int(a, 16), int(b, 16)))
    return out


@pytest.mark.parametrize("kind,x,want", golden_vectors())
def test_published_mixer_vectors(kind, x, want):
    if kind == "fmix32":
        assert int(oracle.fmix32(np.array([x], dtype=np.uint32))[0]) == want
    else:
        assert oracle.sm64(x) == want


# ---- a second implementation, written independently with Python integers ----
def _fmix32_int(h):
    h ^= h >> 16
    h = (h * 0x85EBCA6B) & 0xFFFFFFFF
    h ^= h >> 13
    h = (h * 0xC2B2AE35) & 0xFFFFFFFF
    h ^= h >> 16
    return h


def _sm64_int(z):
    M = (1 << 64) - 1
    z ^= z >> 30
    z = (z * 0xBF58476D1CE4E5B9) & M
    z ^= z >> 27
    z = (z * 0x94D049BB133111EB) & M
    return z ^ (z >> 31)


def slow_chunks(data: bytes, chunk: int):
    out = []
    for c in range((len(data) + chunk - 1) // chunk):
        seg = data[c * chunk:(c + 1) * chunk]
        acc = 0
        for k in range(0, len(seg), 4):
            word = int.from_bytes(seg[k:k + 4].ljust(4, b"\0"), "little")
            i = (c * chunk + k) // 4
            acc += _fmix32_int(word ^ ((i * 0x9E3779B9) & 0xFFFFFFFF))
        acc &= (1 << 64) - 1
        out.append(_sm64_int(acc ^ (c << 32) ^ len(seg)))
    return out


@pytest.mark.parametrize("nbytes,chunk", [(0, 64), (1, 64), (3, 16), (64, 64), (65, 64), (1000, 64),
                                          (4099, 1024), (5000, 16)])
def test_two_implementations_agree(nbytes, chunk):
    data = np.random.default_rng(nbytes).integers(0, 256, nbytes, dtype=np.uint8).tobytes()
    fast = oracle.fingerprint_chunks(data, chunk)
    assert [int(v) for v in fast] == slow_chunks(data, chunk)


def test_single_bit_flip_changes_exactly_one_chunk():
    rng = np.random.default_rng(1)
    data = bytearray(rng.integers(0, 256, 4096 + 13, dtype=np.uint8).tobytes())
    base = oracle.fingerprint_chunks(bytes(data), 256)
    for pos in rng.integers(0, len(data), 40):
        bit = int(rng.integers(8))
        data[pos] ^= 1 << bit
        new = oracle.fingerprint_chunks(bytes(data), 256)
        data[pos] ^= 1 << bit
        diff = np.nonzero(new != base)[0].tolist()
        assert diff == [pos // 256]


def test_word_swap_and_chunk_move_change_hash():
    rng = np.random.default_rng(2)
    w = rng.integers(0, 2 ** 32, 512, dtype=np.uint32)
    base = oracle.fingerprint_chunks(w.tobytes(), 1024)
    sw = w.copy()
    sw[[3, 77]] = sw[[77, 3]]
    assert oracle.fingerprint_chunks(sw.tobytes(), 1024)[0] != base[0]
    # identical content in a different chunk position hashes differently
    same = np.concatenate([w[:256], w[:256]])
    h = oracle.fingerprint_chunks(same.tobytes(), 1024)
    assert h[0] != h[1]


def test_header_records_dtype_shape_numel():
    h = oracle.header_hash(6, (4, 8))
    assert h != oracle.header_hash(7, (4, 8))
    assert h != oracle.header_hash(6, (8, 4))
    assert h != oracle.header_hash(6, (32,))
    assert h == oracle.header_hash(6, [4, 8])


@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "float16", "int32", "int64", "uint8", "int8", "float64"])
def test_xor_mode_matches_torch_hash_tensor(dtype):
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "hash_tensor"):
        pytest.skip("torch.hash_tensor not available")
    tdt = getattr(torch, dtype)
    g = torch.Generator().manual_seed(0)
    if tdt.is_floating_point:
        t = torch.randn(5000, generator=g).to(tdt)
    elif tdt == torch.uint8:
        t = torch.randint(0, 256, (5000,), generator=g, dtype=torch.uint8)
    else:
        t = torch.randint(-1000, 1000, (5000,), generator=g).to(tdt)
    es = t.element_size()
    chunk = 256 * 8
    code = oracle.DTYPE_CODES[dtype]
    raw = t.view(torch.uint8).numpy() if es == 1 else t.view({2: torch.int16, 4: torch.int32, 8: torch.int64}[es]).numpy()
    ours = oracle.xor_chunks(raw, code, chunk)
    per = chunk // es
    want = [int(torch.hash_tensor(t[i:i + per]).view(torch.int64).item()) & ((1 << 64) - 1)
            for i in range(0, t.numel(), per)]
    assert [int(v) for v in ours] == want
