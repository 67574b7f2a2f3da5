"""GPU chunk fingerprint vs the oracle: bit-exact (integer work)."""
import numpy as np
import pytest
import torch

import oracle
from bitwise_deterministic_moe_gb300 import api
from tests import gpu_util

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gpu_util.ensure_built()


@pytest.mark.parametrize("nbytes,chunk", [(0, 1 << 20), (1, 16), (3, 16), (17, 16), (4096, 1024), (100003, 4096),
                                          ((1 << 20) + 5, 1 << 20), (3 * (1 << 20) + 12, 1 << 20),
                                          (200000, 65536 * 3), (1 << 22, 1 << 22),
                                          ((40 << 20) + 7, 4096)])   # 10,241 chunks: every cluster loops
def test_positional_bit_exact(nbytes, chunk):
    data = np.random.default_rng(nbytes).integers(0, 256, nbytes, dtype=np.uint8)
    t = torch.from_numpy(data).cuda()
    got, hdr = api.fingerprint_host(t, chunk)
    want = oracle.fingerprint_chunks(data, chunk)
    assert got == [int(v) for v in want]
    assert hdr == oracle.header_hash(0, (nbytes,))


@pytest.mark.parametrize("offset", [1, 2, 3, 4, 8, 12])
def test_unaligned_views(offset):
    base = np.random.default_rng(offset).integers(0, 256, 70000 + offset, dtype=np.uint8)
    t = torch.from_numpy(base).cuda()[offset:]
    got, _ = api.fingerprint_host(t, 4096)
    assert got == [int(v) for v in oracle.fingerprint_chunks(base[offset:], 4096)]


@pytest.mark.parametrize("dtype,code", [(torch.bfloat16, 6), (torch.float32, 7), (torch.float16, 5),
                                        (torch.int32, 3), (torch.int64, 4), (torch.uint8, 0), (torch.int8, 1),
                                        (torch.float64, 8), (torch.int16, 2)])
def test_xor_mode_bit_exact(dtype, code):
    g = torch.Generator().manual_seed(code)
    if dtype.is_floating_point:
        t = torch.randn(30011, generator=g).to(dtype)
    elif dtype == torch.uint8:
        t = torch.randint(0, 256, (30011,), generator=g, dtype=torch.uint8)
    else:
        t = torch.randint(-30000, 30000, (30011,), generator=g).to(dtype)
    es = t.element_size()
    raw = t.view(torch.uint8).numpy() if es == 1 else t.view({2: torch.int16, 4: torch.int32, 8: torch.int64}[es]).numpy()
    got, hdr = api.fingerprint_host(t.cuda(), 4096, mode=1)
    assert got == [int(v) for v in oracle.xor_chunks(raw, code, 4096)]
    assert hdr == oracle.header_hash(code, (30011,))


def test_bf16_tensor_with_shape():
    x = torch.randn(37, 129, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    got, hdr = api.fingerprint_host(x.cuda(), 1024)
    raw = x.view(torch.int16).numpy().view(np.uint16)
    assert got == [int(v) for v in oracle.fingerprint_chunks(raw, 1024)]
    assert hdr == oracle.header_hash(6, (37, 129))


def test_single_bit_flip_changes_one_chunk():
    data = np.random.default_rng(9).integers(0, 256, 5 * 65536 + 3, dtype=np.uint8)
    t = torch.from_numpy(data).cuda()
    base, _ = api.fingerprint_host(t, 65536)
    t[3 * 65536 + 77] ^= 4
    new, _ = api.fingerprint_host(t, 65536)
    assert [i for i in range(len(base)) if base[i] != new[i]] == [3]
