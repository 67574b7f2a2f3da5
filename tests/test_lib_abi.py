"""The C-ABI library builds for sm_103a, loads, and exports every entry point
include/dmoe.h declares.  Host-side argument validation is exercised with
calls that are rejected before any CUDA call is made (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

from bitwise_deterministic_moe_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dmoe.h")


@pytest.fixture(scope="module")
def lib():
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b((?:dmoe|moe)_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_binding_constants_match_the_header():
    """The binding's launch flags and limits are the header's #defines."""
    from bitwise_deterministic_moe_gb300 import api
    defines = dict(re.findall(r"^#define (DMOE_\w+) (\d+)", open(HEADER).read(), flags=re.M))
    pairs = {"DMOE_LAUNCH_TEST_STALL": api.LAUNCH_TEST_STALL, "DMOE_LAUNCH_SINGLE_CTA": api.LAUNCH_SINGLE_CTA,
             "DMOE_LAUNCH_CTA_PAIRS": api.LAUNCH_CTA_PAIRS, "DMOE_LAUNCH_NARROW_TILES": api.LAUNCH_NARROW_TILES,
             "DMOE_SLOT_COLS": api.SLOT_COLS, "DMOE_MAX_EXPERTS": api.MAX_EXPERTS}
    for name, value in pairs.items():
        assert int(defines[name]) == value, name
    flags = [v for k, v in pairs.items() if k.startswith("DMOE_LAUNCH_")]
    assert all(f & (f - 1) == 0 for f in flags) and len(set(flags)) == len(flags)   # distinct single bits


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ["moe_grouped_gemm_fwd", "moe_grouped_gemm_dprob", "moe_grouped_gemm_dprob_atomic",
                 "moe_dprob_epilogue", "moe_dprob_combine", "dmoe_permute_indices", "dmoe_fingerprint",
                 "dmoe_read_status", "dmoe_workspace_bytes", "moe_dispatch_gather", "moe_token_combine",
                 "moe_grouped_gemm_wgrad", "moe_grouped_gemm_dprob_serial", "dmoe_quantize_mxfp8",
                 "dmoe_quantize_nvfp4"]:
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_sizes(lib):
    lib.dmoe_status_string.restype = ctypes.c_char_p
    assert lib.dmoe_status_string(0) == b"ok"
    assert b"routing" in lib.dmoe_status_string(3)
    lib.dmoe_workspace_bytes.restype = ctypes.c_size_t
    # status region + per-expert counts of ceil(R/1024) blocks + totals, rounded to 256
    assert lib.dmoe_workspace_bytes(8192, 22, 512) == 256 + ((512 * 176 * 4 + 512 * 4 + 255) // 256) * 256
    assert lib.dmoe_workspace_bytes(0, 4, 8) == 256 + 256
    lib.dmoe_fingerprint_num_chunks.restype = ctypes.c_size_t
    lib.dmoe_fingerprint_num_chunks.argtypes = [ctypes.c_size_t, ctypes.c_size_t]
    assert lib.dmoe_fingerprint_num_chunks(0, 1 << 20) == 0
    assert lib.dmoe_fingerprint_num_chunks((1 << 20) + 1, 1 << 20) == 2


def test_invalid_arguments_rejected_on_host(lib):
    P, I, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    f = lib.moe_grouped_gemm_fwd
    f.argtypes = [P, P, P, I, I, I, I, P, P, P, SZ, P]
    f.restype = I
    # null operands -> DMOE_ERR_INVALID_ARG (1)
    assert f(None, None, None, 16, 2, 64, 256, None, None, None, 0, None) == 1
    # misaligned pointers -> invalid argument
    assert f(8, 16, 16, 16, 2, 64, 256, 16, None, 16, 4096, None) == 1
    # N not a multiple of 128 -> DMOE_ERR_UNSUPPORTED (2); too many experts too
    assert f(16, 16, 16, 16, 2, 64, 200, 16, None, 16, 4096, None) == 2
    assert f(16, 16, 16, 16, 2000, 64, 256, 16, None, 16, 4096, None) == 2
    # K not a multiple of 8 -> unsupported
    assert f(16, 16, 16, 16, 2, 60, 256, 16, None, 16, 4096, None) == 2
    # missing workspace -> DMOE_ERR_WORKSPACE (6)
    assert f(16, 16, 16, 16, 2, 64, 256, 16, None, None, 0, None) == 6
    g = lib.moe_grouped_gemm_dprob
    g.argtypes = [P, P, P, I, I, I, I, P, P, P, I, I, P, P, P, P, SZ, P]
    g.restype = I
    # R != T * topk -> invalid argument
    assert g(16, 16, 16, 10, 2, 64, 256, 16, 16, 16, 3, 4, 16, 16, None, 16, 4096, None) == 1
    p = lib.dmoe_permute_indices
    p.argtypes = [P, I, I, I, P, P, P, P, SZ, P]
    p.restype = I
    assert p(16, 4, 2, 0, 16, 16, None, 16, 4096, None) == 1          # E = 0
    assert p(16, 4, 2, 4096, 16, 16, None, 16, 4096, None) == 2       # E > 1024
    assert p(16, 4, 2, 8, 16, 16, 16, 16, 8, None) == 6               # workspace too small
    d = lib.moe_dispatch_gather
    d.argtypes = [P, P, I, I, I, P, P, SZ, P]
    d.restype = I
    assert d(16, 16, 4, 2, 12, 16, None, 0, None) == 2       # H not a multiple of 8
    assert d(8, 16, 4, 2, 16, 16, None, 0, None) == 1        # misaligned hidden
    assert d(None, 16, 4, 2, 16, 16, None, 0, None) == 1     # null hidden
    assert d(16, 16, 4, 2, 16, 16, 16, 8, None) == 6         # workspace below the status region
    assert d(None, None, 0, 2, 16, None, None, 0, None) == 0  # no tokens: nothing to launch
    c = lib.moe_token_combine
    c.argtypes = [P, P, P, I, I, I, P, P, SZ, P]
    c.restype = I
    assert c(16, 16, 16, 4, 65, 16, 16, None, 0, None) == 2   # topk above the combine's limit
    assert c(16, 16, 16, 4, 2, 20, 16, None, 0, None) == 2    # N not a multiple of 8
    assert c(16, 16, 16, 4, 0, 16, 16, None, 0, None) == 1    # topk = 0
    assert c(16, 16, 16, 4, 2, 16, 24, None, 0, None) == 1    # misaligned y
    assert c(None, None, None, 0, 2, 16, None, None, 0, None) == 0
    q = lib.dmoe_quantize_mxfp8
    q.argtypes = [P, I, I, P, P, P]
    q.restype = I
    assert q(16, 4, 48, 16, 16, None) == 2        # cols not a multiple of 32
    assert q(8, 4, 64, 16, 16, None) == 1         # misaligned input
    assert q(None, 0, 64, None, None, None) == 0  # empty: nothing to launch
    v = lib.dmoe_quantize_nvfp4
    v.argtypes = [P, I, I, P, P, P, P, SZ, P]
    v.restype = I
    assert v(16, 4, 24, 16, 16, 16, 16, 4096, None) == 2     # cols not a multiple of 16
    assert v(16, 4, 32, 16, 16, None, 16, 4096, None) == 1   # no tensor-scale output
    assert v(16, 4, 32, 16, 16, 16, 16, 200, None) == 6      # workspace below status + scratch
    fp = lib.dmoe_fingerprint
    fp.argtypes = [P, SZ, I, I, ctypes.POINTER(ctypes.c_int64), SZ, I, P, ctypes.POINTER(ctypes.c_uint64), P]
    fp.restype = I
    shape = (ctypes.c_int64 * 1)(10)
    h = ctypes.c_uint64()
    assert fp(16, 10, 0, 1, shape, 100, 0, 16, ctypes.byref(h), None) == 1   # chunk not a multiple of 16
    assert fp(16, 11, 0, 1, shape, 64, 0, 16, ctypes.byref(h), None) == 1    # nbytes != numel * size


def test_header_hash_matches_oracle_without_gpu(lib):
    """An empty tensor makes no device call, so its header can be checked here."""
    import oracle
    P, I, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    fp = lib.dmoe_fingerprint
    fp.argtypes = [P, SZ, I, I, ctypes.POINTER(ctypes.c_int64), SZ, I, P, ctypes.POINTER(ctypes.c_uint64), P]
    fp.restype = I
    for code, shape in [(6, (0, 4)), (7, (3, 0, 5)), (0, (0,))]:
        arr = (ctypes.c_int64 * len(shape))(*shape)
        h = ctypes.c_uint64()
        assert fp(None, 0, code, len(shape), arr, 1 << 20, 0, None, ctypes.byref(h), None) == 0
        assert h.value == oracle.header_hash(code, shape)


def test_header_is_c99_and_the_library_links_from_c(lib, tmp_path):
    """A plain C99 program includes the header (-std=c99 -pedantic -Werror),
    links libdmoe.so and calls the entry points that need no GPU."""
    here = os.path.dirname(os.path.abspath(__file__))
    libdir = os.path.dirname(build.LIB)
    exe = str(tmp_path / "abi_consumer")
    subprocess.run(["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
                    "-I", os.path.join(build.ROOT, "include"), os.path.join(here, "c", "abi_consumer.c"),
                    "-L", libdir, "-ldmoe", "-Wl,-rpath," + libdir, "-o", exe], check=True)
    res = subprocess.run([exe], capture_output=True, text=True, check=True)
    assert res.stdout.strip() == "ok"
