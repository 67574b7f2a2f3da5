"""CPU oracle for the bitwise-deterministic routed-token grouped GEMM.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline / reference legs may import this package.  The product library
(``bitwise_deterministic_moe_gb300``) never imports it, and this package never
imports the product library: the two share no code, tables or constants.

Contents and the passage each part follows:

* ``routing`` -- the deterministic permutation of routed (token, choice)
  entries into expert-contiguous rows.  Routing maps are order-sensitive data
  ("NVIDIA fait passer le déterminisme bit à bit de Megatron Core à 2432 GPU
  ...", section "Méthodologie de débogage du non-déterminisme"), so the order
  is fixed: experts ascending, and inside an expert the flat index t*topk + j
  ascending.  Plain definition: a stable sort by expert id (numpy's stable
  argsort) and a bincount prefix.
* ``expert_rows`` -- grouped GEMM, bf16 rounding, private-slot partials and
  dprob, in binary64 (C, ``dmoe_oracle.c``), following "Trillion-Parameter
  Pretraining Goes Bitwise-Deterministic: NVIDIA Cuts the Determinism Tax to
  About 2%", section "Interpretation".
* ``combine`` -- dprob[t, j] from the per-row values: a scatter through
  row_src (the fixed-order slot combine reaches the plain dot product).
* ``inverse_rows``, ``dispatch``, ``token_combine`` -- the steps either side
  of the grouped GEMM: the gather that forms the expert-permuted rows from the
  token hidden states, and the routing-probability-weighted combine of each
  token's expert outputs.  Both are plain definitions (an index copy; a sum
  over the token's choices in ascending j, binary64, then one rounding to
  bf16).  The pages treat routing maps and dispatch outputs as order-sensitive
  data to fingerprint ("NVIDIA fait passer ...", section "Méthodologie de
  débogage du non-déterminisme"), and dprob is the derivative of this combine
  with respect to the routing probability.
* ``wgrad_entries`` / ``wgrad_expert`` -- the grouped GEMM's weight gradient
  dW[e] = dY_e^T X_e over the expert's rows (binary64, rows ascending).  A
  weight-gradient path is one of the three workloads whose determinism
  overhead the pages measure ("Trillion-Parameter Pretraining ...", section
  "Synopsis"; "NVIDIA fait passer ...", section "Optimisation pour le
  Nemotron à mille milliards de paramètres").
* ``mxfp8_quantize`` / ``nvfp4_quantize`` -- the block-scaled encodings whose
  encoded values and scale buffers the pages fingerprint ("NVIDIA fait passer
  ...", section "Méthodologie de débogage du non-déterminisme"); E4M3, E2M1
  and E8M0 decoded and encoded from their format definitions.
* ``mxfp8_decode`` / ``nvfp4_decode`` / ``block_scaled_rows`` -- the expert
  GEMM on block-scaled operands: each operand decoded to binary64 from its
  codes and scales by the format definitions, then the same grouped GEMM,
  bf16 rounding, private-slot partials and dprob as ``expert_rows``
  ("NVIDIA fait passer ...", section "Méthodologie de débogage du
  non-déterminisme", for MXFP8 / NVFP4 operands in the fingerprinted path;
  "Nemotron 3 Ultra 的 tech report ...", NVFP4 pretraining section, for NVFP4
  GEMMs; "Trillion-Parameter Pretraining ...", section "Interpretation", for
  the slots).  The GEMM step is a binary64 matrix product (a library
  primitive).
* ``fingerprint`` -- chunk-wise tensor fingerprint with a header over dtype,
  shape and numel (same French page, section "Méthodologie de débogage du
  non-déterminisme": fingerprints computed on the GPU with shape, dtype and
  element count recorded; chunk-wise for order-sensitive data).  Mode
  "positional" hashes raw bits with position mixing; mode "xor" reduces each
  chunk the way ``torch.hash_tensor`` reduces a tensor.

The hash is the library's own definition (the pages name only the
``torch.hash_tensor`` xor reduction):
    fmix32  -- MurmurHash3's 32-bit finalizer (A. Appleby, public domain)
    sm64    -- the splitmix64 output function (Steele, Lea, Flood 2014)
    chunk c, words w_i (little-endian uint32, global word index i, zero-padded tail):
        acc_c = sum_i fmix32(w_i ^ (i * 0x9E3779B9 mod 2^32))  mod 2^64
        h_c   = sm64(acc_c ^ (c << 32) ^ chunk_len_bytes)
    header: h = sm64(dtype_code); then h = sm64(h ^ v) for v in
        (ndim, shape..., numel, nbytes)
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dmoe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libdmoe_oracle.so")
SLOT_WIDTH = 128   # columns per private dprob slot

MASK64 = (1 << 64) - 1
MASK32 = (1 << 32) - 1
GOLDEN32 = 0x9E3779B9

# dtype codes recorded in the fingerprint header (the library's ABI uses the
# same numbering; it is an interface, written out separately on each side)
DTYPE_CODES = {
    "uint8": 0, "int8": 1, "int16": 2, "int32": 3, "int64": 4,
    "float16": 5, "bfloat16": 6, "float32": 7, "float64": 8, "bool": 9,
    "uint16": 10, "uint32": 11, "uint64": 12,
}

_lib = None


def build(force: bool = False) -> str:
    """Compile the C part of the oracle (gcc, -O2, no FP contraction, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        ci = ctypes.c_int
        lib.oracle_bf16_rne.argtypes = [ctypes.c_double]
        lib.oracle_bf16_rne.restype = ctypes.c_uint16
        lib.oracle_bf16_rne_array.argtypes = [P, i64, P]
        lib.oracle_bf16_rne_array.restype = None
        lib.oracle_expert_rows.argtypes = [P, P, P, P, P, i64, ci, ci, ci, ci, P, i64, ci, P, P, P, P]
        lib.oracle_expert_rows.restype = ci
        lib.oracle_dprob_from_output.argtypes = [P, P, P, i64, ci, ci, P, i64, ci, P, P]
        lib.oracle_dprob_from_output.restype = None
        lib.oracle_wgrad_entries.argtypes = [P, P, P, ci, ci, ci, P, i64, P]
        lib.oracle_wgrad_entries.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ci
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


# --------------------------------------------------------------------------
# bf16 helpers (the oracle's own)
# --------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> binary64 values (bf16 = upper half of a binary32)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_rne(x) -> np.ndarray:
    """binary64 -> bf16 bits, round to nearest even, from the IEEE rule (C)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_bf16_rne_array(_ptr(x), x.size, _ptr(out))
    return out


# --------------------------------------------------------------------------
# routing
# --------------------------------------------------------------------------
def routing(topk_ids: np.ndarray, E: int):
    """Deterministic permutation of routed entries into expert-contiguous rows.

    Returns (expert_offsets int32 [E+1], row_src int32 [R]) where rows
    [off[e], off[e+1]) belong to expert e and row_src[r] is the flat routing
    index t*topk + j of permuted row r (ascending within each expert)."""
    eid = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    if eid.size and (eid.min() < 0 or eid.max() >= E):
        raise ValueError("expert id out of range")
    row_src = np.argsort(eid, kind="stable").astype(np.int32)
    counts = np.bincount(eid, minlength=E)
    off = np.zeros(E + 1, dtype=np.int64)
    np.cumsum(counts, out=off[1:])
    return off.astype(np.int32), row_src


# --------------------------------------------------------------------------
# grouped GEMM, slots, dprob (binary64, C)
# --------------------------------------------------------------------------
def expert_rows(X, W, off, rows, G=None, row_src=None, topk=1, want_Y=True, want_Yb=True,
                want_P=False, want_D=False, slot_width=SLOT_WIDTH):
    """Compute Y (binary64), Yb (bf16 bits), P [nrows,S] and D [nrows] for the
    requested permuted rows.  X [R,K], W [E,N,K], G [T,N] are bf16 bit arrays."""
    X = np.ascontiguousarray(X, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    off = np.ascontiguousarray(off, dtype=np.int32)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    R, K = X.shape
    E, N, K2 = W.shape
    assert K2 == K and off.shape == (E + 1,)
    S = (N + slot_width - 1) // slot_width
    n = rows.size
    Y = np.empty((n, N), np.float64) if want_Y else None
    Yb = np.empty((n, N), np.uint16) if (want_Yb or want_D) else None
    P = np.empty((n, S), np.float64) if want_P else None
    D = np.empty((n,), np.float64) if want_D else None
    if want_P or want_D:
        G = np.ascontiguousarray(G, dtype=np.uint16)
        row_src = np.ascontiguousarray(row_src, dtype=np.int32)
    else:
        G = None
        row_src = None
    rc = _load().oracle_expert_rows(_ptr(X), _ptr(W), _ptr(G), _ptr(off), _ptr(row_src),
                                    R, E, K, N, int(topk), _ptr(rows), n, slot_width,
                                    _ptr(Y), _ptr(Yb), _ptr(P), _ptr(D))
    if rc != 0:
        raise ValueError("a requested row is not covered by any expert")
    return Y, Yb, P, D


def dprob_from_output(G, expert_out, row_src, topk, rows=None, slot_width=SLOT_WIDTH):
    """Slot partials P [nrows,S] and dots D [nrows] from a stored bf16 expert_out."""
    G = np.ascontiguousarray(G, dtype=np.uint16)
    Yb = np.ascontiguousarray(expert_out, dtype=np.uint16)
    row_src = np.ascontiguousarray(row_src, dtype=np.int32)
    R, N = Yb.shape
    if rows is None:
        rows = np.arange(R, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    S = (N + slot_width - 1) // slot_width
    P = np.empty((rows.size, S), np.float64)
    D = np.empty((rows.size,), np.float64)
    _load().oracle_dprob_from_output(_ptr(G), _ptr(Yb), _ptr(row_src), R, N, int(topk),
                                     _ptr(rows), rows.size, slot_width, _ptr(P), _ptr(D))
    return P, D


def combine(D_rows, row_src, T, topk, rows=None):
    """dprob [T, topk] (binary64) from per-row dots: dprob[row_src[r]] = D[r].
    Entries of rows not requested are NaN."""
    out = np.full(T * topk, np.nan, dtype=np.float64)
    row_src = np.asarray(row_src)
    if rows is None:
        out[row_src] = D_rows
    else:
        out[row_src[np.asarray(rows)]] = D_rows
    return out.reshape(T, topk)


def full(inputs, slot_width=SLOT_WIDTH):
    """Everything for a whole (small) problem: routing, Yb, P, dprob."""
    cfg = inputs.cfg
    off, row_src = routing(inputs.topk_ids, cfg.E)
    rows = np.arange(cfg.R, dtype=np.int64)
    Y, Yb, P, D = expert_rows(inputs.X, inputs.W, off, rows, G=inputs.G, row_src=row_src,
                              topk=cfg.topk, want_Y=True, want_Yb=True, want_P=True, want_D=True,
                              slot_width=slot_width)
    dprob = combine(D, row_src, cfg.T, cfg.topk)
    return dict(off=off, row_src=row_src, Y=Y, Yb=Yb, P=P, D=D, dprob=dprob)


# --------------------------------------------------------------------------
# weight gradient of the grouped GEMM
# --------------------------------------------------------------------------
def wgrad_entries(X, dY, off, entries):
    """dW[e, n, c] = sum over the expert's rows r (ascending) of dY[r, n] * X[r, c],
    binary64 (C), for each (e, n, c) row of `entries` [m, 3]."""
    X = np.ascontiguousarray(X, dtype=np.uint16)
    dY = np.ascontiguousarray(dY, dtype=np.uint16)
    off = np.ascontiguousarray(off, dtype=np.int32)
    ent = np.ascontiguousarray(entries, dtype=np.int64).reshape(-1, 3)
    R, K = X.shape
    R2, N = dY.shape
    E = off.size - 1
    assert R2 == R and int(off[-1]) == R
    if ent.size and (ent[:, 0].min() < 0 or ent[:, 0].max() >= E or ent[:, 1].max() >= N or ent[:, 2].max() >= K):
        raise ValueError("entry out of range")
    out = np.empty(ent.shape[0], dtype=np.float64)
    _load().oracle_wgrad_entries(_ptr(X), _ptr(dY), _ptr(off), E, K, N, _ptr(ent), ent.shape[0], _ptr(out))
    return out


def wgrad_expert(X, dY, off, e):
    """The whole dW[e] [N, K] (binary64) by the same definition."""
    N, K = np.asarray(dY).shape[1], np.asarray(X).shape[1]
    n, c = np.meshgrid(np.arange(N), np.arange(K), indexing="ij")
    ent = np.stack([np.full(N * K, e), n.ravel(), c.ravel()], axis=1)
    return wgrad_entries(X, dY, off, ent).reshape(N, K)


# --------------------------------------------------------------------------
# dispatch gather and token combine
# --------------------------------------------------------------------------
def inverse_rows(row_src) -> np.ndarray:
    """row_of [R] int32 with row_src[row_of[f]] = f: the permuted row that holds
    flat routing index f = t*topk + j.  row_src must be a permutation of [0,R)."""
    row_src = np.asarray(row_src, dtype=np.int64).reshape(-1)
    R = row_src.size
    if R and not np.array_equal(np.sort(row_src), np.arange(R)):
        raise ValueError("row_src is not a permutation")
    row_of = np.empty(R, dtype=np.int32)
    row_of[row_src] = np.arange(R, dtype=np.int32)
    return row_of


def dispatch(hidden, row_src, topk: int) -> np.ndarray:
    """X_perm[r, :] = hidden[row_src[r] // topk, :]: the token's hidden state
    copied (bf16 bits, unchanged) to every permuted row it was routed to."""
    hidden = np.asarray(hidden, dtype=np.uint16)
    tok = np.asarray(row_src, dtype=np.int64).reshape(-1) // topk
    return hidden[tok]


def token_combine(expert_out, probs, row_src, tokens=None):
    """y[t, n] = sum over j = 0..topk-1 (ascending) of
    prob[t, j] * expert_out[row_of[t*topk + j], n], in binary64 (each product of
    a float32 and a bf16 is exact there), and its bf16 rounding.

    Returns (y binary64 [ntok, N], y bf16 bits [ntok, N]) for the requested
    tokens (all when None)."""
    Yb = np.asarray(expert_out, dtype=np.uint16)
    probs = np.asarray(probs, dtype=np.float32)
    T, topk = probs.shape
    row_of = inverse_rows(row_src).reshape(T, topk)
    tokens = np.arange(T, dtype=np.int64) if tokens is None else np.asarray(tokens, dtype=np.int64)
    acc = np.zeros((tokens.size, Yb.shape[1]), dtype=np.float64)
    for j in range(topk):
        acc += probs[tokens, j].astype(np.float64)[:, None] * bf16_to_f64(Yb[row_of[tokens, j]])
    return acc, bf16_rne(acc)


# --------------------------------------------------------------------------
# block-scaled low-precision encodings (MXFP8, NVFP4)
# --------------------------------------------------------------------------
def e4m3_value(code) -> np.ndarray:
    """binary64 value of FP8 E4M3 codes (1 sign, 4 exponent bits with bias 7,
    3 fraction bits; exponent field 0 is subnormal, m/8 * 2^-6; S.1111.111 is
    NaN; no infinities; largest finite 1.75 * 2^8 = 448)."""
    c = np.asarray(code, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


def e2m1_value(code) -> np.ndarray:
    """binary64 value of FP4 E2M1 codes (1 sign, 2 exponent bits with bias 1,
    1 fraction bit): 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives."""
    c = np.asarray(code, dtype=np.int64)
    sign = np.where(c & 0x8, -1.0, 1.0)
    e = (c >> 1) & 0x3
    m = c & 0x1
    mag = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(e - 1.0))
    return sign * mag


def _encode_rne_sat(x, codes_pos, values_pos, sign_bit):
    """Nearest representable value (ties to the even code), magnitudes above
    the largest finite value saturate to it; the sign is kept (-0 stays -0).
    codes_pos / values_pos: the non-negative finite codes, values ascending."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    idx = np.searchsorted(values_pos, a, side="right") - 1           # largest value <= a
    idx = np.clip(idx, 0, len(values_pos) - 1)
    hi = np.clip(idx + 1, 0, len(values_pos) - 1)
    lo_v, hi_v = values_pos[idx], values_pos[hi]
    d_lo, d_hi = a - lo_v, hi_v - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (codes_pos[hi] % 2 == 0) & (hi != idx))
    code = np.where(pick_hi, codes_pos[hi], codes_pos[idx])
    code = np.where(a >= values_pos[-1], codes_pos[-1], code)           # saturate
    neg = np.signbit(x)
    return (code | np.where(neg, sign_bit, 0)).astype(np.uint8)


_E4M3_CODES = np.arange(0x7F, dtype=np.int64)                            # 0x00..0x7E: non-negative finite
_E4M3_VALS = e4m3_value(_E4M3_CODES)
_E2M1_CODES = np.arange(8, dtype=np.int64)
_E2M1_VALS = e2m1_value(_E2M1_CODES)


def e4m3_encode(x) -> np.ndarray:
    """binary64 -> E4M3 code, round to nearest even, saturating at +-448."""
    return _encode_rne_sat(x, _E4M3_CODES, _E4M3_VALS, 0x80)


def e2m1_encode(x) -> np.ndarray:
    """binary64 -> E2M1 code (low 4 bits), round to nearest even, saturating at +-6."""
    return _encode_rne_sat(x, _E2M1_CODES, _E2M1_VALS, 0x8)


MX_BLOCK = 32
NV_BLOCK = 16


def mxfp8_quantize(x_bits):
    """MXFP8 (OCP Microscaling Formats v1.0): each run of 32 consecutive values
    of a row shares one E8M0 scale X = 2^s with s = floor(log2(amax)) - 8 (8 =
    the E4M3 maximum exponent), clamped to s >= -127; the elements are E4M3
    codes of V/X (round to nearest even, saturating).  An all-zero block gets
    s = -127.  A block holding a NaN or an infinity gets scale 0xFF (NaN) and
    NaN elements (0x7F).
    x_bits: bf16 bit patterns [rows, cols], cols % 32 == 0.
    Returns (values uint8 [rows, cols], scales uint8 [rows, cols/32])."""
    x = bf16_to_f64(x_bits)
    rows, cols = x.shape
    assert cols % MX_BLOCK == 0
    blk = x.reshape(rows, cols // MX_BLOCK, MX_BLOCK)
    finite = np.isfinite(blk).all(axis=2)
    amax = np.where(finite, np.abs(np.where(np.isfinite(blk), blk, 0.0)).max(axis=2), 0.0)
    _, ex = np.frexp(amax)                           # amax = f * 2^ex, f in [0.5, 1)
    s = np.where(amax > 0, ex - 1 - 8, -127)
    s = np.maximum(s, -127)
    scales = np.where(finite, s + 127, 0xFF).astype(np.uint8)
    scaled = np.where(finite[..., None], blk * np.exp2(-s.astype(np.float64))[..., None], 0.0)
    vals = e4m3_encode(scaled)
    vals = np.where(finite[..., None], vals, np.uint8(0x7F)).astype(np.uint8)
    return vals.reshape(rows, cols), scales


def nvfp4_quantize(x_bits, amax=None):
    """NVFP4 with two-level scaling, every step in binary32 in this order:
      amax_t   = max |x| over the tensor (finite inputs)
      S_enc    = 2688 / amax_t  (2688 = 448 * 6; 1 when amax_t == 0)
      per run of 16 consecutive values of a row:
        amax_b  = max |x| over the block
        s_b     = E4M3( (amax_b / 6) * S_enc )      round to nearest even, saturating
        q_i     = E2M1( (x_i * S_enc) / value(s_b) )  (q_i = 0 when s_b encodes 0)
    Two E2M1 codes per byte, element 2i in the low nibble.
    x_bits: bf16 bit patterns [rows, cols], cols % 16 == 0.  amax: the tensor
    maximum when x_bits holds only some rows of the tensor.
    Returns (packed uint8 [rows, cols/2], scales uint8 [rows, cols/16], S_enc float32)."""
    x32 = bf16_to_f64(x_bits).astype(np.float32)
    rows, cols = x32.shape
    assert cols % NV_BLOCK == 0
    if amax is not None:
        amax_t = np.float32(amax)
    else:
        amax_t = np.float32(np.abs(x32).max()) if x32.size else np.float32(0)
    s_enc = np.float32(1.0) if amax_t == 0 else np.float32(np.float32(2688.0) / amax_t)
    blk = x32.reshape(rows, cols // NV_BLOCK, NV_BLOCK)
    amax_b = np.abs(blk).max(axis=2)
    dec = (amax_b / np.float32(6.0)).astype(np.float32)
    dec = (dec * s_enc).astype(np.float32)
    scales = e4m3_encode(dec.astype(np.float64))
    sv = e4m3_value(scales).astype(np.float32)
    t = (blk * s_enc).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (t / sv[..., None]).astype(np.float32)
    r = np.where(sv[..., None] == 0, np.float32(0), r)
    q = e2m1_encode(r.astype(np.float64)).reshape(rows, cols)
    packed = (q[:, 0::2] & 0xF) | ((q[:, 1::2] & 0xF) << 4)
    return packed.astype(np.uint8), scales, s_enc


def mxfp8_decode(codes, scales) -> np.ndarray:
    """binary64 values of an MXFP8 tensor: E4M3(code) * 2^(scale - 127) for each
    run of 32 consecutive values of a row sharing one E8M0 scale byte (OCP
    Microscaling Formats v1.0; scale 0xFF encodes NaN).
    codes uint8 [rows, cols], scales uint8 [rows, cols/32]."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    rows, cols = codes.shape
    assert scales.shape == (rows, cols // MX_BLOCK)
    sc = np.where(scales == 0xFF, np.nan, np.exp2(scales.astype(np.float64) - 127.0))
    v = e4m3_value(codes).reshape(rows, cols // MX_BLOCK, MX_BLOCK) * sc[..., None]
    return v.reshape(rows, cols)


def nvfp4_decode(packed, scales, s_enc) -> np.ndarray:
    """binary64 values of an NVFP4 tensor: E2M1(code) * E4M3(scale) / S_enc,
    one E4M3 scale per run of 16 consecutive values of a row, S_enc the
    tensor's fp32 encode scale; two codes per byte, element 2i in the low nibble.
    packed uint8 [rows, cols/2], scales uint8 [rows, cols/16]."""
    packed = np.asarray(packed, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    rows, half = packed.shape
    cols = 2 * half
    assert scales.shape == (rows, cols // NV_BLOCK)
    codes = np.empty((rows, cols), dtype=np.uint8)
    codes[:, 0::2] = packed & 0xF
    codes[:, 1::2] = packed >> 4
    v = e2m1_value(codes).reshape(rows, cols // NV_BLOCK, NV_BLOCK) * e4m3_value(scales)[..., None]
    return v.reshape(rows, cols) / float(np.float32(s_enc))


def block_scaled_rows(Xd, W_decoded, off, rows, G=None, row_src=None, topk=1, slot_width=SLOT_WIDTH):
    """The grouped GEMM on decoded operands for the requested permuted rows:
    Y[i, n] = sum_c Xd[rows[i], c] * Wd[e][n, c] in binary64 (e = the expert whose
    range holds rows[i]; Wd[e] = W_decoded(e), [N, K] binary64), Yb = bf16_rne(Y),
    and, when G is given, the slot partials P [nrows, S] and dots D [nrows] of the
    stored Yb exactly as for bf16 operands.  Returns (Y, Yb, P, D)."""
    Xd = np.asarray(Xd, dtype=np.float64)
    off = np.asarray(off, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= off[-1]):
        raise ValueError("a requested row is not covered by any expert")
    experts = np.searchsorted(off, rows, side="right") - 1
    Y = None
    for e in np.unique(experts):
        sel = np.where(experts == e)[0]
        We = np.asarray(W_decoded(int(e)), dtype=np.float64)
        Ye = Xd[rows[sel]] @ We.T
        if Y is None:
            Y = np.empty((rows.size, We.shape[0]), dtype=np.float64)
        Y[sel] = Ye
    if Y is None:
        return np.zeros((0, 0)), np.zeros((0, 0), np.uint16), None, None
    Yb = bf16_rne(Y)
    P = D = None
    if G is not None:
        src = np.asarray(row_src, dtype=np.int32)[rows]
        P, D = dprob_from_output(G, Yb, src, topk, rows=np.arange(rows.size), slot_width=slot_width)
    return Y, Yb, P, D


# --------------------------------------------------------------------------
# fingerprint
# --------------------------------------------------------------------------
def fmix32(h: np.ndarray) -> np.ndarray:
    h = np.asarray(h, dtype=np.uint32).copy()
    h ^= h >> np.uint32(16)
    h *= np.uint32(0x85EBCA6B)
    h ^= h >> np.uint32(13)
    h *= np.uint32(0xC2B2AE35)
    h ^= h >> np.uint32(16)
    return h


def sm64(z: int) -> int:
    z &= MASK64
    z ^= z >> 30
    z = (z * 0xBF58476D1CE4E5B9) & MASK64
    z ^= z >> 27
    z = (z * 0x94D049BB133111EB) & MASK64
    z ^= z >> 31
    return z


def header_hash(dtype_code: int, shape) -> int:
    shape = [int(s) for s in shape]
    numel = 1
    for s in shape:
        numel *= s
    nbytes = numel * _itemsize(dtype_code)
    h = sm64(dtype_code)
    for v in [len(shape)] + shape + [numel, nbytes]:
        h = sm64(h ^ (v & MASK64))
    return h


_ITEMSIZE = {0: 1, 1: 1, 2: 2, 3: 4, 4: 8, 5: 2, 6: 2, 7: 4, 8: 8, 9: 1, 10: 2, 11: 4, 12: 8}


def _itemsize(code: int) -> int:
    return _ITEMSIZE[code]


def num_chunks(nbytes: int, chunk_bytes: int) -> int:
    return (nbytes + chunk_bytes - 1) // chunk_bytes


def fingerprint_chunks(data: bytes | np.ndarray, chunk_bytes: int = 1 << 20) -> np.ndarray:
    """Positional chunk hashes of a byte buffer (numpy, vectorised)."""
    buf = np.frombuffer(memoryview(data).cast("B"), dtype=np.uint8) if not isinstance(data, np.ndarray) \
        else np.ascontiguousarray(data).reshape(-1).view(np.uint8)
    nbytes = buf.size
    assert chunk_bytes % 4 == 0 and chunk_bytes > 0
    nch = num_chunks(nbytes, chunk_bytes)
    out = np.zeros(nch, dtype=np.uint64)
    wpc = chunk_bytes // 4
    for c in range(nch):
        b0 = c * chunk_bytes
        b1 = min(nbytes, b0 + chunk_bytes)
        seg = buf[b0:b1]
        pad = (-seg.size) % 4
        if pad:
            seg = np.concatenate([seg, np.zeros(pad, np.uint8)])
        w = seg.view("<u4").astype(np.uint32)
        i = (np.arange(w.size, dtype=np.uint64) + np.uint64(c * wpc))
        key = ((i * np.uint64(GOLDEN32)) & np.uint64(MASK32)).astype(np.uint32)
        acc = int(fmix32(w ^ key).astype(np.uint64).sum(dtype=np.uint64))
        out[c] = sm64(acc ^ ((c << 32) & MASK64) ^ (b1 - b0))
    return out


_XOR_KIND = {0: "u", 1: "i", 2: "i", 3: "i", 4: "i", 5: "f", 6: "bf", 7: "f", 8: "f", 9: "u", 10: "u",
             11: "u", 12: "u"}
_NP_DTYPE = {0: np.uint8, 1: np.int8, 2: np.int16, 3: np.int32, 4: np.int64, 5: np.float16, 6: np.uint16,
             7: np.float32, 8: np.float64, 9: np.uint8, 10: np.uint16, 11: np.uint32, 12: np.uint64}


def xor_chunks(data: np.ndarray, dtype_code: int, chunk_bytes: int = 1 << 20) -> np.ndarray:
    """Per-chunk xor of the elements widened to 64 bits (floats to binary64
    bit patterns, signed integers sign-extended, unsigned zero-extended)."""
    es = _itemsize(dtype_code)
    assert chunk_bytes % es == 0
    a = np.ascontiguousarray(data).reshape(-1).view(np.uint8).view(_NP_DTYPE[dtype_code])
    kind = _XOR_KIND[dtype_code]
    if kind == "f":
        w = a.astype(np.float64).view(np.uint64)
    elif kind == "bf":
        w = bf16_to_f64(a).view(np.uint64)
    elif kind == "i":
        w = a.astype(np.int64).view(np.uint64)
    else:
        w = a.astype(np.uint64)
    per = chunk_bytes // es
    nch = num_chunks(a.size * es, chunk_bytes)
    out = np.zeros(nch, dtype=np.uint64)
    for c in range(nch):
        out[c] = np.bitwise_xor.reduce(w[c * per:(c + 1) * per]) if w[c * per:(c + 1) * per].size else 0
    return out


def fingerprint(arr: np.ndarray, dtype_code: int, shape=None, chunk_bytes: int = 1 << 20, mode: str = "positional"):
    """(chunk hashes uint64 [nchunks], header hash) of an array's raw bytes."""
    arr = np.ascontiguousarray(arr)
    if shape is None:
        shape = arr.shape
    if mode == "positional":
        ch = fingerprint_chunks(arr, chunk_bytes)
    elif mode == "xor":
        ch = xor_chunks(arr, dtype_code, chunk_bytes)
    else:
        raise ValueError(mode)
    return ch, header_hash(dtype_code, shape)
