"""Thin ctypes binding of libdmoe.so (C ABI in include/dmoe.h).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  Tensors must be CUDA tensors on the current device;
calls are enqueued on torch's current stream and are asynchronous.  torch
provides device memory and streams, nothing else.

If the library has not been built, the first call raises -- there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

from . import build as _build

SLOT_COLS = 128
MAX_EXPERTS = 1024

OK = 0
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "invalid routing data",
                4: "device wait timed out", 5: "CUDA error", 6: "workspace missing or too small"}

DTYPE_CODES = {
    torch.uint8: 0, torch.int8: 1, torch.int16: 2, torch.int32: 3, torch.int64: 4,
    torch.float16: 5, torch.bfloat16: 6, torch.float32: 7, torch.float64: 8, torch.bool: 9,
}
for _name, _code in (("uint16", 10), ("uint32", 11), ("uint64", 12)):
    if hasattr(torch, _name):
        DTYPE_CODES[getattr(torch, _name)] = _code


class DmoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} (status {status})")
        self.status = status


class _Launch(ctypes.Structure):
    _fields_ = [("num_ctas", ctypes.c_int), ("flags", ctypes.c_int)]


LAUNCH_TEST_STALL = 1
LAUNCH_SINGLE_CTA = 2   # force the one-SM-per-tile kernel
LAUNCH_CTA_PAIRS = 4    # force the 2-SM (CTA pair) kernel
LAUNCH_NARROW_TILES = 8  # block-scaled MXFP8: one-slot (128 x 128) tiles only


_lib = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libdmoe.so; raises if it is missing (build it with build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"libdmoe.so is not built ({path}); run bitwise_deterministic_moe_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I, SZ, U64P = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.POINTER(ctypes.c_uint64)
    LP = ctypes.POINTER(_Launch)
    sig = {
        "dmoe_status_string": ([I], ctypes.c_char_p),
        "dmoe_version": ([], I),
        "dmoe_workspace_bytes": ([I, I, I], SZ),
        "dmoe_read_status": ([P, P], I),
        "dmoe_reserve_l2_persisting": ([SZ, ctypes.POINTER(ctypes.c_size_t)], I),
        "dmoe_permute_indices": ([P, I, I, I, P, P, P, P, SZ, P], I),
        "moe_dispatch_gather": ([P, P, I, I, I, P, P, SZ, P], I),
        "moe_token_combine": ([P, P, P, I, I, I, P, P, SZ, P], I),
        "moe_grouped_gemm_fwd": ([P, P, P, I, I, I, I, P, LP, P, SZ, P], I),
        "moe_grouped_gemm_dprob": ([P, P, P, I, I, I, I, P, P, P, I, I, P, P, LP, P, SZ, P], I),
        "moe_grouped_gemm_dprob_fp": ([P, P, P, I, I, I, I, P, P, P, I, I, P, P, SZ, P, P, LP, P, SZ, P], I),
        "moe_grouped_gemm_dprob_atomic": ([P, P, P, I, I, I, I, P, P, P, I, I, P, LP, P, SZ, P], I),
        "moe_grouped_gemm_dprob_serial": ([P, P, P, I, I, I, I, P, P, P, I, I, P, LP, P, SZ, P], I),
        "moe_grouped_gemm_wgrad": ([P, P, P, I, I, I, I, P, I, LP, P, SZ, P], I),
        "dmoe_quantize_mxfp8": ([P, I, I, P, P, P], I),
        "dmoe_quantize_nvfp4": ([P, I, I, P, P, P, P, SZ, P], I),
        "moe_grouped_gemm_dprob_mxfp8": ([P, P, P, P, P, I, I, I, I, P, P, P, I, I, P, P, LP, P, SZ, P], I),
        "moe_grouped_gemm_dprob_nvfp4": ([P, P, P, P, P, P, P, I, I, I, I, P, P, P, I, I, P, P, LP, P, SZ, P], I),
        "moe_dprob_epilogue": ([P, P, P, P, I, I, I, I, I, P, P], I),
        "moe_dprob_combine": ([P, P, I, I, I, I, P, P], I),
        "dmoe_fingerprint_num_chunks": ([SZ, SZ], SZ),
        "dmoe_fingerprint": ([P, SZ, I, I, ctypes.POINTER(ctypes.c_int64), SZ, I, P, U64P, P], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _check(st: int, what: str):
    if st != OK:
        raise DmoeError(st, what)


def _need(t: torch.Tensor, dtype, name: str, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _launch(num_ctas: int, flags: int = 0):
    return ctypes.byref(_Launch(int(num_ctas), int(flags)))


# ------------------------------------------------------------------ workspace
def workspace_bytes(T: int, topk: int, E: int) -> int:
    return int(load().dmoe_workspace_bytes(T, topk, E))


def workspace(T: int, topk: int, E: int, device=None) -> torch.Tensor:
    """Zero-filled device workspace for a problem of this size."""
    n = workspace_bytes(T, topk, E)
    return torch.zeros(n, dtype=torch.uint8, device=device or torch.cuda.current_device())


def reserve_l2_persisting(nbytes: int) -> int:
    """Sets the context's persisting-L2 set-aside that keeps grad_out
    resident for the dprob epilogue (clamped to half of L2 and the device
    maximum; 0 releases it).  Returns the bytes in effect."""
    if nbytes < 0:
        raise ValueError("nbytes must be >= 0")
    got = ctypes.c_size_t(0)
    _check(load().dmoe_reserve_l2_persisting(int(nbytes), ctypes.byref(got)), "dmoe_reserve_l2_persisting")
    return int(got.value)


def read_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronise, return and clear the device status word (0 = ok)."""
    return int(load().dmoe_read_status(_ptr(ws), _stream(stream)))


# ------------------------------------------------------------------ routing
def permute_indices(topk_ids: torch.Tensor, E: int, ws: torch.Tensor,
                    expert_offsets: Optional[torch.Tensor] = None, row_src: Optional[torch.Tensor] = None,
                    stream=None, row_of: Optional[torch.Tensor] = None, with_row_of: bool = False):
    """Returns (expert_offsets, row_src), plus row_of (the inverse map) when
    with_row_of is set or a row_of buffer is passed."""
    _need(topk_ids, torch.int32, "topk_ids")
    T, topk = topk_ids.shape
    dev = topk_ids.device
    if expert_offsets is None:
        expert_offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    if row_src is None:
        row_src = torch.empty(T * topk, dtype=torch.int32, device=dev)
    _need(expert_offsets, torch.int32, "expert_offsets", (E + 1,))
    _need(row_src, torch.int32, "row_src", (T * topk,))
    want = with_row_of or row_of is not None
    if want and row_of is None:
        row_of = torch.empty(T * topk, dtype=torch.int32, device=dev)
    if row_of is not None:
        _need(row_of, torch.int32, "row_of", (T * topk,))
    st = load().dmoe_permute_indices(_ptr(topk_ids), T, topk, E, _ptr(expert_offsets), _ptr(row_src),
                                     _ptr(row_of), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "dmoe_permute_indices")
    if want:
        return expert_offsets, row_src, row_of
    return expert_offsets, row_src


# ------------------------------------------------------------------ dispatch / combine
def dispatch_gather(hidden, row_src, topk: int, ws=None, out=None, stream=None):
    """x_perm [T*topk, H] = hidden[row_src // topk] (bits copied)."""
    _need(hidden, hidden.dtype, "hidden")
    if hidden.element_size() != 2 or hidden.dim() != 2:
        raise TypeError("hidden must be a 2-D tensor of a 2-byte type")
    T, H = hidden.shape
    R = T * topk
    if out is None:
        out = torch.empty(R, H, dtype=hidden.dtype, device=hidden.device)
    _need(out, hidden.dtype, "x_perm", (R, H))
    _need(row_src, torch.int32, "row_src", (R,))
    st = load().moe_dispatch_gather(_ptr(hidden), _ptr(row_src), T, topk, H, _ptr(out), _ptr(ws),
                                    0 if ws is None else ws.numel(), _stream(stream))
    _check(st, "moe_dispatch_gather")
    return out


def token_combine(expert_out, probs, row_of, ws=None, out=None, stream=None):
    """y [T, N] bf16 = sum_j probs[t, j] * expert_out[row_of[t*topk + j]], fp32, j ascending."""
    _need(expert_out, torch.bfloat16, "expert_out")
    _need(probs, torch.float32, "probs")
    T, topk = probs.shape
    R, N = expert_out.shape
    if R != T * topk:
        raise ValueError("expert_out must have T*topk rows")
    if out is None:
        out = torch.empty(T, N, dtype=torch.bfloat16, device=expert_out.device)
    _need(out, torch.bfloat16, "y", (T, N))
    _need(row_of, torch.int32, "row_of", (R,))
    st = load().moe_token_combine(_ptr(expert_out), _ptr(probs), _ptr(row_of), T, topk, N, _ptr(out), _ptr(ws),
                                  0 if ws is None else ws.numel(), _stream(stream))
    _check(st, "moe_token_combine")
    return out


# ------------------------------------------------------------------ GEMM
def _gemm_shapes(X, W, offs):
    _need(X, torch.bfloat16, "X_perm")
    _need(W, torch.bfloat16, "W")
    _need(offs, torch.int32, "expert_offsets")
    R, K = X.shape
    E, N, K2 = W.shape
    if K2 != K:
        raise ValueError("X_perm and W disagree on K")
    if offs.shape != (E + 1,):
        raise ValueError("expert_offsets must have E+1 entries")
    return R, E, K, N


def grouped_gemm_fwd(X_perm, W, expert_offsets, ws, out=None, num_ctas: int = 0, stream=None, flags: int = 0):
    R, E, K, N = _gemm_shapes(X_perm, W, expert_offsets)
    if out is None:
        out = torch.empty(R, N, dtype=torch.bfloat16, device=X_perm.device)
    _need(out, torch.bfloat16, "expert_out", (R, N))
    st = load().moe_grouped_gemm_fwd(_ptr(X_perm), _ptr(W), _ptr(expert_offsets), R, E, K, N, _ptr(out),
                                     _launch(num_ctas, flags), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "moe_grouped_gemm_fwd")
    return out


def grouped_gemm_dprob(X_perm, W, expert_offsets, grad_out, row_src, topk: int, ws, out=None, slots=None,
                       dprob=None, num_ctas: int = 0, stream=None, flags: int = 0):
    """Deterministic path: returns (expert_out bf16 [R,N], dprob fp32 [T,topk], slots fp32 [S,R])."""
    R, E, K, N = _gemm_shapes(X_perm, W, expert_offsets)
    T = R // topk
    dev = X_perm.device
    S = N // SLOT_COLS
    if out is None:
        out = torch.empty(R, N, dtype=torch.bfloat16, device=dev)
    if slots is None:
        slots = torch.empty(S, R, dtype=torch.float32, device=dev)
    if dprob is None:
        dprob = torch.empty(T, topk, dtype=torch.float32, device=dev)
    _need(out, torch.bfloat16, "expert_out", (R, N))
    _need(grad_out, torch.bfloat16, "grad_out", (T, N))
    _need(row_src, torch.int32, "row_src", (R,))
    _need(slots, torch.float32, "slots", (S, R))
    _need(dprob, torch.float32, "dprob", (T, topk))
    st = load().moe_grouped_gemm_dprob(_ptr(X_perm), _ptr(W), _ptr(expert_offsets), R, E, K, N, _ptr(out),
                                       _ptr(grad_out), _ptr(row_src), T, topk, _ptr(slots), _ptr(dprob),
                                       _launch(num_ctas, flags), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "moe_grouped_gemm_dprob")
    return out, dprob, slots


def grouped_gemm_dprob_fp(X_perm, W, expert_offsets, grad_out, row_src, topk: int, ws, out=None, slots=None,
                          dprob=None, chunk_bytes: int = 1 << 20, row_src_hash=None, dprob_hash=None,
                          num_ctas: int = 0, stream=None, flags: int = 0):
    """Deterministic path plus the positional chunk fingerprints of row_src and
    dprob (those of fingerprint(row_src) and fingerprint(dprob) with the same
    chunk_bytes).  Returns (expert_out, dprob, slots, row_src_hash, dprob_hash);
    the hashes are int64 tensors holding uint64 bit patterns."""
    R, E, K, N = _gemm_shapes(X_perm, W, expert_offsets)
    T = R // topk
    dev = X_perm.device
    S = N // SLOT_COLS
    nch = fingerprint_num_chunks(R * 4, chunk_bytes)
    if out is None:
        out = torch.empty(R, N, dtype=torch.bfloat16, device=dev)
    if slots is None:
        slots = torch.empty(S, R, dtype=torch.float32, device=dev)
    if dprob is None:
        dprob = torch.empty(T, topk, dtype=torch.float32, device=dev)
    if row_src_hash is None:
        row_src_hash = torch.empty(max(nch, 1), dtype=torch.int64, device=dev)
    if dprob_hash is None:
        dprob_hash = torch.empty(max(nch, 1), dtype=torch.int64, device=dev)
    _need(out, torch.bfloat16, "expert_out", (R, N))
    _need(grad_out, torch.bfloat16, "grad_out", (T, N))
    _need(row_src, torch.int32, "row_src", (R,))
    _need(slots, torch.float32, "slots", (S, R))
    _need(dprob, torch.float32, "dprob", (T, topk))
    for h, name in ((row_src_hash, "row_src_hash"), (dprob_hash, "dprob_hash")):
        _need(h, torch.int64, name)
        if h.numel() < nch:
            raise ValueError(f"{name} needs {nch} entries")
    st = load().moe_grouped_gemm_dprob_fp(_ptr(X_perm), _ptr(W), _ptr(expert_offsets), R, E, K, N, _ptr(out),
                                          _ptr(grad_out), _ptr(row_src), T, topk, _ptr(slots), _ptr(dprob),
                                          chunk_bytes, _ptr(row_src_hash), _ptr(dprob_hash),
                                          _launch(num_ctas, flags), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "moe_grouped_gemm_dprob_fp")
    return out, dprob, slots, row_src_hash[:nch], dprob_hash[:nch]


def grouped_gemm_dprob_atomic(X_perm, W, expert_offsets, grad_out, row_src, topk: int, ws, out=None, dprob=None,
                              num_ctas: int = 0, stream=None, flags: int = 0):
    """Nondeterministic atomicAdd control: returns (expert_out, dprob)."""
    R, E, K, N = _gemm_shapes(X_perm, W, expert_offsets)
    T = R // topk
    dev = X_perm.device
    if out is None:
        out = torch.empty(R, N, dtype=torch.bfloat16, device=dev)
    if dprob is None:
        dprob = torch.empty(T, topk, dtype=torch.float32, device=dev)
    _need(out, torch.bfloat16, "expert_out", (R, N))
    _need(grad_out, torch.bfloat16, "grad_out", (T, N))
    _need(row_src, torch.int32, "row_src", (R,))
    _need(dprob, torch.float32, "dprob", (T, topk))
    st = load().moe_grouped_gemm_dprob_atomic(_ptr(X_perm), _ptr(W), _ptr(expert_offsets), R, E, K, N, _ptr(out),
                                              _ptr(grad_out), _ptr(row_src), T, topk, _ptr(dprob),
                                              _launch(num_ctas, flags), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "moe_grouped_gemm_dprob_atomic")
    return out, dprob


def grouped_gemm_dprob_serial(X_perm, W, expert_offsets, grad_out, row_src, topk: int, ws, out=None, dprob=None,
                              num_ctas: int = 0, stream=None, flags: int = 0):
    """Serialized-writer control (deterministic, no slots): returns (expert_out, dprob)."""
    R, E, K, N = _gemm_shapes(X_perm, W, expert_offsets)
    T = R // topk
    dev = X_perm.device
    if out is None:
        out = torch.empty(R, N, dtype=torch.bfloat16, device=dev)
    if dprob is None:
        dprob = torch.empty(T, topk, dtype=torch.float32, device=dev)
    _need(out, torch.bfloat16, "expert_out", (R, N))
    _need(grad_out, torch.bfloat16, "grad_out", (T, N))
    _need(row_src, torch.int32, "row_src", (R,))
    _need(dprob, torch.float32, "dprob", (T, topk))
    st = load().moe_grouped_gemm_dprob_serial(_ptr(X_perm), _ptr(W), _ptr(expert_offsets), R, E, K, N, _ptr(out),
                                              _ptr(grad_out), _ptr(row_src), T, topk, _ptr(dprob),
                                              _launch(num_ctas, flags), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "moe_grouped_gemm_dprob_serial")
    return out, dprob


def grouped_gemm_wgrad(X_perm, dY, expert_offsets, ws, dW=None, E: Optional[int] = None, accumulate: bool = False,
                       num_ctas: int = 0, stream=None):
    """Deterministic weight gradient dW[e] (+)= dY_e^T X_e: fp32 [E, N, K]."""
    _need(X_perm, torch.bfloat16, "X_perm")
    _need(dY, torch.bfloat16, "dY")
    _need(expert_offsets, torch.int32, "expert_offsets")
    R, K = X_perm.shape
    R2, N = dY.shape
    if R2 != R:
        raise ValueError("X_perm and dY must have the same rows")
    E = expert_offsets.numel() - 1 if E is None else E
    if dW is None:
        if accumulate:
            raise ValueError("accumulate needs an existing dW")
        dW = torch.empty(E, N, K, dtype=torch.float32, device=X_perm.device)
    _need(dW, torch.float32, "dW", (E, N, K))
    st = load().moe_grouped_gemm_wgrad(_ptr(X_perm), _ptr(dY), _ptr(expert_offsets), R, E, K, N, _ptr(dW),
                                       1 if accumulate else 0, _launch(num_ctas), _ptr(ws), ws.numel(),
                                       _stream(stream))
    _check(st, "moe_grouped_gemm_wgrad")
    return dW


def dprob_epilogue(grad_out, expert_out, expert_offsets, row_src, topk: int, slots=None, stream=None):
    _need(expert_out, torch.bfloat16, "expert_out")
    R, N = expert_out.shape
    T = R // topk
    E = expert_offsets.numel() - 1
    S = N // SLOT_COLS
    if slots is None:
        slots = torch.empty(S, R, dtype=torch.float32, device=expert_out.device)
    _need(grad_out, torch.bfloat16, "grad_out", (T, N))
    _need(expert_offsets, torch.int32, "expert_offsets")
    _need(row_src, torch.int32, "row_src", (R,))
    _need(slots, torch.float32, "slots", (S, R))
    st = load().moe_dprob_epilogue(_ptr(grad_out), _ptr(expert_out), _ptr(expert_offsets), _ptr(row_src), R, E, T,
                                   topk, N, _ptr(slots), _stream(stream))
    _check(st, "moe_dprob_epilogue")
    return slots


def dprob_combine(slots, row_src, topk: int, dprob=None, stream=None):
    _need(slots, torch.float32, "slots")
    S, R = slots.shape
    T = R // topk
    if dprob is None:
        dprob = torch.empty(T, topk, dtype=torch.float32, device=slots.device)
    _need(row_src, torch.int32, "row_src", (R,))
    _need(dprob, torch.float32, "dprob", (T, topk))
    st = load().moe_dprob_combine(_ptr(slots), _ptr(row_src), R, S, T, topk, _ptr(dprob), _stream(stream))
    _check(st, "moe_dprob_combine")
    return dprob


# ------------------------------------------------------------------ block-scaled encodings
def quantize_mxfp8(x: torch.Tensor, values=None, scales=None, stream=None):
    """MXFP8 encoding of a bf16 [rows, cols] tensor: (E4M3 codes uint8 [rows, cols],
    E8M0 scales uint8 [rows, cols/32])."""
    _need(x, torch.bfloat16, "x")
    rows, cols = x.shape
    if values is None:
        values = torch.empty(rows, cols, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(rows, cols // 32, dtype=torch.uint8, device=x.device)
    _need(values, torch.uint8, "values", (rows, cols))
    _need(scales, torch.uint8, "scales", (rows, cols // 32))
    st = load().dmoe_quantize_mxfp8(_ptr(x), rows, cols, _ptr(values), _ptr(scales), _stream(stream))
    _check(st, "dmoe_quantize_mxfp8")
    return values, scales


def quantize_nvfp4(x: torch.Tensor, ws: torch.Tensor, packed=None, scales=None, s_enc=None, stream=None):
    """NVFP4 encoding of a bf16 [rows, cols] tensor: (packed E2M1 uint8 [rows, cols/2],
    E4M3 scales uint8 [rows, cols/16], tensor scale fp32 [1])."""
    _need(x, torch.bfloat16, "x")
    rows, cols = x.shape
    dev = x.device
    if packed is None:
        packed = torch.empty(rows, cols // 2, dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty(rows, cols // 16, dtype=torch.uint8, device=dev)
    if s_enc is None:
        s_enc = torch.empty(1, dtype=torch.float32, device=dev)
    _need(packed, torch.uint8, "packed", (rows, cols // 2))
    _need(scales, torch.uint8, "scales", (rows, cols // 16))
    _need(s_enc, torch.float32, "s_enc", (1,))
    st = load().dmoe_quantize_nvfp4(_ptr(x), rows, cols, _ptr(packed), _ptr(scales), _ptr(s_enc), _ptr(ws),
                                    ws.numel(), _stream(stream))
    _check(st, "dmoe_quantize_nvfp4")
    return packed, scales, s_enc


# ------------------------------------------------------------------ block-scaled grouped GEMM
def _block_scaled(kind, Xq, Xs, Xg, Wq, Ws, Wg, expert_offsets, K, grad_out, row_src, topk, ws, out, slots, dprob,
                  num_ctas, stream, flags=0):
    R = Xq.shape[0]
    E = expert_offsets.numel() - 1
    N = Wq.shape[1]
    kb = K if kind == 0 else K // 2
    sb = K // 32 if kind == 0 else K // 16
    dev = Xq.device
    _need(Xq, torch.uint8, "X codes", (R, kb))
    _need(Xs, torch.uint8, "X scales", (R, sb))
    _need(Wq, torch.uint8, "W codes", (E, N, kb))
    _need(Ws, torch.uint8, "W scales", (E * N, sb))
    _need(expert_offsets, torch.int32, "expert_offsets", (E + 1,))
    if kind == 1:
        _need(Xg, torch.float32, "X tensor scale", (1,))
        _need(Wg, torch.float32, "W tensor scale", (1,))
    if out is None:
        out = torch.empty(R, N, dtype=torch.bfloat16, device=dev)
    _need(out, torch.bfloat16, "expert_out", (R, N))
    T = 0
    if grad_out is not None:
        T = R // topk
        S = N // SLOT_COLS
        if slots is None:
            slots = torch.empty(S, R, dtype=torch.float32, device=dev)
        if dprob is None:
            dprob = torch.empty(T, topk, dtype=torch.float32, device=dev)
        _need(grad_out, torch.bfloat16, "grad_out", (T, N))
        _need(row_src, torch.int32, "row_src", (R,))
        _need(slots, torch.float32, "slots", (S, R))
        _need(dprob, torch.float32, "dprob", (T, topk))
    lib = load()
    if kind == 0:
        st = lib.moe_grouped_gemm_dprob_mxfp8(_ptr(Xq), _ptr(Xs), _ptr(Wq), _ptr(Ws), _ptr(expert_offsets), R, E, K, N,
                                              _ptr(out), _ptr(grad_out), _ptr(row_src), T, topk, _ptr(slots),
                                              _ptr(dprob), _launch(num_ctas, flags), _ptr(ws), ws.numel(), _stream(stream))
        _check(st, "moe_grouped_gemm_dprob_mxfp8")
    else:
        st = lib.moe_grouped_gemm_dprob_nvfp4(_ptr(Xq), _ptr(Xs), _ptr(Xg), _ptr(Wq), _ptr(Ws), _ptr(Wg),
                                              _ptr(expert_offsets), R, E, K, N, _ptr(out), _ptr(grad_out),
                                              _ptr(row_src), T, topk, _ptr(slots), _ptr(dprob), _launch(num_ctas, flags),
                                              _ptr(ws), ws.numel(), _stream(stream))
        _check(st, "moe_grouped_gemm_dprob_nvfp4")
    return out, dprob, slots


def grouped_gemm_dprob_mxfp8(X_q, X_scales, W_q, W_scales, expert_offsets, grad_out, row_src, topk: int, ws,
                             out=None, slots=None, dprob=None, num_ctas: int = 0, stream=None, flags: int = 0):
    """MXFP8 operands (E4M3 codes [R, K], [E, N, K]; E8M0 scales [R, K/32], [E*N, K/32]):
    returns (expert_out bf16 [R, N], dprob, slots); grad_out None = forward only (dprob, slots None)."""
    K = X_q.shape[1]
    return _block_scaled(0, X_q, X_scales, None, W_q, W_scales, None, expert_offsets, K, grad_out, row_src, topk, ws,
                         out, slots, dprob, num_ctas, stream, flags)


def grouped_gemm_dprob_nvfp4(X_packed, X_scales, X_s_enc, W_packed, W_scales, W_s_enc, expert_offsets, grad_out,
                             row_src, topk: int, ws, out=None, slots=None, dprob=None, num_ctas: int = 0,
                             stream=None):
    """NVFP4 operands (packed E2M1 [R, K/2], [E, N, K/2]; E4M3 scales [R, K/16], [E*N, K/16]; fp32
    tensor scales [1]): returns (expert_out bf16 [R, N], dprob, slots)."""
    K = X_packed.shape[1] * 2
    return _block_scaled(1, X_packed, X_scales, X_s_enc, W_packed, W_scales, W_s_enc, expert_offsets, K, grad_out,
                         row_src, topk, ws, out, slots, dprob, num_ctas, stream)


# ------------------------------------------------------------------ fingerprint
def fingerprint_num_chunks(nbytes: int, chunk_bytes: int = 1 << 20) -> int:
    return int(load().dmoe_fingerprint_num_chunks(nbytes, chunk_bytes))


def fingerprint(t: torch.Tensor, chunk_bytes: int = 1 << 20, mode: int = 0, out=None, stream=None):
    """Chunk-wise fingerprint of a contiguous CUDA tensor's bytes.

    Returns (chunk hashes as an int64 tensor holding uint64 bit patterns, header
    hash as a Python int)."""
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("fingerprint needs a contiguous CUDA tensor")
    code = DTYPE_CODES[t.dtype]
    nbytes = t.numel() * t.element_size()
    nch = fingerprint_num_chunks(nbytes, chunk_bytes)
    if out is None:
        out = torch.empty(max(nch, 1), dtype=torch.int64, device=t.device)
    shape = (ctypes.c_int64 * max(t.dim(), 1))(*t.shape)
    header = ctypes.c_uint64(0)
    st = load().dmoe_fingerprint(_ptr(t) if nbytes else None, nbytes, code, t.dim(), shape, chunk_bytes, mode,
                                 _ptr(out), ctypes.byref(header), _stream(stream))
    _check(st, "dmoe_fingerprint")
    return out[:nch], int(header.value)


def fingerprint_host(t: torch.Tensor, chunk_bytes: int = 1 << 20, mode: int = 0):
    """Fingerprint, returned as (list of Python ints, header int) after a sync."""
    ch, h = fingerprint(t, chunk_bytes, mode)
    vals = [v & ((1 << 64) - 1) for v in ch.cpu().tolist()]
    return vals, h
