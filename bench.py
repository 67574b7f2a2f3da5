"""Benchmark of the bitwise-deterministic MoE grouped GEMM + dprob path on GB300.

One step = one pass of the whole hot path over one batch of seeded synthetic
routed tokens shaped like the LatentMoE layer (T=8192 tokens, 512 experts,
top-22, K=1024, N=2048 latent, Zipf(1.1) expert popularity):
  1. routing indices (dmoe_permute_indices)
  2. chunk fingerprint of the routing map row_src (order-sensitive data)
  3. grouped GEMM with the fused private-slot dprob epilogue + fixed-order
     combine (moe_grouped_gemm_dprob)
  4. chunk fingerprint of dprob
The metric is algorithmic grouped-GEMM TFLOP/s (2*R*K*N per step) over the
whole step time.  The determinism tax compares the deterministic GEMM call
with the atomicAdd control (memset + moe_grouped_gemm_dprob_atomic); the
serialized-writer control (moe_grouped_gemm_dprob_serial: deterministic, the
N-tiles of a row block take turns) is timed beside them.

Usage: python bench.py [--gpus N --steps K --warmup W] [--impl reference]
For N > 1 (torchrun) every rank runs an independent replica on its own GPU
(the path has no data exchange on one node); value = all ranks' flops / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import atexit
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bitwise_deterministic_moe_gb300 import synth  # noqa: E402

WORKLOAD = "latent"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "grouped_gemm_latent_traffic.txt")
KERNEL_FLAGS = {"auto": 0, "single": 2, "pairs": 4}   # the C ABI's DMOE_LAUNCH_SINGLE_CTA / _CTA_PAIRS


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def algorithmic(cfg, off):
    """Algorithmic flops and HBM bytes of one grouped-GEMM+dprob call."""
    counts = np.diff(off)
    used = int((counts > 0).sum())
    R, K, N, T, S = cfg.R, cfg.K, cfg.N, cfg.T, cfg.S
    flops = 2.0 * R * K * N
    bytes_ = (R * K * 2 + used * N * K * 2 + R * N * 2 + T * N * 2 + 2 * S * R * 4 + R * 4 + R * 4
              + (cfg.E + 1) * 4)
    return flops, bytes_


def gemm_kernel_source_hash():
    """sha256 (16 hex digits) of the device code of grouped_gemm.cu: the file up
    to its host-side section, without comments and layout, so launcher-only or
    comment-only edits keep the capture valid."""
    import hashlib
    import re
    src = os.path.join(ROOT, "bitwise_deterministic_moe_gb300", "csrc", "grouped_gemm.cu")
    text = open(src, encoding="utf-8").read()
    marker = "// ---------------------------------------------------------------- host side"
    code = text[:text.index(marker)]
    # comments and layout do not change the kernel
    code = re.sub(r"/\*.*?\*/", " ", code, flags=re.S)
    code = re.sub(r"//[^\n]*", " ", code)
    code = " ".join(code.split())
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def gemm_traffic_per_launch(config):
    """dram read+write bytes of the GEMM kernel from the committed ncu summary
    of `config`, or None when there is none for it or the kernel's device code
    changed after the capture."""
    try:
        kv = {}
        for line in open(TRAFFIC_FILE):
            if "=" in line and not line.startswith("#"):
                k, v = line.split("=", 1)
                kv[k.strip()] = v.strip()
        if kv.get("workload") != config or kv.get("kernel_device_code_sha256_16") != gemm_kernel_source_hash():
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            atexit.register(self._kill)   # no sampler outlives the process, even after an error
        except Exception:
            self.proc = None

    def _kill(self):
        if self.proc is not None and self.proc.poll() is None:
            self.proc.kill()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's time (host all-reduce over gloo; replicas exchange
    nothing else)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step: float, steps: int, world: int, ms_max: float) -> float:
    """Units all ranks processed over the slowest rank's time (weak scaling:
    every replica runs the full workload)."""
    return world * flops_per_step * steps / (ms_max * 1e-3) / 1e12


def cpu_baseline(cfg, inp, target_s=12.0, full_configs=()):
    """The oracle as it stands, timed on this host's cores on a bounded sample
    of rows of the same workload (GEMM + bf16 rounding + slot partials + dprob)."""
    import oracle
    off, src = oracle.routing(inp.topk_ids, cfg.E)
    rng = np.random.default_rng(7)
    n = 64
    t = 0.0
    while True:
        rows = np.sort(rng.choice(cfg.R, n, replace=False)).astype(np.int64)
        t0 = time.perf_counter()
        oracle.expert_rows(inp.X, inp.W, off, rows, G=inp.G, row_src=src, topk=cfg.topk, want_Y=False,
                           want_Yb=True, want_P=True, want_D=True)
        t = time.perf_counter() - t0
        if t >= target_s * 0.5 or n >= cfg.R:
            break
        n = min(cfg.R, int(n * max(2.0, min(16.0, target_s / max(t, 1e-3)))))
    flops = 2.0 * n * cfg.K * cfg.N
    res = {"value": flops / t / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
           "sample": f"{n} of {cfg.R} permuted rows of the {cfg.name} workload (GEMM+bf16+slots+dprob, fp64), "
                     f"{t:.1f} s"}
    # the whole oracle on the larger configs, extrapolated from this sample:
    # its cost per row is one K x N row product plus the row's slots, so it
    # scales with R * K * N (labelled as an extrapolation, not a run)
    per_row_kn = t / (n * cfg.K * cfg.N)
    res["extrapolated_full_oracle"] = {
        name: {"s": per_row_kn * c.R * c.K * c.N, "rows": c.R,
               "basis": f"the {cfg.name} sample's time per row scaled by R*K*N (not run)"}
        for name, c in ((nm, synth.CONFIGS[nm]) for nm in ("imbal", "stress"))}
    if full_configs:
        # the whole oracle (routing, every row's GEMM, bf16 output, slots, dprob)
        # on the configs small enough to finish in seconds
        res["full_oracle"] = {}
        for name in full_configs:
            c = synth.CONFIGS[name]
            ci = synth.make_inputs(c)
            t0 = time.perf_counter()
            oracle.full(ci)
            dt = time.perf_counter() - t0
            res["full_oracle"][name] = {"s": dt, "tflops": 2.0 * c.R * c.K * c.N / dt / 1e12}
    return res


def run_reference(args):
    """Reference arm: the oracle (the only reference this path has) on the host
    cores, each step a bounded sample of the workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    cfg = synth.CONFIGS[args.config]
    inp = synth.make_inputs(cfg)
    import oracle
    off, src = oracle.routing(inp.topk_ids, cfg.E)
    rows_per_step = args.ref_rows
    rng = np.random.default_rng(11)
    samples = [np.sort(rng.choice(cfg.R, rows_per_step, replace=False)).astype(np.int64)
               for _ in range(args.warmup + args.steps)]
    for i in range(args.warmup):
        oracle.expert_rows(inp.X, inp.W, off, samples[i], G=inp.G, row_src=src, topk=cfg.topk, want_Y=False,
                           want_Yb=True, want_P=True, want_D=True)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.routing(inp.topk_ids, cfg.E)
        oracle.expert_rows(inp.X, inp.W, off, samples[args.warmup + i], G=inp.G, row_src=src, topk=cfg.topk,
                           want_Y=False, want_Yb=True, want_P=True, want_D=True)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows_per_step * cfg.K * cfg.N * args.steps
    value = flops / dt / 1e12
    line = {
        "impl": "reference", "metric": "grouped-GEMM+dprob TFLOP/s", "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{cfg.name}: T={cfg.T} E={cfg.E} topk={cfg.topk} K={cfg.K} N={cfg.N} "
                               f"routing={cfg.routing}", "rows_per_step": rows_per_step},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"{rows_per_step} of {cfg.R} permuted rows per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _mix64(z: int) -> int:
    """splitmix64's output function (folds chunk hashes into one digest)."""
    m = (1 << 64) - 1
    z &= m
    z ^= z >> 30
    z = (z * 0xBF58476D1CE4E5B9) & m
    z ^= z >> 27
    z = (z * 0x94D049BB133111EB) & m
    z ^= z >> 31
    return z


def output_digest(api, t):
    """One 64-bit digest of a device tensor: its fingerprint header folded with
    every 1 MiB chunk hash, in chunk order (hex)."""
    chunks, header = api.fingerprint_host(t)
    h = header
    for c in chunks:
        h = _mix64(h ^ c)
    return "%016x" % h


def dispatch_combine(api, cfg, inp, src, row_of, expert_out, timed, dev, iters):
    """HBM roofline of the dispatch gather (hidden [T,N] -> x_perm [R,N]) and
    the token combine (expert_out [R,N] -> y [T,N]) on the step's routing and
    GEMM output.  Algorithmic bytes: gather = R*N*2 written + T*N*2 read once +
    R*4 row ids; combine = R*N*2 read + T*N*2 written + R*4 row ids + R*4
    weights.  x_perm and expert_out are larger than L2; hidden (T*N*2) is
    meant to stay in L2 across its topk reads."""
    import torch
    pk, _ = peaks()
    R, T, N = cfg.R, cfg.T, cfg.N
    hidden = torch.from_numpy(synth.hidden_states(cfg).view(np.int16)).view(torch.bfloat16).to(dev)
    probs = torch.from_numpy(inp.probs).to(dev)
    xp = torch.empty(R, N, dtype=torch.bfloat16, device=dev)
    y = torch.empty(T, N, dtype=torch.bfloat16, device=dev)
    g_ms = timed(lambda: api.dispatch_gather(hidden, src, cfg.topk, out=xp), iters)
    c_ms = timed(lambda: api.token_combine(expert_out, probs, row_of, out=y), iters)
    res = {}
    for name, ms, b in (("gather", g_ms, R * N * 2 + T * N * 2 + R * 4),
                        ("combine", c_ms, R * N * 2 + T * N * 2 + R * 4 + R * 4)):
        gbs = b / (ms * 1e-3) / 1e9
        res[name] = {"ms": ms, "algorithmic_bytes": b, "achieved_gbs": gbs, "peak_gbs": pk["hbm_gbs"],
                     "frac": gbs / pk["hbm_gbs"]}
    del hidden, xp, y
    torch.cuda.empty_cache()
    return res


def wgrad_measure(api, cfg, X, dY, off, ws, timed, dev, iters):
    """The deterministic weight gradient dW[e] = dY_e^T X_e (fp32 [E, N, K]) on the
    step's X_perm and, as dY, its expert_out rows.  Algorithmic bytes: X and dY
    read once (R*K*2 + R*N*2) and dW written once (E*N*K*4); flops 2*R*K*N."""
    import torch
    pk, _ = peaks()
    dW = torch.empty(cfg.E, cfg.N, cfg.K, dtype=torch.float32, device=dev)
    ms = timed(lambda: api.grouped_gemm_wgrad(X, dY, off, ws, dW=dW), iters)
    if api.read_status(ws) != 0:
        raise RuntimeError("device status set while timing the weight gradient")
    b = cfg.R * cfg.K * 2 + cfg.R * cfg.N * 2 + cfg.E * cfg.N * cfg.K * 4 + (cfg.E + 1) * 4
    flops = 2.0 * cfg.R * cfg.K * cfg.N
    gbs = b / (ms * 1e-3) / 1e9
    del dW
    torch.cuda.empty_cache()
    return {"ms": ms, "tflops": flops / (ms * 1e-3) / 1e12, "algorithmic_bytes": b, "achieved_gbs": gbs,
            "peak_gbs": pk["hbm_gbs"], "frac": gbs / pk["hbm_gbs"], "bound": "hbm",
            "tensor_frac": flops / (ms * 1e-3) / 1e12 / pk["bf16_tflops"]}


def block_scaled_measure(api, cfg, X, W, G, off, src, ws, timed, iters):
    """The block-scaled grouped GEMM + slot dprob on the workload's operands
    encoded as MXFP8 and as NVFP4 (encoding outside the timed launches).
    Peaks: the measured bf16 burst figure times the nominal dense ratio of the
    format (fp8 4.5 / bf16 2.25 = 2; fp4 13.5 / 2.25 = 6 PFLOP/s on GB300).
    Algorithmic bytes: codes and scales of X and of the used experts' W read
    once, expert_out written, grad_out read once, slots written and read,
    row_src and dprob."""
    import torch
    pk, _ = peaks()
    counts = np.diff(off.cpu().numpy())
    used = int((counts > 0).sum())
    R, K, N, E, T, S = cfg.R, cfg.K, cfg.N, cfg.E, cfg.T, cfg.S
    flops = 2.0 * R * K * N
    W2 = W.view(E * N, K)
    res = {}
    out = torch.empty(R, N, dtype=torch.bfloat16, device=X.device)
    sl = torch.empty(S, R, dtype=torch.float32, device=X.device)
    dp = torch.empty(T, cfg.topk, dtype=torch.float32, device=X.device)
    for kind, ratio in (("mxfp8", 2.0), ("nvfp4", 6.0)):
        if kind == "mxfp8":
            xq, xs = api.quantize_mxfp8(X)
            wq, wsc = api.quantize_mxfp8(W2)
            fn = lambda: api.grouped_gemm_dprob_mxfp8(xq, xs, wq.view(E, N, K), wsc, off, G, src, cfg.topk, ws,
                                                      out=out, slots=sl, dprob=dp)
            opb = R * K + R * K // 32 + used * N * (K + K // 32)
        else:
            xq, xs, xg = api.quantize_nvfp4(X, ws)
            wq, wsc, wg = api.quantize_nvfp4(W2, ws)
            fn = lambda: api.grouped_gemm_dprob_nvfp4(xq, xs, xg, wq.view(E, N, K // 2), wsc, wg, off, G, src,
                                                      cfg.topk, ws, out=out, slots=sl, dprob=dp)
            opb = R * K // 2 + R * K // 16 + used * N * (K // 2 + K // 16)
        ms = timed(fn, iters)
        if api.read_status(ws) != 0:
            raise RuntimeError(f"device status set while timing the {kind} GEMM")
        b = opb + R * N * 2 + T * N * 2 + 2 * S * R * 4 + 2 * R * 4
        tf = flops / (ms * 1e-3) / 1e12
        peak = pk["bf16_tflops"] * ratio
        res[kind] = {"ms": ms, "tflops": tf, "peak_tflops": peak,
                     "peak_source": f"measured bf16 burst x {ratio:g} (nominal dense ratio)",
                     "tensor_frac": tf / peak, "algorithmic_bytes": b, "achieved_gbs": b / (ms * 1e-3) / 1e9,
                     "hbm_frac": b / (ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                     "kernel": ("grouped_gemm_bs_kernel: 128x256 tiles (one N=256 MMA per step over two slots), "
                                "scale boxes in a ring loaded once per four stages, one accumulator pair drained "
                                "to bf16 registers, four stages, one CTA per SM"
                                if kind == "mxfp8" and N % 256 == 0 else
                                "grouped_gemm_bs_kernel: 128x128 tiles, two epilogue groups on alternate tiles, "
                                "three accumulators, one CTA per SM")}
        del xq, xs, wq, wsc
    del out, sl, dp
    torch.cuda.empty_cache()
    return res


def passes_measure(api, cfg, out, slots, src, off, G, timed, iters, set_l2):
    """The HBM passes of the path on buffers of the workload: the chunk
    fingerprint of expert_out (R*N*2 bytes, larger than L2), the fixed-order
    slot combine (slots S*R*4 read, row_src and dprob R*4 each) and the
    unfused slot epilogue (expert_out R*N*2 and row_src R*4 read, grad_out
    T*N*2 read once, slots S*R*4 written)."""
    import torch
    pk, _ = peaks()
    fp = torch.empty(api.fingerprint_num_chunks(out.numel() * 2), dtype=torch.int64, device=out.device)
    dp = torch.empty(cfg.T, cfg.topk, dtype=torch.float32, device=out.device)
    sl = torch.empty_like(slots)
    res = {}
    # set_l2(keep): the persisting-L2 set-aside only for the pass with evict-last loads
    for name, fn, b, keep in (("fingerprint_expert_out", lambda: api.fingerprint(out, out=fp), out.numel() * 2, False),
                              ("slot_combine", lambda: api.dprob_combine(slots, src, cfg.topk, dprob=dp),
                               cfg.S * cfg.R * 4 + 2 * cfg.R * 4, False),
                              ("unfused_epilogue", lambda: api.dprob_epilogue(G, out, off, src, cfg.topk, slots=sl),
                               cfg.R * cfg.N * 2 + cfg.R * 4 + cfg.T * cfg.N * 2 + cfg.S * cfg.R * 4, True)):
        l2b = set_l2(keep)
        ms = timed(fn, iters)
        gbs = b / (ms * 1e-3) / 1e9
        res[name] = {"ms": ms, "algorithmic_bytes": b, "achieved_gbs": gbs, "peak_gbs": pk["hbm_gbs"],
                     "frac": gbs / pk["hbm_gbs"], "l2_persisting_bytes": l2b}
    set_l2(True)
    return res


def quant_measure(api, X, ws, timed, iters):
    """MXFP8 and NVFP4 encodings of the step's X_perm [R, K] bf16.  Algorithmic
    bytes: MXFP8 reads X once and writes R*K codes + R*K/32 scales; NVFP4 reads X
    twice (tensor maximum, then the blocks) and writes R*K/2 + R*K/16 bytes."""
    pk, _ = peaks()
    n = X.numel()
    res = {}
    # outputs allocated once; short kernels get at least 30 timed launches
    iters = max(iters, 30)
    mv, ms_ = api.quantize_mxfp8(X)
    ms = timed(lambda: api.quantize_mxfp8(X, values=mv, scales=ms_), iters)
    b = n * 2 + n + n // 32
    res["mxfp8"] = {"ms": ms, "algorithmic_bytes": b, "achieved_gbs": b / (ms * 1e-3) / 1e9}
    nv = api.quantize_nvfp4(X, ws)
    ms = timed(lambda: api.quantize_nvfp4(X, ws, packed=nv[0], scales=nv[1], s_enc=nv[2]), iters)
    b = 2 * n * 2 + n // 2 + n // 16
    res["nvfp4"] = {"ms": ms, "algorithmic_bytes": b, "achieved_gbs": b / (ms * 1e-3) / 1e9}
    for v in res.values():
        v["peak_gbs"] = pk["hbm_gbs"]
        v["frac"] = v["achieved_gbs"] / pk["hbm_gbs"]
    return res


# ---------------------------------------------------------------------------
def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("gloo")
    cfg = synth.CONFIGS[args.config]

    # the oracle's CPU baseline runs before any GPU work (rank 0, N = 1 only)
    inp = synth.make_inputs(cfg)
    base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        base = cpu_baseline(cfg, inp, target_s=args.cpu_seconds,
                            full_configs=() if args.no_cpu_full else ("tiny", "small"))

    from bitwise_deterministic_moe_gb300 import api, build
    build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    api.load()
    # keep grad_out resident in L2 for the dprob epilogue's gathers: a context
    # setting made once, before any timed work (--no-l2-reserve leaves it unset)
    l2_reserved = api.reserve_l2_persisting(0 if args.no_l2_reserve else cfg.T * cfg.N * 2)

    def set_l2(keep):
        """The set-aside serves the kernels that make evict-last accesses (the
        GEMM epilogues' grad_out gathers, the unfused epilogue, the dispatch
        gather); the others are timed with it released, since it takes L2
        capacity from them (the weight gradient is ~2% slower under it).
        Returns the bytes set aside while the measurement runs."""
        if not l2_reserved:
            return 0
        return api.reserve_l2_persisting(l2_reserved if keep else 0)

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)

    h_ids = torch.from_numpy(inp.topk_ids).pin_memory()
    h_X = bf16(inp.X).pin_memory()
    h_W = bf16(inp.W).pin_memory()
    h_G = bf16(inp.G).pin_memory()
    ids = h_ids.to(dev)
    X = h_X.to(dev)
    W = h_W.to(dev)
    G = h_G.to(dev)
    R, S, T, k = cfg.R, cfg.S, cfg.T, cfg.topk
    ws = api.workspace(T, k, cfg.E, dev)
    off = torch.empty(cfg.E + 1, dtype=torch.int32, device=dev)
    src = torch.empty(R, dtype=torch.int32, device=dev)
    row_of = torch.empty(R, dtype=torch.int32, device=dev)
    out = torch.empty(R, cfg.N, dtype=torch.bfloat16, device=dev)
    slots = torch.empty(S, R, dtype=torch.float32, device=dev)
    dprob = torch.empty(T, k, dtype=torch.float32, device=dev)
    fp_src = torch.empty(api.fingerprint_num_chunks(R * 4), dtype=torch.int64, device=dev)
    fp_dp = torch.empty(api.fingerprint_num_chunks(R * 4), dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)
    # routing 3 (histogram, block scan with offsets, scatter), GEMM 1, slot
    # combine taking the row_src and dprob fingerprints 1 (--separate-fp:
    # fingerprint 1 before the GEMM call and 1 after it instead)
    launches_per_step = 3 + 1 + 2 + 1 if args.separate_fp else 3 + 2

    def step(ev=None, inputs=None):
        ids_, X_, G_ = inputs if inputs is not None else (ids, X, G)
        api.permute_indices(ids_, cfg.E, ws, off, src, row_of=row_of)
        if not args.separate_fp:
            # the deterministic call whose combine also takes the chunk
            # fingerprints of row_src (the routing map) and dprob
            if ev is not None:
                ev[0].record(stream)
            api.grouped_gemm_dprob_fp(X_, W, off, G_, src, k, ws, out=out, slots=slots, dprob=dprob,
                                      row_src_hash=fp_src, dprob_hash=fp_dp,
                                      num_ctas=args.num_ctas, flags=KERNEL_FLAGS[args.kernel])
            if ev is not None:
                ev[1].record(stream)
            return
        api.fingerprint(src, out=fp_src)
        if ev is not None:
            ev[0].record(stream)
        api.grouped_gemm_dprob(X_, W, off, G_, src, k, ws, out=out, slots=slots, dprob=dprob,
                               num_ctas=args.num_ctas, flags=KERNEL_FLAGS[args.kernel])
        if ev is not None:
            ev[1].record(stream)
        api.fingerprint(dprob, out=fp_dp)

    # the clock sampler starts (and takes its first samples) before the
    # warm-up steps, so that no idle pause separates them from the timed steps
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st = api.read_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")
    off_np = off.cpu().numpy()
    flops, abytes = algorithmic(cfg, off_np)

    # ---------------- timed region: K steps, inputs resident in HBM (> L2)
    # The GEMM call is bracketed by events on the last step of every group of
    # ev_every steps only: an event between two programmatically chained
    # launches exposes the next launch's latency (~6 us a step with events on
    # every step), and the first timed step follows the host's checks above
    # after a short pause.
    ev_every = max(1, min(4, args.steps // 3))
    gemm_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               if i % ev_every == ev_every - 1 else None for i in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_start.record(stream)
    for i in range(args.steps):
        step(gemm_ev[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    ms = t_start.elapsed_time(t_end)
    gemm_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in gemm_ev if e is not None]))
    gemm_calls_timed = sum(e is not None for e in gemm_ev)
    if api.read_status(ws) != 0:
        raise RuntimeError("device status set during the timed region")
    ms_max = max_over_ranks(ms, world)
    ms_per_step = ms_max / args.steps
    value = whole_job_tflops(flops, args.steps, world, ms_max)

    # ---------------- determinism tax: deterministic call vs atomic control
    def timed(fn, iters):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        fn()
        torch.cuda.synchronize(dev)
        a.record(stream)
        for _ in range(iters):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / iters

    # L2 flush: write a buffer twice the size of L2, then read another one of
    # that size, before a timed launch: the launch starts with nothing of its
    # inputs in L2, and with clean lines there, so it does not pay for writing
    # back the flush's own dirty data (cold-L2 protocol)
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (128 << 20))
    flush_buf = torch.empty(2 * l2_bytes // 4, dtype=torch.int32, device=dev)
    flush_rd = torch.ones(2 * l2_bytes // 4, dtype=torch.int32, device=dev)
    flush_sink = torch.empty((), dtype=torch.int64, device=dev)

    def timed_each(fn, n, flush):
        """Median, min and max (ms) of n single launches, each bracketed by its
        own events on the launching stream, after an L2 flush when `flush`."""
        fn()
        torch.cuda.synchronize(dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in evs:
            if flush:
                flush_buf.fill_(1)
                torch.sum(flush_rd, dim=0, out=flush_sink)
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        t = [a.elapsed_time(b) for a, b in evs]
        return {"median_ms": float(np.median(t)), "min_ms": float(np.min(t)), "max_ms": float(np.max(t)),
                "runs": n}

    def gemm_call():
        api.grouped_gemm_dprob(X, W, off, G, src, k, ws, out=out, slots=slots, dprob=dprob,
                               num_ctas=args.num_ctas, flags=KERNEL_FLAGS[args.kernel])

    call_cold = timed_each(gemm_call, args.call_runs, True)
    call_hot = timed_each(gemm_call, args.call_runs, False)
    call_unreserved = None
    if l2_reserved:
        # the same call with no persisting-L2 set-aside, for comparison
        api.reserve_l2_persisting(0)
        call_unreserved = timed_each(gemm_call, args.call_runs, False)
        api.reserve_l2_persisting(l2_reserved)
    if api.read_status(ws) != 0:
        raise RuntimeError("device status set while timing single calls")

    def combine_pass(sl_, src_, c_):
        """The fixed-order slot combine as an HBM pass: slots S*R*4 read, row_src
        and dprob R*4 each; every launch after an L2 flush (the buffer is
        smaller than L2)."""
        pk_, _ = peaks()
        dp_ = torch.empty(c_.T, c_.topk, dtype=torch.float32, device=dev)
        set_l2(False)
        t = timed_each(lambda: api.dprob_combine(sl_, src_, c_.topk, dprob=dp_), 30, True)
        set_l2(True)
        b = c_.S * c_.R * 4 + 2 * c_.R * 4
        gbs = b / (t["median_ms"] * 1e-3) / 1e9
        return {"ms": t["median_ms"], "ms_range": [t["min_ms"], t["max_ms"]], "runs": t["runs"],
                "algorithmic_bytes": b, "achieved_gbs": gbs, "peak_gbs": pk_["hbm_gbs"], "frac": gbs / pk_["hbm_gbs"],
                "l2": "flushed before each launch", "rows": c_.R, "slots": c_.S, "l2_persisting_bytes": 0}

    combine_sizes = {}
    dprob_a = torch.empty_like(dprob)
    tax = {}
    for name in (args.config, "imbal"):
        if name == args.config:
            tX, tW, tG, toff, tsrc, tcfg, tws = X, W, G, off, src, cfg, ws
        else:
            if args.skip_imbal:
                continue
            tcfg = synth.CONFIGS[name]
            ti = synth.make_inputs(tcfg)
            tX, tW, tG = bf16(ti.X).to(dev), bf16(ti.W).to(dev), bf16(ti.G).to(dev)
            tws = api.workspace(tcfg.T, tcfg.topk, tcfg.E, dev)
            toff, tsrc = api.permute_indices(torch.from_numpy(ti.topk_ids).to(dev), tcfg.E, tws)
        to = torch.empty(tcfg.R, tcfg.N, dtype=torch.bfloat16, device=dev)
        tsl = torch.empty(tcfg.S, tcfg.R, dtype=torch.float32, device=dev)
        tdp = torch.empty(tcfg.T, tcfg.topk, dtype=torch.float32, device=dev)
        tda = torch.empty_like(tdp)
        det_ms, atom_ms, ser_ms, fwd_ms, unf_ms = [], [], [], [], []

        def unfused():
            api.grouped_gemm_fwd(tX, tW, toff, tws, out=to)
            api.dprob_epilogue(tG, to, toff, tsrc, tcfg.topk, slots=tsl)
            api.dprob_combine(tsl, tsrc, tcfg.topk, dprob=tda)

        for _ in range(args.tax_rounds):   # interleave to share clock/thermal conditions
            det_ms.append(timed(lambda: api.grouped_gemm_dprob(tX, tW, toff, tG, tsrc, tcfg.topk, tws, out=to,
                                                               slots=tsl, dprob=tdp), args.tax_iters))
            fwd_ms.append(timed(lambda: api.grouped_gemm_fwd(tX, tW, toff, tws, out=to), args.tax_iters))
            unf_ms.append(timed(unfused, args.tax_iters))
            atom_ms.append(timed(lambda: api.grouped_gemm_dprob_atomic(tX, tW, toff, tG, tsrc, tcfg.topk, tws,
                                                                       out=to, dprob=tda), args.tax_iters))
            ser_ms.append(timed(lambda: api.grouped_gemm_dprob_serial(tX, tW, toff, tG, tsrc, tcfg.topk, tws,
                                                                      out=to, dprob=tda), args.tax_iters))
        if api.read_status(tws) != 0:
            raise RuntimeError("device status set while timing the controls")
        if name != args.config:
            combine_sizes[name] = combine_pass(tsl, tsrc, tcfg)
        d, a, sr = float(np.median(det_ms)), float(np.median(atom_ms)), float(np.median(ser_ms))
        tf, _ = algorithmic(tcfg, toff.cpu().numpy())
        fw, un = float(np.median(fwd_ms)), float(np.median(unf_ms))
        per_round = [(x / y - 1.0) * 100.0 for x, y in zip(det_ms, atom_ms)]
        # the tax is a paired comparison: each round times both calls under
        # the same clock and thermal conditions, so the headline is the median
        # of the per-round ratios; the ratio of the medians is kept beside it
        tax[name] = {"det_ms": d, "atomic_ms": a, "tax_pct": float(np.median(per_round)),
                     "tax_pct_ratio_of_medians": (d / a - 1.0) * 100.0,
                     "rounds": len(det_ms), "iters_per_round": args.tax_iters,
                     "det_ms_range": [float(min(det_ms)), float(max(det_ms))],
                     "atomic_ms_range": [float(min(atom_ms)), float(max(atom_ms))],
                     "tax_pct_per_round_range": [float(min(per_round)), float(max(per_round))],
                     "det_tflops": tf / (d * 1e-3) / 1e12,
                     "serial_ms": sr, "serial_tax_pct": (sr / a - 1.0) * 100.0,
                     # the GEMM alone, and the same dprob through separate
                     # epilogue and combine launches (same bits): what fusing saves
                     "fwd_ms": fw, "unfused_ms": un,
                     "fused_epilogue_ns_per_row": (d - fw) * 1e6 / tcfg.R,
                     "unfused_epilogue_ns_per_row": (un - fw) * 1e6 / tcfg.R}
        if name != args.config:
            del tX, tW, tG, to, tsl, tdp, tda
            torch.cuda.empty_cache()
    del dprob_a

    # ---------------- the steps either side of the GEMM (not in the step)
    around = None if args.skip_dispatch else dispatch_combine(api, cfg, inp, src, row_of, out, timed, dev,
                                                              args.tax_iters)
    bsg = None if args.skip_block_scaled else block_scaled_measure(api, cfg, X, W, G, off, src, ws, timed,
                                                                    args.tax_iters)
    # no evict-last accesses in the weight gradient and the encoders
    l2_off = set_l2(False)
    wg = None if args.skip_wgrad else wgrad_measure(api, cfg, X, out, off, ws, timed, dev, args.tax_iters)
    qz = None if args.skip_quant else quant_measure(api, X, ws, timed, args.tax_iters)
    l2_on = set_l2(True)
    for v in (around, bsg):
        if v:
            v["l2_persisting_bytes"] = l2_on
    if wg:
        wg["l2_persisting_bytes"] = l2_off
    if qz:
        qz["l2_persisting_bytes"] = l2_off
    hp = passes_measure(api, cfg, out, slots, src, off, G, timed, max(args.tax_iters, 20), set_l2)
    hp["slot_combine"].update({"l2": "back to back, buffer smaller than L2"})
    hp["slot_combine_latent_cold"] = combine_pass(slots, src, cfg)
    for name, v in combine_sizes.items():
        hp[f"slot_combine_{name}"] = v
    if not args.skip_stress_combine:
        scfg = synth.CONFIGS["stress"]
        gen = torch.Generator(device=dev).manual_seed(scfg.seed)
        s_sl = torch.randn(scfg.S, scfg.R, device=dev, generator=gen)
        s_src = torch.randperm(scfg.R, device=dev, generator=gen).to(torch.int32)
        hp["slot_combine_stress"] = combine_pass(s_sl, s_src, scfg)
        hp["slot_combine_stress"]["inputs"] = "seeded normal slot values and a random permutation as row_src"
        del s_sl, s_src

    # ---------------- end to end through the public API, host buffers
    e2e = None
    if not args.skip_e2e:
        h_dprob = torch.empty(T, k, dtype=torch.float32).pin_memory()
        # the resident path's results, to check the host-buffer path's bits against
        ref_dprob, ref_fp = dprob.cpu(), fp_dp.cpu()
        h_fp = torch.empty_like(fp_dp, device="cpu").pin_memory()
        h_fps = torch.empty_like(fp_src, device="cpu").pin_memory()

        # per-step inputs come from pinned host memory every step; the expert
        # weights are model parameters, resident on the device across steps
        W.copy_(h_W)
        # Two sets of device input buffers, as a data loader double-buffers:
        # step i+1's inputs are copied on a copy stream while step i computes.
        # Every timed step still copies its own inputs; the first copy is not
        # overlapped (pipeline fill) and nothing is copied past the last step.
        sets = [(ids, X, G), (torch.empty_like(ids), torch.empty_like(X), torch.empty_like(G))]
        copy_stream = torch.cuda.Stream(dev)
        ev_copied = [torch.cuda.Event(), torch.cuda.Event()]
        ev_used = [torch.cuda.Event(), torch.cuda.Event()]

        def copy_in(i):
            sl = i % 2
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(ev_used[sl])      # the step two back is done with this set
                for dst, hsrc in zip(sets[sl], (h_ids, h_X, h_G)):
                    dst.copy_(hsrc, non_blocking=True)
                ev_copied[sl].record(copy_stream)

        def compute(i):
            sl = i % 2
            stream.wait_event(ev_copied[sl])
            step(inputs=sets[sl])
            ev_used[sl].record(stream)
            h_dprob.copy_(dprob, non_blocking=True)
            h_fp.copy_(fp_dp, non_blocking=True)
            h_fps.copy_(fp_src, non_blocking=True)

        def run(n, start_ev=None):
            if start_ev is not None:
                copy_stream.wait_event(start_ev)
            copy_in(0)
            for i in range(n):
                if i + 1 < n:
                    copy_in(i + 1)
                compute(i)

        for e in ev_used:
            e.record(stream)
        run(2)
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run(args.e2e_steps, start_ev=a)
        b.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(a.elapsed_time(b), world)
        h2d = sum(t.numel() * t.element_size() for t in (h_ids, h_X, h_G))
        d2h = sum(t.numel() * t.element_size() for t in (h_dprob, h_fp, h_fps))
        # the host link's own rate on this machine: the same per-step input copies
        # alone, back to back on the copy stream (median of five)
        link_ms = []
        for _ in range(5):
            la, lb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            la.record(copy_stream)
            with torch.cuda.stream(copy_stream):
                for dst, hsrc in zip(sets[1], (h_ids, h_X, h_G)):
                    dst.copy_(hsrc, non_blocking=True)
            lb.record(copy_stream)
            torch.cuda.synchronize(dev)
            link_ms.append(la.elapsed_time(lb))
        link_ms = float(np.median(link_ms))
        e2e = {"value": whole_job_tflops(flops, args.e2e_steps, world, e_ms), "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e_ms / args.e2e_steps,
               "copied": "topk_ids, X_perm, grad_out in (pinned host -> device, every step, the next step's "
                         "copy overlapping the current step's compute); dprob and both fingerprints out; "
                         "expert weights resident",
               "bitwise_equal_to_resident": bool(torch.equal(h_dprob, ref_dprob) and torch.equal(h_fp, ref_fp)),
               "h2d_copy_alone_ms": link_ms, "h2d_copy_alone_gbs": h2d / (link_ms * 1e-3) / 1e9}

    # digests of the step's outputs (chunk fingerprints folded with the header):
    # identical inputs give identical digests on every run
    fingerprints = {name: output_digest(api, t) for name, t in
                    (("row_src", src), ("expert_offsets", off), ("expert_out", out), ("slots", slots),
                     ("dprob", dprob))}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    pk, pk_kind = peaks()
    gemm_s = gemm_ms * 1e-3
    achieved_gbs = abytes / gemm_s / 1e9
    achieved_tf = flops / gemm_s / 1e12
    t_hbm = abytes / (pk["hbm_gbs"] * 1e9)
    # The tensor peak that matches the timed region: the burst cuBLAS figure for
    # a region under a second (the clocks stay up), the sustained one (seconds
    # back to back under the power limit) for a longer region.
    burst = pk.get("bf16_tflops") or FALLBACK_PEAKS["bf16_tflops"]
    sustained = pk.get("bf16_tflops_sustained") or FALLBACK_PEAKS["bf16_tflops_sustained"]
    peak_kind = "burst" if ms_max < 1000.0 else "sustained"
    tc_peak = burst if peak_kind == "burst" else sustained
    t_tc = flops / (tc_peak * 1e12)
    traffic = gemm_traffic_per_launch(args.config)
    if t_hbm >= t_tc:
        roof = {"bound": "hbm", "achieved": achieved_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved_gbs / pk["hbm_gbs"], "traffic": traffic}
    else:
        roof = {"bound": "tensor", "achieved": achieved_tf, "peak": tc_peak, "unit": "TFLOP/s",
                "frac": achieved_tf / tc_peak, "traffic": traffic}
    # the call's default kernel choice: CTA pairs when R >= 512*E (mean rows per expert)
    pairs = args.kernel == "pairs" or (args.kernel == "auto" and cfg.R >= 512 * cfg.E)
    gemm_kernel = "grouped_gemm_pair_kernel<slots>" if pairs else "grouped_gemm_kernel<slots>"
    roof.update({"kernel": gemm_kernel + " + combine (moe_grouped_gemm_dprob)",
                 "launch_ms": gemm_ms, "launch_ms_calls": f"{gemm_calls_timed} of the {args.steps} timed calls (one in every {ev_every} steps)",
                 "launch_call": "moe_grouped_gemm_dprob" if args.separate_fp else
                                "moe_grouped_gemm_dprob_fp (the same call, its combine also fingerprinting row_src and dprob)",
                 "single_call_runs": "moe_grouped_gemm_dprob (call_l2_flushed, call_l2_hot)",
                 "algorithmic_bytes": abytes, "algorithmic_flops": flops,
                 "peak_source": f"{pk_kind} ({os.path.basename(PEAKS_FILE) if pk_kind == 'measured' else 'profiling recipe'})",
                 "tensor_frac": achieved_tf / tc_peak, "tensor_tflops": achieved_tf,
                 "tensor_peak": {"tflops": tc_peak, "kind": peak_kind,
                                 "why": "timed region %.3f s: %s" % (ms_max * 1e-3,
                                        "under 1 s, burst figure" if peak_kind == "burst"
                                        else "1 s or longer, sustained figure")},
                 # the combined bound max(flops / tensor peak, bytes / HBM peak) and the
                 # fraction of it the call reaches
                 "combined_bound": {"ms": max(t_tc, t_hbm) * 1e3, "tensor_ms": t_tc * 1e3, "hbm_ms": t_hbm * 1e3,
                                    "frac": max(t_tc, t_hbm) / gemm_s},
                 "tensor_frac_of_burst": achieved_tf / burst,
                 "tensor_frac_of_sustained": achieved_tf / sustained,
                 "hbm_frac": achieved_gbs / pk["hbm_gbs"],
                 # single calls, median of call_runs launches: each after an L2
                 # flush (cold) and back to back (hot)
                 "call_l2_flushed": dict(call_cold, tflops=flops / (call_cold["median_ms"] * 1e-3) / 1e12),
                 "call_l2_hot": dict(call_hot, tflops=flops / (call_hot["median_ms"] * 1e-3) / 1e12)})
    if call_unreserved is not None:
        roof["call_l2_hot_no_l2_reserve"] = dict(call_unreserved,
                                                 tflops=flops / (call_unreserved["median_ms"] * 1e-3) / 1e12)
    line = {
        "metric": "grouped-GEMM+dprob TFLOP/s", "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{cfg.name}: T={cfg.T} E={cfg.E} topk={cfg.topk} K={cfg.K} N={cfg.N} "
                               f"routing={cfg.routing} (seed {cfg.seed})",
                   "step": ("permute + grouped GEMM/slot dprob/combine, the combine also fingerprinting row_src and dprob"
                            if not args.separate_fp else
                            "permute + fingerprint(row_src) + grouped GEMM/slot dprob/combine + fingerprint(dprob)"),
                   "l2": "inputs larger than L2 (X+W+grad_out = %.2f GB)" % ((cfg.R * cfg.K + cfg.E * cfg.N * cfg.K
                                                                            + cfg.T * cfg.N) * 2 / 1e9),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "maxvio": synth.maxvio(inp.topk_ids, cfg.E),
                   "gemm_launch": {"kernel": gemm_kernel, "num_ctas": args.num_ctas or "all resident"},
                   "l2_persisting_bytes": l2_reserved},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": roof,
        "determinism_tax": tax,
        "dispatch_combine": around,
        "wgrad": wg,
        "quantize": qz,
        "block_scaled_gemm": bsg,
        "hbm_passes": hp,
        "e2e": e2e,
        "clocks": clocks,
        "fingerprints": fingerprints,
    }
    if base is not None:
        line["cpu_baseline"] = base
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def combine_only(args):
    """The fixed-order slot combine alone, on the slot buffer of --config
    (S x R fp32, seeded normal values, a seeded random permutation as
    row_src): 3 warm-up launches, then 5 launches each after an L2 flush.
    Prints one JSON object; not part of the bench line (a short command for
    an ncu capture of this one kernel)."""
    import torch
    from bitwise_deterministic_moe_gb300 import api, build
    build.build()
    api.load()
    dev = torch.device("cuda", 0)
    cfg = synth.CONFIGS[args.config]
    gen = torch.Generator(device=dev).manual_seed(cfg.seed)
    sl = torch.randn(cfg.S, cfg.R, device=dev, generator=gen)
    src = torch.randperm(cfg.R, device=dev, generator=gen).to(torch.int32)
    dp = torch.empty(cfg.T, cfg.topk, dtype=torch.float32, device=dev)
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (128 << 20))
    flush_buf = torch.empty(2 * l2_bytes // 4, dtype=torch.int32, device=dev)
    flush_rd = torch.ones(2 * l2_bytes // 4, dtype=torch.int32, device=dev)
    flush_sink = torch.empty((), dtype=torch.int64, device=dev)
    for _ in range(3):
        api.dprob_combine(sl, src, cfg.topk, dprob=dp)
    t = []
    for _ in range(5):
        flush_buf.fill_(1)
        torch.sum(flush_rd, dim=0, out=flush_sink)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        api.dprob_combine(sl, src, cfg.topk, dprob=dp)
        b.record()
        torch.cuda.synchronize(dev)
        t.append(a.elapsed_time(b))
    pk, _ = peaks()
    b = cfg.S * cfg.R * 4 + 2 * cfg.R * 4
    ms = float(np.median(t))
    print(json.dumps({"pass": "slot_combine", "config": cfg.name, "rows": cfg.R, "slots": cfg.S,
                      "algorithmic_bytes": b, "ms": ms, "frac": b / (ms * 1e-3) / 1e9 / pk["hbm_gbs"]}))
    return 0


def dense_compare(args):
    """The grouped GEMM on dense shapes (one expert holding every row, or equal
    experts) next to cuBLAS (torch.matmul / torch.bmm) on the same bf16
    operands: separates the kernel's own efficiency from the MoE routing.
    Prints one JSON object; not part of the bench line."""
    import torch
    from bitwise_deterministic_moe_gb300 import api, build
    build.build()
    api.load()
    torch.manual_seed(0)
    res = {}
    for E, Me, K, N in ((1, 131072, 1024, 2048), (64, 2048, 1024, 2048), (128, 1088, 1024, 2048)):
        R = E * Me
        X = torch.randn(R, K, device="cuda").to(torch.bfloat16)
        W = (torch.randn(E, N, K, device="cuda") * 0.03).to(torch.bfloat16)
        off = (torch.arange(E + 1, dtype=torch.int32, device="cuda") * Me).contiguous()
        ws = api.workspace(R, 1, E)
        out = torch.empty(R, N, dtype=torch.bfloat16, device="cuda")
        ref = torch.empty(E, Me, N, dtype=torch.bfloat16, device="cuda")

        def t(fn):
            for _ in range(max(args.warmup, 3)):
                fn()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(max(args.steps, 1)):
                fn()
            b.record()
            torch.cuda.synchronize()
            return a.elapsed_time(b) / max(args.steps, 1)

        if E == 1:
            ms_ref = t(lambda: torch.matmul(X, W[0].t(), out=ref[0]))
        else:
            ms_ref = t(lambda: torch.bmm(X.view(E, Me, K), W.transpose(1, 2), out=ref))
        ms_1 = t(lambda: api.grouped_gemm_fwd(X, W, off, ws, out=out, flags=api.LAUNCH_SINGLE_CTA))
        same_1 = bool(torch.equal(out, ref.view(R, N)))
        ms_2 = t(lambda: api.grouped_gemm_fwd(X, W, off, ws, out=out, flags=api.LAUNCH_CTA_PAIRS))
        same_2 = bool(torch.equal(out, ref.view(R, N)))
        fl = 2.0 * R * K * N
        res[f"{E}x{Me}x{K}->{N}"] = {
            "tflops": {"cublas": fl / ms_ref / 1e9, "single_cta": fl / ms_1 / 1e9, "cta_pairs": fl / ms_2 / 1e9},
            "bitwise_equal_to_cublas": {"single_cta": same_1, "cta_pairs": same_2}}
        del X, W, out, ref
        torch.cuda.empty_cache()
    print(json.dumps({"dense_compare": res}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)   # ~0.3 s timed: the clock sampler lands inside
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=WORKLOAD, choices=sorted(synth.CONFIGS))
    ap.add_argument("--tax-iters", type=int, default=10)
    ap.add_argument("--tax-rounds", type=int, default=11, help="interleaved rounds of the determinism tax")
    ap.add_argument("--call-runs", type=int, default=20, help="single GEMM calls timed cold-L2 and hot-L2")
    ap.add_argument("--skip-stress-combine", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-rows", type=int, default=1024)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cpu-full", action="store_true", help="skip the whole-oracle runs on tiny and small")
    ap.add_argument("--skip-imbal", action="store_true")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-dispatch", action="store_true")
    ap.add_argument("--skip-wgrad", action="store_true")
    ap.add_argument("--skip-quant", action="store_true")
    ap.add_argument("--skip-block-scaled", action="store_true")
    ap.add_argument("--separate-fp", action="store_true",
                    help="step through moe_grouped_gemm_dprob with separate fingerprint launches for row_src "
                         "and dprob, instead of moe_grouped_gemm_dprob_fp whose combine takes them")
    ap.add_argument("--no-l2-reserve", action="store_true",
                    help="do not set aside persisting L2 for grad_out (dmoe_reserve_l2_persisting)")
    ap.add_argument("--num-ctas", type=int, default=0, help="persistent CTAs of the GEMM (0 = all resident)")
    ap.add_argument("--kernel", default="auto", choices=sorted(KERNEL_FLAGS),
                    help="GEMM kernel: the call's own choice, or force one (same bits)")
    ap.add_argument("--dense-compare", action="store_true",
                    help="time the grouped GEMM on dense shapes next to cuBLAS and exit")
    ap.add_argument("--combine-only", action="store_true",
                    help="time the slot combine alone on --config's buffer sizes and exit")
    args = ap.parse_args()
    if args.dense_compare:
        return dense_compare(args)
    if args.combine_only:
        return combine_only(args)
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
