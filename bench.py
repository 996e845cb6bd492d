#!/usr/bin/env python
"""Benchmark of the MXFP4 speculative-verification step on GB300.

One step = the verification pass of a Llama-3-8B-shaped decoder over MX-FP4
weights (32 layers x {QKV 4096->6144, O 4096->4096, gate+up 4096->28672,
down 14336->4096} + lm_head 4096->128256 = 129 verify GEMMs at
M = batch * (K_spec + 1) = 5) followed by spec_accept over the 128256-token
vocabulary.  Weights are random MX-FP4 (exponents 118..132), X ~ N(0, 1)
bf16, laws are softmaxed N(0, 2) logits; all synthetic and seeded.

Reported value: algorithmic bytes of the step (W + scales + X + Y of every GEMM,
plus the bytes spec_accept must read) / step time, in TB/s, with inputs
resident in HBM (the 3.99 GB of weights per step exceed the 129 MB L2, so no
flush is needed).  `e2e` repeats the step through the public API with the
step's inputs copied from pinned host memory and the emitted tokens copied
back inside the timed region.  `--impl reference` times the CPU oracle on a
bounded sample of the same workload.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mxs|reference]
                       [--workload llama8b|llama8b_b4|llama8b_b16|llama8b_b64|
                                   llama70b|llama70b_b1|llama70b_b4]
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "MXFP4 verify-GEMM achieved HBM TB/s (% of peak); spec_accept rows/sec"
FALLBACK_HBM_GBS = 6800.0

# Per-launch DRAM traffic of each verify-GEMM kernel (read + write bytes)
# divided by its algorithmic bytes, from the ncu captures summarised in
# profiles/, valid for the device sources of that kernel whose sha256 prefix,
# taken over the code with comments removed, is recorded beside it; traffic
# is reported as null otherwise (ratio None: not yet captured on the current
# sources).
GEMM_TRAFFIC = {
    # mxfp4_gemm_kernel, passes of <= 8 rows, as the step launches it: the grouped
    # instance over the 8B stack's first 8 layers (32 GEMMs, 936 MB) at M=5
    # (a single lm_head call at M=5 measured 1.0064)
    "mma": {"ratio": 1.0001, "sha": "d39faf7c557d3a85"},
    # mxfp4_gemm_bs_kernel, kind::mxf8f6f4 (passes of 33..64 rows): lm_head at M=64
    "bs8": {"ratio": 0.9171, "sha": "f1ace49f13d1d758"},
    # mxfp4_gemm_bs_kernel, kind::mxf4 (passes of 9..32 rows): lm_head at M=20
    "bs4": {"ratio": 0.9851, "sha": "f1ace49f13d1d758"},
    # mxfp4_gemm_bs_kernel, W4A4 (X quantised in the call, passes of <= 256 rows): lm_head at M=256
    "w4a4": {"ratio": 0.8927, "sha": "f1ace49f13d1d758"},
}
# sm__pipe_tensor_cycles_active (% of peak, elapsed) of each kernel, from the
# same captures as GEMM_TRAFFIC (keyed alike: None once the kernel changed)
GEMM_TENSOR_PCT = {
    "mma": 28.21,   # grouped instance, 8 layers at M=5
    "bs8": 37.94,   # lm_head at M=64
    "bs4": 34.30,   # lm_head at M=20
    "w4a4": 25.52,  # lm_head at M=256
}


def tensor_pct(passes):
    """Captured tensor-pipe activity of each pass's kernel, or None per kernel
    whose capture predates its current sources."""
    out = {}
    for rows, kind in passes:
        t = GEMM_TRAFFIC[kind]
        out[f"{rows} rows: {kind}"] = GEMM_TENSOR_PCT[kind] if t["sha"] == src_sha(kind) else None
    return out


BS_MIN_ROWS = 9     # passes of at least this many rows run on the block-scaled kernel
BS4_MAX_ROWS = 32   # its mxf4 kind takes passes of up to this many rows
GROUP_MAX = 84      # GEMMs per grouped launch at most (the problem table is a kernel parameter)

WORKLOADS = {
    # name: (model, B, K_spec)
    "llama8b": ("llama8b", 1, 4),
    "llama8b_b4": ("llama8b", 4, 4),
    "llama8b_b16": ("llama8b", 16, 4),
    "llama8b_b64": ("llama8b", 64, 4),
    "llama70b": ("llama70b", 16, 4),
    "llama70b_b1": ("llama70b", 1, 4),
    "llama70b_b4": ("llama70b", 4, 4),
}


def gemm_bytes(M: int, N: int, K: int) -> int:
    """Algorithmic bytes of one verify GEMM: W nibbles + E8M0 scales + bf16 X + fp32 Y."""
    return N * K // 2 + N * K // 32 + 2 * M * K + 4 * M * N


def accept_bytes(B: int, K: int, V: int, n_emitted: np.ndarray) -> int:
    """Bytes spec_accept must read/write: gathers, uniforms, ids, the sampled law
    (residual p_j, q_j when a draft was rejected, else p_K), outputs."""
    total = 0
    for b in range(B):
        j = int(n_emitted[b]) - 1
        law = 8 * V if j < K else 4 * V
        total += 8 * K + 4 * (K + 1) + 4 * K + law + 4 * (K + 1) + 4
    return total


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def in_process_peaks(mxs, torch, dev, nbytes: int = 2 << 30, reps: int = 5):
    """HBM figures measured in this process: the library's device copy kernel
    (read + write bytes) and its read-only probe, each over buffers far larger
    than L2.  Reported beside the MEASURED_PEAKS.json denominator."""
    src = torch.empty(nbytes // 4, dtype=torch.float32, device=dev)
    src.fill_(1.0)
    dst = torch.empty_like(src)
    sink = torch.zeros(4096, dtype=torch.int64, device=dev)
    out = {}
    for name, fn, moved in (("copy_gbs", lambda: mxs.hbm_copy_probe(dst, src), 2 * nbytes),
                            ("read_gbs", lambda: mxs.hbm_read_probe(src, sink), nbytes)):
        for _ in range(2):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize(dev)
        out[name] = moved * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9
    del src, dst
    return out


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of every rank's x (the whole job is as slow as its slowest rank)."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tbps(world: int, bytes_per_rank: float, seconds: float) -> float:
    """Whole-job throughput: every rank processes bytes_per_rank in the (max) time."""
    return world * bytes_per_rank / seconds / 1e12


def code_only(src: str) -> str:
    """C++ source without comments and blank lines (comment edits keep a kernel's key)."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in src.splitlines())
    return "\n".join(ln for ln in lines if ln)


# Device code each GEMM main kernel is built from (the host launchers in
# gemm.cu and the preparation kernel, a launch of its own, are not part of it).
KERNEL_SOURCES = {
    "mma": ("mxs_device.cuh", "gemm_common.cuh", "gemm_mma.cuh"),
    "bs8": ("mxs_device.cuh", "gemm_common.cuh", "gemm_bs.cuh"),
    "bs4": ("mxs_device.cuh", "gemm_common.cuh", "gemm_bs.cuh"),
    "w4a4": ("mxs_device.cuh", "gemm_common.cuh", "gemm_bs.cuh"),
}


def src_sha(kind: str, root: str = ROOT) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kind]:
        with open(os.path.join(root, "mxfp4_speculative_verification_gb300", "csrc", name)) as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


ACCEPT_LOGIT_STD = 3.0   # target logits N(0, 3) as in the acceptance-heavy configuration
ACCEPT_OVERLAP = 0.86    # mean per-token acceptance the pages report for code and math prompts
_SIGMA = {}


def draft_sigma() -> float:
    """Draft-logit noise giving a mean overlap sum_t min(p_t, q_t) of ACCEPT_OVERLAP."""
    if "s" not in _SIGMA:
        _SIGMA["s"] = workloads.tune_draft_noise(ACCEPT_OVERLAP, 4096, ACCEPT_LOGIT_STD, seed=0, samples=8)
    return _SIGMA["s"]


def compute_desc(kinds) -> str:
    """What the step computes in, for the kernels its passes use."""
    parts = []
    if "mma" in kinds:
        parts.append("E2M1 weights decoded exactly to fp16, X rows power-of-two scaled to fp16, "
                     "fp16 tensor-core products, fp32 accumulation")
    if "bs8" in kinds:
        parts.append("E2M1 weights x X as two E4M3 terms with UE8M0 block factors on the block-scaled "
                     "tensor core (kind::mxf8f6f4; exact for bf16 X within 2^16 of its block maximum), "
                     "fp32 accumulation")
    if "bs4" in kinds:
        parts.append("E2M1 weights x X as six E2M1 terms with UE8M0 block factors on the block-scaled "
                     "tensor core (kind::mxf4; X to within max|x|/4^6 of each 32-block), fp32 accumulation")
    parts.append("acceptance predicate exact (f64), sampling CDF in float-float above fp32 128-element sums")
    return "; ".join(parts)


def pass_traffic(shapes, passes, n_main):
    """DRAM bytes per grouped launch implied by the captured traffic ratios:
    every pass streams the whole W again plus its own X and Y rows, so a
    step of several passes moves more than its algorithmic bytes.  None when
    a kernel's ratio was not captured on its current sources."""
    total = 0.0
    for rows, kind in passes:
        t = GEMM_TRAFFIC[kind]
        if t["ratio"] is None or t["sha"] != src_sha(kind):
            return None
        total += t["ratio"] * sum(gemm_bytes(rows, N, K) for _, K, N in shapes)
    return total / n_main


def w4a4_passes(M: int):
    """Row passes of the W4A4 GEMM as the library plans them: as few as 256
    rows allow, of equal size rounded up to 16 (320 rows: 2 x 160)."""
    out, left = [], M
    while left > 0:
        n = -(-left // 256)
        rows = min(left, -(-(-(-left // n)) // 16) * 16)
        out.append((rows, "w4a4"))
        left -= rows
    return out


def gemm_passes(M: int):
    """Row passes of the grouped GEMM and the kernel of each, as the library
    plans them for K % 128 == 0: fewer than BS_MIN_ROWS rows left go to
    mma.sync, up to BS4_MAX_ROWS to the mxf4 kind, else 64 rows at a time to
    the mxf8f6f4 kind."""
    passes, m0 = [], 0
    while m0 < M:
        left = M - m0
        if left < BS_MIN_ROWS:
            passes.append((min(64, left), "mma"))
        elif left <= BS4_MAX_ROWS:
            passes.append((left, "bs4"))
        else:
            passes.append((min(64, left), "bs8"))
        m0 += passes[-1][0]
    return passes


# ----------------------------------------------------------------------------
# CPU oracle timings (the reference arm and the cpu_baseline leg)
# ----------------------------------------------------------------------------
def oracle_sample(model: str, M: int, B: int, K_spec: int, target_s: float):
    """Time the oracle on whole layers of the stack (plus the lm_head and one
    acceptance row per sequence) until about target_s seconds of work.
    Returns (bytes, seconds, rows_per_s, description, threads)."""
    import oracle

    oracle.build()
    threads = oracle.default_threads()
    shapes = workloads.stack_shapes(model)
    layer = shapes[:4]
    head = shapes[-1]
    total_b, total_t, n_layers = 0, 0.0, 0
    x_cache = {}
    while True:
        for li, (_, K, N) in enumerate(layer):
            nib, sc = workloads.mxfp4_weights(N, K, *workloads.LLAMA_EXP_RANGE, seed=n_layers, tensor_id=li)
            if K not in x_cache:
                x_cache[K] = workloads.bf16_normal(M, K, seed=0, tensor_id=K)
            t0 = time.perf_counter()
            oracle.gemm(x_cache[K], nib, sc, nthreads=threads)
            total_t += time.perf_counter() - t0
            total_b += gemm_bytes(M, N, K)
        n_layers += 1
        if total_t >= target_s or n_layers >= 2:
            break
    # a slice of the lm_head rows
    _, K, N = head
    rows = max(1024, int(N * min(1.0, 0.25 * target_s / max(total_t, 1e-3))))
    rows = min(rows, N)
    nib, sc = workloads.mxfp4_weights(rows, K, *workloads.LLAMA_EXP_RANGE, seed=99, tensor_id=9)
    t0 = time.perf_counter()
    oracle.gemm(x_cache.get(K, workloads.bf16_normal(M, K, seed=0, tensor_id=K)), nib, sc, nthreads=threads)
    total_t += time.perf_counter() - t0
    total_b += gemm_bytes(M, rows, K)
    # acceptance rows
    V = workloads.VOCAB_LLAMA
    p, q, d, u = workloads.spec_inputs(B, K_spec, V, seed=0, logit_std=2.0)
    t0 = time.perf_counter()
    _, n, _, _ = oracle.spec_accept(p, q, d, u, nthreads=threads)
    ta = time.perf_counter() - t0
    total_t += ta
    total_b += accept_bytes(B, K_spec, V, n)
    desc = (f"{n_layers} full layer(s) of 4 GEMMs + {rows} of {N} lm_head rows at M={M}, "
            f"plus spec_accept over {B} row(s), V={V}")
    return total_b, total_t, B / ta, desc, threads


def run_reference(args, world, rank):
    if rank != 0:
        return
    model, B, K_spec = WORKLOADS[args.workload]
    M = B * (K_spec + 1)
    times, bytes_ = [], 0
    desc, threads, rows_s = "", 1, 0.0
    for it in range(args.warmup + args.steps):
        b, t, rs, desc, threads = oracle_sample(model, M, B, K_spec, target_s=1.0)
        if it >= args.warmup:
            times.append(t)
            bytes_ = b
            rows_s = rs
    t_step = statistics.mean(times)
    value = bytes_ / t_step / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(args.workload, model, B, K_spec),
        "cpu_baseline": {"value": value, "unit": "TB/s", "cores": threads, "kind": "oracle",
                         "sample": desc},
        "spec_accept_rows_per_s": rows_s,
        "e2e": {"value": value, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_block(name, model, B, K_spec):
    shapes = workloads.stack_shapes(model)
    M = B * (K_spec + 1)
    wbytes = sum(N * K // 2 + N * K // 32 for _, K, N in shapes)
    return {"workload": f"{name}: {model}-shaped verification step, {len(shapes)} MXFP4 GEMMs at "
                        f"M={M} (B={B}, K_spec={K_spec}) + spec_accept V={workloads.VOCAB_LLAMA}",
            "gemms": len(shapes), "M": M, "B": B, "K_spec": K_spec, "V": workloads.VOCAB_LLAMA,
            "weight_bytes_per_step": wbytes,
            "l2": "weights per step exceed the 129 MB L2 (each GEMM's W is read once): no flush"}


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------
def run_mxs(args, world, rank, local):
    import torch

    import mxfp4_speculative_verification_gb300 as mxs

    mxs.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    model, B, K_spec = WORKLOADS[args.workload]
    M = B * (K_spec + 1)
    V = workloads.VOCAB_LLAMA
    shapes = workloads.stack_shapes(model)
    lo, hi = workloads.LLAMA_EXP_RANGE

    # resident weights, one distinct MXFP4 matrix per GEMM
    weights = []
    for i, (_, K, N) in enumerate(shapes):
        weights.append(workloads.device_mxfp4_weights(N, K, lo, hi, seed=1000 * rank + i, device=dev))
    ks = sorted({K for _, K, _ in shapes})
    x_host = {K: torch.from_numpy(workloads.bf16_normal(M, K, seed=rank, tensor_id=K).view(np.int16))
              .view(torch.bfloat16).pin_memory() for K in ks}
    x_dev = {K: x_host[K].to(dev) for K in ks}
    # one output per GEMM (they are independent problems of the step)
    ys = [torch.empty((M, N), dtype=torch.float32, device=dev) for _, _, N in shapes]
    ws_bytes = max(mxs.mxfp4_verify_gemm_workspace_size(M, N, K) for _, K, N in shapes)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    problems = [(x_dev[K], nib, sc, y) for (_, K, _), (nib, sc), y in zip(shapes, weights, ys)]
    gws = torch.empty(mxs.mxfp4_verify_gemm_grouped_workspace_size(problems), dtype=torch.uint8,
                      device=dev)
    # acceptance inputs as in the pages' workloads: draft law = target law with
    # noise tuned to a mean per-token overlap of 0.86, drafts drawn from it
    sigma = draft_sigma()
    p, q, d, u = workloads.spec_inputs(B, K_spec, V, seed=rank, logit_std=ACCEPT_LOGIT_STD, draft_noise=sigma)
    alpha = float(np.minimum(p[:, :K_spec, :].astype(np.float64), q.astype(np.float64)).sum(axis=-1).mean())
    acc_host = [torch.from_numpy(a).pin_memory() for a in (p, q, d, u)]
    acc_dev = [a.to(dev) for a in acc_host]
    out_tok = torch.empty((B, K_spec + 1), dtype=torch.int32, device=dev)
    n_emit = torch.empty((B,), dtype=torch.int32, device=dev)
    tok_host = torch.empty_like(out_tok, device="cpu").pin_memory()
    n_host = torch.empty_like(n_emit, device="cpu").pin_memory()

    def gemms_grouped():
        mxs.mxfp4_verify_gemm_grouped(problems, workspace=gws)

    def gemms_per_call():
        for (_, K, N), (nib, sc), y in zip(shapes, weights, ys):
            mxs.mxfp4_verify_gemm(x_dev[K], nib, sc, out=y, workspace=ws)

    def accept(reps=1):
        for _ in range(reps):
            mxs.spec_accept(*acc_dev, out_tokens=out_tok, n_emitted=n_emit)

    def step():
        gemms_grouped()
        accept()

    def step_per_call():
        gemms_per_call()
        accept()

    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream(dev))  # inputs were made on the current stream
    ACC_REPS = 20
    graphs = {}
    with torch.cuda.stream(stream):
        step()  # eager warm-up: kernel attributes, first launches
        step_per_call()
        torch.cuda.synchronize(dev)
        n_emitted = n_emit.cpu().numpy()
        for name, fn in (("step", step), ("step_pc", step_per_call), ("gemm", gemms_grouped),
                         ("gemm_pc", gemms_per_call), ("acc", lambda: accept(ACC_REPS))):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            graphs[name] = g
    torch.cuda.synchronize(dev)

    gemm_b = sum(gemm_bytes(M, N, K) for _, K, N in shapes)
    acc_b = accept_bytes(B, K_spec, V, n_emitted)
    step_b = gemm_b + acc_b

    def timed(graph, steps):
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                graph.replay()
            torch.cuda.synchronize(dev)
            if world > 1:
                torch.distributed.barrier()
            ev0.record(stream)
            for _ in range(steps):
                graph.replay()
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        return max_over_ranks(ev0.elapsed_time(ev1), world, dev) / steps

    clocks = ClockSampler(local)
    clocks.start()
    ms_step = timed(graphs["step"], args.steps)
    ms_gemm = timed(graphs["gemm"], args.steps)
    ms_step_pc = timed(graphs["step_pc"], args.steps)
    ms_gemm_pc = timed(graphs["gemm_pc"], args.steps)
    ms_acc = timed(graphs["acc"], args.steps) / ACC_REPS
    clk = clocks.stop()

    # end to end through the public API: pinned host inputs in, tokens out
    # A pipelined serving loop: every step uploads its inputs and reads its
    # tokens back, on a second (copy) stream that overlaps the GEMMs.  Step k
    # uploads the laws its acceptance reads and the X of step k + 1 (X is
    # double-buffered), once step k - 1 is done with both buffers; its GEMMs
    # read the X that step k - 1 uploaded; acceptance waits for the laws; the
    # tokens go back once acceptance is done.
    copy_stream = torch.cuda.Stream(device=dev)
    x_bufs = [x_dev, {K: torch.empty_like(x_dev[K]) for K in ks}]
    grouped_for = [mxs.GroupedGemm(problems, workspace=gws),
                   mxs.GroupedGemm([(x_bufs[1][K], nib, sc, y)
                                    for (_, K, _), (nib, sc), y in zip(shapes, weights, ys)], workspace=gws)]
    e2e_k = [0]

    def e2e_step():
        k = e2e_k[0]
        e2e_k[0] += 1
        copy_stream.wait_stream(stream)
        with torch.cuda.stream(copy_stream):
            for a_d, a_h in zip(acc_dev, acc_host):
                a_d.copy_(a_h, non_blocking=True)
            nxt = x_bufs[(k + 1) % 2]
            for K in ks:
                nxt[K].copy_(x_host[K], non_blocking=True)
        grouped_for[k % 2]()
        stream.wait_stream(copy_stream)
        accept()
        copy_stream.wait_stream(stream)
        with torch.cuda.stream(copy_stream):
            tok_host.copy_(out_tok, non_blocking=True)
            n_host.copy_(n_emit, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            e2e_step()
        torch.cuda.synchronize(dev)
        e2e_s = (time.perf_counter() - t0) / args.steps
    e2e_s = max_over_ranks(e2e_s, world, dev)
    h2d = sum(x_host[K].numel() * 2 for K in ks) + sum(a.numel() * a.element_size() for a in acc_host)
    d2h = tok_host.numel() * 4 + n_host.numel() * 4

    peak, peak_kind = load_peaks()
    inproc = in_process_peaks(mxs, torch, dev) if rank == 0 else None
    achieved_gbs = gemm_b / (ms_gemm * 1e-3) / 1e9
    passes = gemm_passes(M)
    n_main = len(passes) * ((len(shapes) + GROUP_MAX - 1) // GROUP_MAX)  # grouped launches
    n_prep = len(passes) * ((len(ks) + 15) // 16)      # one X preparation per pass
    kinds = sorted({k for _, k in passes})
    kernel_name = {"mma": "mxfp4_gemm_kernel (mma.sync)",
                   "bs8": "mxfp4_gemm_bs_kernel (tcgen05 kind::mxf8f6f4 block-scaled)",
                   "bs4": "mxfp4_gemm_bs_kernel (tcgen05 kind::mxf4 block-scaled)"}
    traffic = pass_traffic(shapes, passes, n_main)

    if args.detail and rank == 0:
        per_shape_detail(mxs, torch, stream, dev, shapes, weights, x_dev, ws, M)

    # the other configurations, each timed the same way (weights of the same
    # stack reused; the 70B stack generated once on the device)
    sweep, acc_sweep, logits_acc, nv, kvc, w4 = [], None, None, None, None, None
    if not args.no_sweep and rank == 0 and world == 1:
        wcache = {model: weights}
        clocks2 = ClockSampler(local)
        clocks2.start()
        for wl in SWEEP_WORKLOADS:
            if wl == args.workload:
                continue
            m2, b2, k2 = WORKLOADS[wl]
            if m2 not in wcache:
                wcache[m2] = [workloads.device_mxfp4_weights(N, K, lo, hi, seed=i, device=dev)
                              for i, (_, K, N) in enumerate(workloads.stack_shapes(m2))]
            sweep.append(sweep_point(mxs, torch, dev, stream, wl, wcache[m2], args, peak_for_sweep()))
            if wl in W4A4_SWEEP:
                sweep.append(sweep_point(mxs, torch, dev, stream, wl, wcache[m2], args, peak_for_sweep(), w4a4=True))
        clk2 = clocks2.stop()
        for rec in sweep:
            rec["clocks"] = clk2
        del wcache
        torch.cuda.empty_cache()
        acc_sweep = accept_sweep_rows(mxs, torch, dev, peak)
        logits_acc = logits_accept_rows(mxs, torch, dev, peak)
        nv = nvfp4_rows(mxs, torch, dev, peak)
        kvc = kv_cache_rows(mxs, torch, dev, peak)
        w4 = w4a4_rows(mxs, torch, dev, peak)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        b, t, rs, desc, threads = oracle_sample(model, M, B, K_spec, target_s=args.cpu_seconds)
        cpu = {"value": b / t / 1e12, "unit": "TB/s", "cores": threads, "kind": "oracle",
               "sample": desc, "spec_accept_rows_per_s": rs}

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    value = job_tbps(world, step_b, ms_step * 1e-3)
    line = {
        "metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32",
        "compute": compute_desc(kinds),
        "data": "synthetic",
        "config": config_block(args.workload, model, B, K_spec),
        "pct_of_peak": value * 1e3 / peak / world,
        "roofline": {"bound": "hbm",
                     "kernel": " + ".join(f"{kernel_name[k]} for {r} rows" for r, k in passes)
                               + " (grouped launches, incl. X preparation)",
                     "achieved": achieved_gbs, "peak": peak, "unit": "GB/s",
                     "frac": achieved_gbs / peak, "peak_source": f"{peak_kind} hbm_gbs",
                     "bytes_per_launch": gemm_b / n_main, "launches_per_step": n_main,
                     "avg_launch_us": ms_gemm * 1e3 / n_main, "traffic": traffic,
                     "tensor_pipe_pct_captured": tensor_pct(passes)},
        "per_call": {"value": job_tbps(world, step_b, ms_step_pc * 1e-3), "unit": "TB/s",
                     "ms_per_step": ms_step_pc,
                     "gemm_gbs": gemm_b / (ms_gemm_pc * 1e-3) / 1e9,
                     "path": "one mxfp4_verify_gemm call per GEMM (prep + main kernel each), "
                             "CUDA graph with programmatic dependent launch"},
        "spec_accept": {"rows_per_s": B / (ms_acc * 1e-3), "us_per_call": ms_acc * 1e3,
                        "bytes_per_call": acc_b, "mean_emitted": float(np.mean(n_emitted)),
                        "mean_overlap": alpha,
                        "closed_form_emitted": (1.0 - alpha ** (K_spec + 1)) / (1.0 - alpha),
                        "inputs": f"target logits N(0,{ACCEPT_LOGIT_STD:g}), draft = target + N(0,{sigma:.3f}) "
                                  f"(mean overlap {ACCEPT_OVERLAP}), drafts drawn from the draft law",
                        "timing": f"{ACC_REPS} calls on the same inputs in one CUDA graph (L2-warm: "
                                  f"{acc_b / 1e6:.1f} MB read per call); latency-bound at this batch",
                        "pct_of_peak": acc_b / (ms_acc * 1e-3) / 1e9 / peak},
        "e2e": {"value": job_tbps(world, step_b, e2e_s), "unit": "TB/s",
                "ms_per_step": e2e_s * 1e3, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "path": "public Python API -> C ABI (GroupedGemm plans: the problems checked once, one C call "
                        "a step), eager launches, pinned host copies every step on a copy stream overlapping the "
                        "GEMMs (the laws and the next step's X, double-buffered; tokens back after acceptance)"},
        "gpu_launches": args.steps * (n_prep + n_main + 1),
        "clocks": clk,
        "cpu_baseline": cpu,
        "peaks_in_process": inproc,
        "sweep": sweep,
        "accept_sweep": acc_sweep,
        "accept_logits": logits_acc,
        "nvfp4_lm_head": nv,
        "kv_cache": kvc,
        "w4a4": w4,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# The configurations reported beside the headline (each a sub-record of the
# same JSON line): the 8B batch sweep and the 70B stack at three batch sizes.
SWEEP_WORKLOADS = ("llama8b_b4", "llama8b_b16", "llama8b_b64", "llama70b_b1", "llama70b_b4", "llama70b")
# of which these are also run in the grouped W4A4 form (beside the W4A16 step)
W4A4_SWEEP = SWEEP_WORKLOADS


def peak_for_sweep() -> float:
    return load_peaks()[0]


def sweep_point(mxs, torch, dev, stream, wl, weights, args, peak, w4a4=False):
    """One configuration: its grouped GEMM step and its acceptance call, each
    captured in a CUDA graph and timed with CUDA events after warm-up (w4a4:
    the grouped W4A4 form, X quantised to MX-FP4, passes of up to 256 rows)."""
    model, B, K_spec = WORKLOADS[wl]
    M = B * (K_spec + 1)
    V = workloads.VOCAB_LLAMA
    shapes = workloads.stack_shapes(model)
    ks = sorted({K for _, K, _ in shapes})
    x_dev = {K: workloads.device_bf16_normal(M, K, seed=K, device=dev) for K in ks}
    ys = [torch.empty((M, N), dtype=torch.float32, device=dev) for _, _, N in shapes]
    problems = [(x_dev[K], nib, sc, y) for (_, K, _), (nib, sc), y in zip(shapes, weights, ys)]
    gws = torch.empty(mxs.mxfp4_verify_gemm_grouped_workspace_size(problems, w4a4=w4a4), dtype=torch.uint8,
                      device=dev)
    p, q, d, u = workloads.spec_inputs(B, K_spec, V, seed=1, logit_std=ACCEPT_LOGIT_STD, draft_noise=draft_sigma())
    acc = [torch.from_numpy(a).to(dev) for a in (p, q, d, u)]
    out_tok = torch.empty((B, K_spec + 1), dtype=torch.int32, device=dev)
    n_emit = torch.empty((B,), dtype=torch.int32, device=dev)
    reps = 10
    with torch.cuda.stream(stream):
        mxs.mxfp4_verify_gemm_grouped(problems, workspace=gws, w4a4=w4a4)
        mxs.spec_accept(*acc, out_tokens=out_tok, n_emitted=n_emit)
        torch.cuda.synchronize(dev)
        n_emitted = n_emit.cpu().numpy()
        g_gemm, g_acc = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_gemm, stream=stream):
            mxs.mxfp4_verify_gemm_grouped(problems, workspace=gws, w4a4=w4a4)
        with torch.cuda.graph(g_acc, stream=stream):
            for _ in range(reps):
                mxs.spec_accept(*acc, out_tokens=out_tok, n_emitted=n_emit)
    torch.cuda.synchronize(dev)

    def timed(graph, steps):
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                graph.replay()
            torch.cuda.synchronize(dev)
            ev0.record(stream)
            for _ in range(steps):
                graph.replay()
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        return ev0.elapsed_time(ev1) / steps

    steps = max(3, min(args.steps, 10))
    ms_gemm = timed(g_gemm, steps)
    ms_acc = timed(g_acc, steps) / reps
    gemm_b = sum(gemm_bytes(M, N, K) for _, K, N in shapes)
    acc_b = accept_bytes(B, K_spec, V, n_emitted)
    passes = w4a4_passes(M) if w4a4 else gemm_passes(M)
    n_main = len(passes) * ((len(shapes) + GROUP_MAX - 1) // GROUP_MAX)
    gbs = gemm_b / (ms_gemm * 1e-3) / 1e9
    flops = sum(2 * M * N * K for _, K, N in shapes)
    alpha = float(np.minimum(p[:, :K_spec, :].astype(np.float64), q.astype(np.float64)).sum(axis=-1).mean())
    kinds = sorted({k for _, k in passes})
    traffic = pass_traffic(shapes, passes, n_main)
    del x_dev, ys, problems, gws, acc
    return {
        "workload": config_block(wl, model, B, K_spec)["workload"]
                    + (" (W4A4: X quantised to MX-FP4 by the pack rule)" if w4a4 else ""),
        "mode": "w4a4" if w4a4 else "w4a16", "M": M,
        "ms_per_step": ms_gemm + ms_acc, "value": (gemm_b + acc_b) / ((ms_gemm + ms_acc) * 1e-3) / 1e12,
        "unit": "TB/s", "steps": steps,
        "passes": [f"{r} rows: {k}" for r, k in passes],
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "bytes_per_launch": gemm_b / n_main, "launches_per_step": n_main,
                     "avg_launch_us": ms_gemm * 1e3 / n_main, "traffic": traffic,
                     "useful_tflops": flops / (ms_gemm * 1e-3) / 1e12,
                     "tensor_pipe_pct_captured": tensor_pct(passes)},
        "spec_accept": {"B": B, "us_per_call": ms_acc * 1e3, "rows_per_s": B / (ms_acc * 1e-3),
                        "mean_emitted": float(np.mean(n_emitted)), "mean_overlap": alpha,
                        "closed_form_emitted": (1.0 - alpha ** (K_spec + 1)) / (1.0 - alpha),
                        "pct_of_peak": acc_b / (ms_acc * 1e-3) / 1e9 / peak},
    }


def per_shape_detail(mxs, torch, stream, dev, shapes, weights, x_dev, ws, M):
    """Per-shape GEMM bandwidth (stderr), each shape timed over all its layers."""
    seen = {}
    for i, (name, K, N) in enumerate(shapes):
        seen.setdefault((K, N), []).append(i)
    for (K, N), idx in seen.items():
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in idx:
                    mxs.mxfp4_verify_gemm(x_dev[K], *weights[i], out=y, workspace=ws)
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            reps = 10
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) * 1e3 / (reps * len(idx))
        gbs = gemm_bytes(M, N, K) / (us * 1e-6) / 1e9
        print(f"detail K={K} N={N} M={M}: {us:.2f} us/launch, {gbs:.0f} GB/s", file=sys.stderr)


def profile_target(args):
    """A few launches of one kernel, for ncu (no timing, no JSON)."""
    import torch

    import mxfp4_speculative_verification_gb300 as mxs

    mxs.build()
    dev = torch.device("cuda:0")
    model, B, K_spec = WORKLOADS[args.workload]
    M = args.profile_m or B * (K_spec + 1)
    if args.profile_grouped:
        # the first LAYERS layers of the stack (4 GEMMs each) in one grouped
        # launch: the kernel instance of the step's grouped launches, small
        # enough for a counter capture
        shapes = workloads.stack_shapes(model)[: 4 * args.profile_grouped]
        lo, hi = workloads.LLAMA_EXP_RANGE
        xs = {K: workloads.device_bf16_normal(M, K, seed=K, device=dev) for K in sorted({K for _, K, _ in shapes})}
        problems = []
        for i, (_, K, N) in enumerate(shapes):
            nib, sc = workloads.device_mxfp4_weights(N, K, lo, hi, seed=i, device=dev)
            problems.append((xs[K], nib, sc, torch.empty((M, N), dtype=torch.float32, device=dev)))
        w4 = bool(args.profile_w4a4)
        ws = torch.empty(mxs.mxfp4_verify_gemm_grouped_workspace_size(problems, w4a4=w4), dtype=torch.uint8,
                         device=dev)
        for _ in range(4):
            mxs.mxfp4_verify_gemm_grouped(problems, workspace=ws, w4a4=w4)
    elif args.profile_gemm:
        K, N = (int(v) for v in args.profile_gemm.split(","))
        x = workloads.device_bf16_normal(M, K, seed=1, device=dev)
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        if args.profile_nvfp4:
            nib, sc = workloads.device_nvfp4_weights(N, K, seed=0, device=dev)
            for _ in range(4):
                mxs.nvfp4_verify_gemm(x, nib, sc, 0.0731, out=y)
        elif args.profile_w4a4:
            nib, sc = workloads.device_mxfp4_weights(N, K, *workloads.LLAMA_EXP_RANGE, seed=0, device=dev)
            for _ in range(4):
                mxs.mxfp4_verify_gemm_w4a4(x, nib, sc, out=y)
        else:
            nib, sc = workloads.device_mxfp4_weights(N, K, *workloads.LLAMA_EXP_RANGE, seed=0, device=dev)
            for _ in range(4):
                mxs.mxfp4_verify_gemm(x, nib, sc, out=y)
    elif args.profile_law:
        # the sampling law of the workload's B (K + 1) target rows, T = 0.8, top-p 0.9
        gen = torch.Generator(device=dev)
        gen.manual_seed(0)
        logits = torch.randn((B * (K_spec + 1), workloads.VOCAB_LLAMA), generator=gen, device=dev) * 3.0
        out = torch.empty_like(logits)
        for _ in range(4):
            mxs.spec_sampling_law(logits, out=out, **LOGITS_SAMPLING)
    else:
        V = workloads.VOCAB_LLAMA
        p, q, d, u = (torch.from_numpy(a).to(dev) for a in workloads.spec_inputs(
            B, K_spec, V, seed=0, logit_std=ACCEPT_LOGIT_STD, draft_noise=draft_sigma()))
        for _ in range(4):
            mxs.spec_accept(p, q, d, u)
    torch.cuda.synchronize()


ACCEPT_SETS = 4  # input copies the acceptance sweep rotates through (cold L2)


def accept_sweep_rows(mxs, torch, dev, peak, max_rounds=1500):
    """Acceptance-heavy sweep: B=64, K in {1,3,7}, V=128256, target logits N(0,3),
    draft logits = target + N(0, sigma) with sigma bisected so that the mean
    overlap sum_t min(p_t, q_t) is about 0.86.  p and q are drawn once per K;
    drafts (sampled from q on the device) and uniforms are redrawn every round
    until the standard error of the mean emitted count is below 0.01.  Reports
    the mean against the closed form (1 - a^(K+1)) / (1 - a) at the mean overlap
    a, and against the exact tail sum over each row's own overlaps,
    E_b = sum_k prod_{i<k} a_{b,i}."""
    B, V, std = 64, workloads.VOCAB_LLAMA, ACCEPT_LOGIT_STD
    sigma = draft_sigma()
    rows = []
    for K in (1, 3, 7):
        p, q, _, _ = workloads.spec_inputs(B, K, V, seed=100 + K, logit_std=std, draft_noise=sigma)
        alpha = np.minimum(p[:, :K, :].astype(np.float64), q.astype(np.float64)).sum(axis=-1)  # [B, K]
        tail = np.concatenate([np.ones((B, 1)), np.cumprod(alpha, axis=1)], axis=1).sum(axis=1)
        a_mean = float(alpha.mean())
        closed = (1.0 - a_mean ** (K + 1)) / (1.0 - a_mean)
        p_d, q_d = torch.from_numpy(p).to(dev), torch.from_numpy(q).to(dev)
        q_rows = q_d.view(B * K, V)
        out_tok = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
        n_emit = torch.empty((B,), dtype=torch.int32, device=dev)
        gen = torch.Generator(device=dev)
        gen.manual_seed(200 + K)
        counts = []
        rounds = 0
        while True:
            rounds += 1
            d_d = torch.multinomial(q_rows, 1, generator=gen).view(B, K).to(torch.int32)
            u_d = torch.rand((B, K + 1), generator=gen, device=dev, dtype=torch.float32)
            mxs.spec_accept(p_d, q_d, d_d, u_d, out_tokens=out_tok, n_emitted=n_emit)
            counts.append(n_emit.to(torch.float64))
            if rounds >= 4 and (rounds % 16 == 0 or rounds >= max_rounds):
                allc = torch.cat(counts).cpu().numpy()
                se = float(allc.std(ddof=1) / np.sqrt(allc.size))
                if se < 0.01 or rounds >= max_rounds:
                    break
        # timing on the last round's inputs, cold in L2: ACCEPT_SETS copies of
        # p and q rolled along the vocabulary (drafts shifted alike, so every
        # call takes the same decisions on other memory), called in turn in one
        # CUDA graph; more than 200 MB are read between two calls on a copy
        sets = []
        for k in range(ACCEPT_SETS):
            sh = 1009 * k
            sets.append((torch.roll(p_d, sh, dims=-1), torch.roll(q_d, sh, dims=-1),
                         ((d_d + sh) % V).to(torch.int32), u_d, torch.empty_like(out_tok), torch.empty_like(n_emit)))
        mxs.spec_accept(*sets[0][:4], out_tokens=sets[0][4], n_emitted=sets[0][5])

        def calls():
            for ps, qs, ds, us_, ot, ne in sets:
                mxs.spec_accept(ps, qs, ds, us_, out_tokens=ot, n_emitted=ne)

        us = graph_us(torch, dev, calls, reps=10) / ACCEPT_SETS
        n_set = sets[0][5].cpu().numpy()
        assert np.array_equal(n_set, n_emit.cpu().numpy()), "rolled copies take the same decisions"
        nb = accept_bytes(B, K, V, n_set)
        del sets
        rows.append({"K": K, "rows": int(allc.size), "rounds": rounds,
                     "mean_emitted": float(allc.mean()), "std_error": se,
                     "mean_overlap": a_mean, "closed_form": closed,
                     "exact_tail_sum": float(tail.mean()),
                     "z_vs_tail_sum": float((allc.mean() - tail.mean()) / se),
                     "us_per_call": us, "rows_per_s": B / (us * 1e-6),
                     "hbm_gbs": nb / (us * 1e-6) / 1e9, "pct_of_peak": nb / (us * 1e-6) / 1e9 / peak})
        del p_d, q_d, q_rows
    return {"metric": "spec_accept acceptance-heavy sweep (mean emitted tokens per step)",
            "B": B, "V": V, "logit_std": std, "draft_noise_sigma": sigma,
            "drafts": "sampled from q on the device (torch.multinomial), uniforms torch.rand",
            "timing": f"CUDA-graph replays of {ACCEPT_SETS} calls on copies of p, q rolled along V "
                      "(same decisions, other memory): cold L2",
            "rows": rows}


LOGITS_SAMPLING = {"temperature": 0.8, "top_k": 0, "top_p": 0.9}


def logits_accept_rows(mxs, torch, dev, peak, reps=20):
    """Acceptance from logits (laws formed on the device, temperature 0.8 and
    top-p 0.9 on the target and the draft alike), B = 1 / 16 / 64, K = 4,
    V = 128256.  Target logits N(0, 3), draft logits = target + N(0, 0.4),
    drafts sampled from the draft's transformed law.  Algorithmic bytes: every
    logit row read once (the statistics pass) plus the rows the acceptance
    reads again (the rejected position's pair, or the bonus row), ids,
    uniforms and outputs."""
    V, K = workloads.VOCAB_LLAMA, 4
    rows = []
    for B in (1, 16, 64):
        gen = torch.Generator(device=dev)
        gen.manual_seed(300 + B)
        tl = torch.randn((B, K + 1, V), generator=gen, device=dev) * 3.0
        dl = tl[:, :K] + torch.randn((B, K, V), generator=gen, device=dev) * 0.4
        q = mxs.spec_sampling_law(dl.contiguous(), **LOGITS_SAMPLING)
        d = torch.multinomial(q.view(B * K, V), 1, generator=gen).view(B, K).to(torch.int32)
        u = torch.rand((B, K + 1), generator=gen, device=dev)
        dlc = dl.contiguous()
        ws = torch.empty(mxs.spec_accept_logits_workspace_size(B, K), dtype=torch.uint8, device=dev)
        out_tok = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
        n_emit = torch.empty((B,), dtype=torch.int32, device=dev)
        call = lambda: mxs.spec_accept_logits(tl, dlc, d, u, workspace=ws, out_tokens=out_tok, n_emitted=n_emit,
                                              **LOGITS_SAMPLING)
        us = graph_us(torch, dev, call, reps)
        n = n_emit.cpu().numpy()
        nb = 4 * B * (2 * K + 1) * V + accept_bytes(B, K, V, n)
        rows.append({"B": B, "K": K, "us_per_call": us, "rows_per_s": B / (us * 1e-6),
                     "mean_emitted": float(n.mean()), "bytes_per_call": nb,
                     "hbm_gbs": nb / (us * 1e-6) / 1e9, "pct_of_peak": nb / (us * 1e-6) / 1e9 / peak})
        del tl, dl, dlc, q, d, u, ws
    return {"metric": "spec_accept_logits: laws from logits (statistics pass + acceptance), us per call",
            "V": V, "sampling": LOGITS_SAMPLING,
            "timing": "CUDA-graph replays on the same inputs: the logit rows (4.6 / 74 / 295 MB at B = 1 / 16 / "
                      "64) stay in L2 between calls at B = 1 and 16; at B = 64 they exceed it",
            "rows": rows}


def graph_us(torch, dev, fn, reps=20, warm=3):
    """Device time of fn (its launches captured in a CUDA graph, so host
    launch overhead is left out), averaged over reps replays."""
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream(dev))  # fn's inputs come from the current stream
    with torch.cuda.stream(stream):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        for _ in range(warm):
            g.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) * 1e3 / reps


def nvfp4_rows(mxs, torch, dev, peak, reps=20):
    """The lm_head of the 8B stack (K = 4096, N = 128256) on NVFP4 weights
    (E4M3 scale per 16 elements, one FP32 tensor scale) at M = 5 / 20 / 64,
    beside the same shape on MXFP4.  Weights and scales (296 MB NVFP4) exceed
    L2, so back-to-back calls stream them from HBM.  Algorithmic bytes:
    nibbles + scale bytes + X (bf16) + Y (fp32)."""
    N, K = workloads.VOCAB_LLAMA, 4096
    nib, sc = workloads.device_nvfp4_weights(N, K, seed=71, device=dev)
    mnib, msc = workloads.device_mxfp4_weights(N, K, *workloads.LLAMA_EXP_RANGE, seed=71, device=dev)
    rows = []
    for M in (5, 20, 64):
        x = workloads.device_bf16_normal(M, K, seed=72 + M, device=dev)
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        for fmt in ("nvfp4", "mxfp4"):
            if fmt == "nvfp4":
                ws = torch.empty(mxs.nvfp4_verify_gemm_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
                call = lambda: mxs.nvfp4_verify_gemm(x, nib, sc, 0.0731, out=y, workspace=ws)
                nb = N * K // 2 + N * K // 16 + M * K * 2 + M * N * 4
            else:
                ws = torch.empty(mxs.mxfp4_verify_gemm_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
                call = lambda: mxs.mxfp4_verify_gemm(x, mnib, msc, out=y, workspace=ws)
                nb = gemm_bytes(M, N, K)
            for _ in range(5):
                call()
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                call()
            e1.record()
            torch.cuda.synchronize(dev)
            us = e0.elapsed_time(e1) * 1e3 / reps
            rows.append({"format": fmt, "M": M, "us_per_call": us, "bytes_per_call": nb,
                         "hbm_gbs": nb / (us * 1e-6) / 1e9, "pct_of_peak": nb / (us * 1e-6) / 1e9 / peak})
            del ws
        del x, y
    del nib, sc, mnib, msc
    torch.cuda.empty_cache()
    return {"metric": "lm_head GEMM (K=4096, N=128256), one call incl. X preparation, us per call",
            "timing": "back-to-back calls; the weights (279 / 296 MB) exceed L2", "rows": rows}


def w4a4_rows(mxs, torch, dev, peak, reps=20):
    """W4A4 (X quantised to MX-FP4 by the pack rule inside the call, block-
    scaled kind::mxf4 product, passes of up to 256 rows) beside the W4A16
    entry point on the same MXFP4 weights: the 8B lm_head (K = 4096,
    N = 128256, 279 MB, beyond L2) at M = 80 / 160 / 256 / 320, back-to-back
    calls; and the whole 8B stack (32 layers x 4 GEMMs + lm_head, 4.3 GB) at
    M = 80 / 256 / 320 as grouped plans, and at M = 80 one call per GEMM, in
    CUDA graphs.  Algorithmic bytes as
    for the verify GEMM: nibbles + scales + bf16 X + fp32 Y."""
    N, K = workloads.VOCAB_LLAMA, 4096
    lo, hi = workloads.LLAMA_EXP_RANGE
    nib, sc = workloads.device_mxfp4_weights(N, K, lo, hi, seed=81, device=dev)
    rows = []
    for M in (80, 160, 256, 320):
        x = workloads.device_bf16_normal(M, K, seed=82 + M, device=dev)
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        for mode in ("w4a4", "w4a16"):
            if mode == "w4a4":
                ws = torch.empty(mxs.mxfp4_verify_gemm_w4a4_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
                call = lambda: mxs.mxfp4_verify_gemm_w4a4(x, nib, sc, out=y, workspace=ws)
                w_passes = len(w4a4_passes(M))
            else:
                ws = torch.empty(mxs.mxfp4_verify_gemm_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
                call = lambda: mxs.mxfp4_verify_gemm(x, nib, sc, out=y, workspace=ws)
                w_passes = len(gemm_passes(M))
            for _ in range(5):
                call()
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                call()
            e1.record()
            torch.cuda.synchronize(dev)
            us = e0.elapsed_time(e1) * 1e3 / reps
            nb = gemm_bytes(M, N, K)
            rows.append({"mode": mode, "M": M, "passes_over_W": w_passes, "us_per_call": us, "bytes_per_call": nb,
                         "hbm_gbs": nb / (us * 1e-6) / 1e9, "pct_of_peak": nb / (us * 1e-6) / 1e9 / peak,
                         "tflops": 2.0 * M * N * K / (us * 1e-6) / 1e12})
            del ws
        del x, y
    del nib, sc
    torch.cuda.empty_cache()
    stack = []
    shapes = workloads.stack_shapes("llama8b")
    weights = [workloads.device_mxfp4_weights(N_, K_, lo, hi, seed=900 + i, device=dev)
               for i, (_, K_, N_) in enumerate(shapes)]
    for M in (80, 256, 320):
        xs = {K_: workloads.device_bf16_normal(M, K_, seed=K_ + M, device=dev) for K_ in sorted({k for _, k, _ in shapes})}
        ys = [torch.empty((M, N_), dtype=torch.float32, device=dev) for _, _, N_ in shapes]
        nb = sum(gemm_bytes(M, N_, K_) for _, K_, N_ in shapes)
        probs = [(xs[K_], wn, wsc, y_) for (_, K_, _), (wn, wsc), y_ in zip(shapes, weights, ys)]
        forms = [("w4a4", "grouped"), ("w4a16", "grouped")] + ([("w4a4", "per_call"), ("w4a16", "per_call")]
                                                               if M == 80 else [])
        for mode, form in forms:
            if form == "grouped":
                plan = mxs.GroupedGemm(probs, w4a4=mode == "w4a4")
                us = graph_us(torch, dev, plan, reps=5)
                del plan
            else:
                size = (mxs.mxfp4_verify_gemm_w4a4_workspace_size if mode == "w4a4"
                        else mxs.mxfp4_verify_gemm_workspace_size)
                fn = mxs.mxfp4_verify_gemm_w4a4 if mode == "w4a4" else mxs.mxfp4_verify_gemm
                ws = torch.empty(max(size(M, N_, K_) for _, K_, N_ in shapes), dtype=torch.uint8, device=dev)

                def stack_call():
                    for (_, K_, N_), (wn, wsc), y_ in zip(shapes, weights, ys):
                        fn(xs[K_], wn, wsc, out=y_, workspace=ws)

                us = graph_us(torch, dev, stack_call, reps=5)
                del ws
            stack.append({"mode": mode, "form": form, "M": M, "gemms": len(shapes), "us_per_stack": us, "bytes": nb,
                          "hbm_gbs": nb / (us * 1e-6) / 1e9, "pct_of_peak": nb / (us * 1e-6) / 1e9 / peak})
        del xs, ys, probs
    del weights
    torch.cuda.empty_cache()
    return {"metric": "W4A4 verify GEMM (X quantised to MX-FP4 in the call) vs W4A16, us per call",
            "timing": "lm_head: back-to-back calls, weights 279 MB beyond L2; stack (4.3 GB of weights, CUDA "
                      "graphs): grouped plans (each distinct X prepared once a pass, every W streamed once a "
                      "pass) and, at M = 80, one call per GEMM",
            "lm_head": rows, "stack_llama8b": stack}


def kv_cache_rows(mxs, torch, dev, peak, reps=20):
    """The MX-FP4 KV cache of the 8B stack's verification block: every layer's
    keys and values of one position (32 layers x 2 x 8 heads x 128 = 65536
    values) as one cache row, T = K + 1 = 5 positions appended from bf16 and
    committed, at B = 1 / 16 / 64; and the read side (the whole cache decoded
    to fp32) at L = 1024.  Algorithmic bytes: append = bf16 rows read + nibbles
    and scales written; dequant = the cache read + fp32 rows written."""
    W, T, L = 65536, 5, 1024
    rows = []
    for B in (1, 16, 64):
        gen = torch.Generator(device=dev)
        gen.manual_seed(400 + B)
        kv = torch.randn((B, T, W), generator=gen, device=dev).to(torch.bfloat16)
        nib = torch.zeros((B, L, W // 2), dtype=torch.uint8, device=dev)
        sc = torch.zeros((B, L, W // 32), dtype=torch.uint8, device=dev)
        lens = torch.full((B,), 100, dtype=torch.int32, device=dev)
        n_emit = torch.zeros((B,), dtype=torch.int32, device=dev)  # commit 0: the lengths stay put
        out = torch.empty((B, L, W), dtype=torch.float32, device=dev) if B == 1 else None

        def step():
            mxs.mxfp4_kv_append(kv, nib, sc, lens)
            mxs.spec_kv_commit(lens, n_emit, L)

        full = torch.full((B,), L, dtype=torch.int32, device=dev)  # the read-back decodes a full cache
        res = {"B": B}
        for name, fn, nb in (("append_commit", step, B * T * W * (2 + 17 / 32)),
                             ("dequant", (lambda: mxs.mxfp4_kv_dequant(nib, sc, full, out=out)) if out is not None
                              else None, B * L * W * (17 / 32 + 4))):
            if fn is None:
                continue
            us = graph_us(torch, dev, fn, reps)
            res[name] = {"us_per_call": us, "bytes_per_call": nb, "hbm_gbs": nb / (us * 1e-6) / 1e9,
                         "pct_of_peak": nb / (us * 1e-6) / 1e9 / peak}
        rows.append(res)
        del kv, nib, sc, lens, n_emit, out, full
    torch.cuda.empty_cache()
    return {"metric": "MX-FP4 KV cache, 8B stack's keys and values (65536 values per position)",
            "timing": "CUDA-graph replays on the same cache: append + commit move 0.8 / 13 / 53 MB (L2-warm); "
                      "the read-back decodes a full cache of 1024 positions: 36 MB read, 268 MB of fp32 written "
                      "(beyond L2)",
            "T": T, "L": L, "rows": rows}


def accept_sweep(args):
    """The acceptance-heavy sweep alone, as its own JSON line."""
    import torch

    import mxfp4_speculative_verification_gb300 as mxs

    mxs.build()
    dev = torch.device("cuda:0")
    peak, peak_kind = load_peaks()
    rec = accept_sweep_rows(mxs, torch, dev, peak)
    rec.update({"peak_gbs": peak, "peak_source": f"{peak_kind} hbm_gbs", "data": "synthetic"})
    print(json.dumps(rec), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mxs", choices=["mxs", "reference"])
    ap.add_argument("--workload", default="llama8b", choices=sorted(WORKLOADS))
    ap.add_argument("--detail", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the sub-records of the other configurations (8B batch sweep, 70B stack)")
    ap.add_argument("--profile-gemm", metavar="K,N",
                    help="only run one verify GEMM of this shape (M from --workload) 4 times "
                         "and exit; a small target for ncu captures")
    ap.add_argument("--profile-m", type=int, default=0,
                    help="rows of the --profile-gemm call (default: the workload's M)")
    ap.add_argument("--profile-grouped", type=int, default=0, metavar="LAYERS",
                    help="only run one grouped verify GEMM over the stack's first LAYERS layers 4 times (ncu target)")
    ap.add_argument("--profile-nvfp4", action="store_true",
                    help="with --profile-gemm: NVFP4 weights (nvfp4_verify_gemm) instead of MXFP4")
    ap.add_argument("--profile-w4a4", action="store_true",
                    help="with --profile-gemm / --profile-grouped: the W4A4 entry points")
    ap.add_argument("--profile-law", action="store_true",
                    help="only run spec_sampling_law on the workload's target rows 4 times and exit (ncu target)")
    ap.add_argument("--profile-accept", action="store_true",
                    help="only run spec_accept of the workload 4 times and exit (ncu target)")
    ap.add_argument("--accept-sweep", action="store_true",
                    help="acceptance-heavy sweep (B=64, K in 1/3/7): mean emitted tokens vs the closed "
                         "form and the per-row tail sum, plus timing; prints its own JSON line")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup(args)
    if args.profile_gemm or args.profile_accept or args.profile_law or args.profile_grouped:
        profile_target(args)
        return
    if args.accept_sweep:
        accept_sweep(args)
        return
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_mxs(args, world, rank, local)


if __name__ == "__main__":
    main()
