"""Benchmark: exact attention forward + backward (bf16) on GB300.

One step = the whole hot path over one batch of the dense d=128 workload
(B=4, H=16, N=8192, d_qk=d_v=128, softmax scale 1/sqrt(128)): forward and
backward, non-causal and causal (four passes, eight kernel launches). The
reported value is whole-job algorithmic TFLOP/s: forward 2*N^2*(d_qk+d_v),
backward 2*N^2*(3*d_qk+2*d_v) per (batch, head), causal counting half the
square. Inputs (Q, K, V, dO: 537 MB per rank) exceed the 129 MB L2, so no
flush is needed between steps.

The JSON line also carries `configs`: forward and backward TFLOP/s of every
other workload the metric covers (the d=128 sequence sweep, the outlier
variant, exp2 emulation shares, the (192,128) shape, the N=16384 training shape
in both backward modes, the 32-sequence varlen batch), timed after the
headline's region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) every rank runs its own batch (weak scaling, no
collective on the data path); timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fwd/bwd attention TFLOPs/s (bf16, causal & non) and % of GB300 dense peak"
UNIT = "TFLOP/s"
NOMINAL_PEAK_TFLOPS = 2250.0
WORKLOAD = dict(batch=4, heads=16, seqlen=8192, d_qk=128, d_v=128)

# DRAM traffic per launch from one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum), scaled to the benchmark's launch, valid only for the
# kernel sources it was measured on (sha256 prefix over the files the kernel
# compiles from, KERNEL_SOURCES, with comments and blank lines removed, so that
# documentation edits keep the figures); null otherwise.
# Measured on the non-causal B=2, H=16, N=8192 case (`bench.py --case`) and
# scaled x2 to the benchmark's B=4 launch (traffic grows with the (batch, head) units).
KERNEL_SOURCES = {
    "dkdv_wide_kernel": ("bwd_kernels.cuh", "bwd_common.cuh", "ptx_sm100.cuh", "score_mod.cuh", "kernels.h"),
    "dq_kernel": ("bwd_kernels.cuh", "bwd_common.cuh", "ptx_sm100.cuh", "score_mod.cuh", "kernels.h"),
    "attn_fwd_kernel": ("fwd_kernel.cuh", "exp2_emu.cuh", "exp2_poly_coeffs.h", "ptx_sm100.cuh", "score_mod.cuh",
                        "kernels.h"),
}
KERNEL_TRAFFIC_NCU = {
    "dkdv_wide_kernel": {"source_sha": "0e5c13170f822e3d", "bytes_per_launch": 2 * (270.638848e6 + 107.483392e6)},
    "dq_kernel": {"source_sha": "0e5c13170f822e3d", "bytes_per_launch": 2 * (270.719488e6 + 50.029568e6)},
    "attn_fwd_kernel": {"source_sha": "3484d0e8f058a718", "bytes_per_launch": 2 * (201.458944e6 + 49.052160e6)},
}


def code_only(text: str) -> str:
    """C/C++ source without comments or blank lines (string literals kept)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':  # a string literal: copy through its closing quote
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            i = text.find("\n", i)
            i = n if i < 0 else i
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def sha_of(*paths: str) -> str:
    h = hashlib.sha256()
    for path in paths:
        with open(path, encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def kernel_sources_sha(kernel: str) -> str:
    return sha_of(*(os.path.join(ROOT, "exact_attention_bf16_gb300", "csrc", f) for f in KERNEL_SOURCES[kernel]))


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def reduce_max(value: float, device=None) -> float:
    """Max over ranks (identity without an initialised process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def step_flops(w) -> dict:
    import workloads
    out = {}
    for causal in (False, True):
        ww = w.with_(causal=causal)
        out[("fwd", causal)] = workloads.workload_flops(ww, "fwd")
        out[("bwd", causal)] = workloads.workload_flops(ww, "bwd")
    return out


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        if not getattr(self, "lines", None):
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ---------------------------------------------------------------------------
# CPU oracle timing (reported baseline and the reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(seqlen: int, n_pairs: int = 1, seed: int = 0):
    """Times the fp64 oracle (forward + backward, both masks) on `n_pairs`
    (batch, head) units of the workload at `seqlen`; returns (TFLOP/s, seconds, flops)."""
    import numpy as np
    import workloads
    from oracle import attention_bwd, attention_fwd
    w = workloads.Workload("oracle_sample", 1, n_pairs, seqlen, seqlen, WORKLOAD["d_qk"], WORKLOAD["d_v"], False,
                           seed=seed)
    t = workloads.make_dense(w, device="cpu")
    q, k, v, do = (t[n][0].double().numpy() for n in ("q", "k", "v", "do"))
    flops = 0.0
    t0 = time.perf_counter()
    for causal in (False, True):
        for h in range(n_pairs):
            attention_fwd(q[:, h], k[:, h], v[:, h], w.scale, causal, row_block=2048)
            attention_bwd(q[:, h], k[:, h], v[:, h], do[:, h], w.scale, causal, row_block=2048)
            flops += workloads.attn_flops(seqlen, seqlen, w.d_qk, w.d_v, causal, "fwd")
            flops += workloads.attn_flops(seqlen, seqlen, w.d_qk, w.d_v, causal, "bwd")
    dt = time.perf_counter() - t0
    del np
    return flops / dt / 1e12, dt, flops


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    seqlen = WORKLOAD["seqlen"]
    for _ in range(args.warmup):
        oracle_sample(seqlen, 1)
    vals, secs = [], []
    for s in range(args.steps):
        v, dt, _ = oracle_sample(seqlen, 1, seed=s)
        vals.append(v)
        secs.append(dt)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"one (batch, head) unit of the workload (N={seqlen}, d=128), forward + backward, "
                                   "non-causal and causal, fp64 numpy oracle per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_dict():
    return {"workload": "dense_d128_B4_H16_N8192 forward+backward, non-causal and causal",
            "batch": WORKLOAD["batch"], "heads": WORKLOAD["heads"], "seqlen": WORKLOAD["seqlen"],
            "d_qk": WORKLOAD["d_qk"], "d_v": WORKLOAD["d_v"], "softmax_scale": 1 / math.sqrt(WORKLOAD["d_qk"]),
            "l2": "inputs (Q, K, V, dO = 537 MB per GPU) exceed the 129 MB L2; no flush",
            "parallelism": "per-GPU batch, weak scaling"}


# ---------------------------------------------------------------------------
# Per-configuration lines (outside the headline's timed region)
# ---------------------------------------------------------------------------
def time_ms(fn, stream, reps: int = 5, warm: int = 2) -> float:
    """Median CUDA-event time of fn() on `stream` after `warm` untimed calls."""
    import torch
    for _ in range(warm):
        fn()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in evs:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs)


def measure_configs(ea, dev, stream) -> dict:
    """Forward and backward TFLOP/s of every workload the metric covers: the
    d=128 sequence sweep (B*N = 32768, both masks), the outlier variant, the
    forward with part of exp2 on the FMA pipe, the two score modifications,
    the forward on FP8 E4M3 inputs, the d=64 backward in its two-kernel and
    single-pass forms, the (192,128) shape, the N=16384 training shape in both backward modes,
    512 queries against 32768 keys (the split-key forward) and the 32-sequence varlen batch. Inputs stay resident; each number is a
    median of 5 launches."""
    import torch
    import workloads
    out = {}

    def rec(name, w, fwd_ms=None, bwd_ms=None, **extra):
        r = dict(extra)
        if fwd_ms is not None:
            r.update(fwd_ms=fwd_ms, fwd_tflops=workloads.workload_flops(w, "fwd") / (fwd_ms * 1e-3) / 1e12)
        if bwd_ms is not None:
            r.update(bwd_ms=bwd_ms, bwd_tflops=workloads.workload_flops(w, "bwd") / (bwd_ms * 1e-3) / 1e12)
        out[name] = r

    def dense(w, bwd=True, emu=0, modes=(False,), mod=None):
        t = workloads.make_dense(w, device=dev)
        mod = dict(mod or {})
        if "alibi_slopes" in mod:
            mod["alibi_slopes"] = torch.tensor(mod["alibi_slopes"], dtype=torch.float32, device=dev)
        o, lse = ea.attn_fwd(t["q"], t["k"], t["v"], causal=w.causal, softmax_scale=w.scale, **mod)
        f = time_ms(lambda: ea.attn_fwd(t["q"], t["k"], t["v"], causal=w.causal, softmax_scale=w.scale, out=o,
                                        lse=lse, exp2_emu_period=emu, **mod), stream)
        res = {"fwd": f}
        if bwd:
            g = tuple(torch.empty_like(t[n]) for n in ("q", "k", "v"))
            for det in modes:
                res[det] = time_ms(lambda: ea.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=w.causal,
                                                       softmax_scale=w.scale, deterministic=det, dq=g[0], dk=g[1],
                                                       dv=g[2], **mod), stream)
        del t, o, lse
        torch.cuda.empty_cache()
        return res

    for n in (1024, 4096, 16384, 32768):
        for causal in (False, True):
            w = workloads.dense_d128(n, causal)
            r = dense(w)
            rec(f"dense_d128_B{w.batch}_N{n}_{'causal' if causal else 'noncausal'}", w, r["fwd"], r[False])
    w = workloads.dense_d128(8192, False, outlier=True)
    r = dense(w, bwd=False)
    rec("dense_d128_B4_N8192_noncausal_outlier", w, r["fwd"])
    for emu in (8, 4):
        for causal in (False, True):
            w = workloads.dense_d128(8192, causal)
            r = dense(w, bwd=False, emu=emu)
            rec(f"dense_d128_B4_N8192_{'causal' if causal else 'noncausal'}_exp2_emu_1_in_{emu}", w, r["fwd"],
                exp2_emu_period=emu)
    for causal in (False, True):  # the two-SM (cta_group::2, M = 256 pair) forward on the headline shape
        w = workloads.dense_d128(8192, causal)
        t = workloads.make_dense(w, device=dev, with_do=False)
        o, lse = ea.attn_fwd(t["q"], t["k"], t["v"], causal=causal, softmax_scale=w.scale, cta_pair=True)
        f = time_ms(lambda: ea.attn_fwd(t["q"], t["k"], t["v"], causal=causal, softmax_scale=w.scale, out=o, lse=lse,
                                        cta_pair=True), stream)
        rec(f"dense_d128_B4_N8192_{'causal' if causal else 'noncausal'}_fwd_cta_pair", w, f, cta_pair=True)
        del t, o, lse
        torch.cuda.empty_cache()
    for causal in (False, True):  # the two-SM (cta_group::2) dK/dV kernel on the headline shape
        w = workloads.dense_d128(8192, causal)
        t = workloads.make_dense(w, device=dev)
        o, lse = ea.attn_fwd(t["q"], t["k"], t["v"], causal=causal, softmax_scale=w.scale)
        g = tuple(torch.empty_like(t[n]) for n in ("q", "k", "v"))
        b = time_ms(lambda: ea.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=causal, softmax_scale=w.scale,
                                        dq=g[0], dk=g[1], dv=g[2], cta_pair=True), stream)
        rec(f"dense_d128_B4_N8192_{'causal' if causal else 'noncausal'}_bwd_cta_pair", w, None, b, cta_pair=True)
        del t, o, lse, g
        torch.cuda.empty_cache()
    for name, mod in (("softcap_30", {"softcap": 30.0}),
                      ("alibi", {"alibi_slopes": [2.0 ** (-8.0 * (h + 1) / 16) for h in range(16)]})):
        for causal in (False, True):  # score modifications on the headline shape
            w = workloads.dense_d128(8192, causal)
            r = dense(w, mod=mod)
            rec(f"dense_d128_B4_N8192_{'causal' if causal else 'noncausal'}_{name}", w, r["fwd"], r[False],
                score_mod=name)
    for causal in (False, True):  # FP8 E4M3 inputs (forward only): S on the 8-bit tensor-core kind
        w = workloads.dense_d128(8192, causal)
        t = workloads.make_dense(w, device=dev, with_do=False)
        f8, ds = {}, {}
        for n in ("q", "k", "v"):
            ds[n] = float(t[n].abs().max()) / 448.0
            f8[n] = (t[n].float() / ds[n]).to(torch.float8_e4m3fn)
        del t
        kw = dict(causal=causal, softmax_scale=w.scale, q_descale=ds["q"], k_descale=ds["k"], v_descale=ds["v"])
        o, lse = ea.attn_fwd(f8["q"], f8["k"], f8["v"], **kw)
        f = time_ms(lambda: ea.attn_fwd(f8["q"], f8["k"], f8["v"], out=o, lse=lse, **kw), stream)
        rec(f"dense_d128_B4_N8192_{'causal' if causal else 'noncausal'}_e4m3_inputs", w, f, input_dtype="e4m3")
        del f8, o, lse
        torch.cuda.empty_cache()
    for causal in (False, True):  # d = 64: two-kernel backward against the single pass (dQ reduced across CTAs)
        w = workloads.Workload(f"d64_N8192{'_causal' if causal else ''}", 4, 16, 8192, 8192, 64, 64, causal, seed=0)
        t = workloads.make_dense(w, device=dev)
        o, lse = ea.attn_fwd(t["q"], t["k"], t["v"], causal=causal, softmax_scale=w.scale)
        g = tuple(torch.empty_like(t[n]) for n in ("q", "k", "v"))
        name = f"dense_d64_B4_H16_N8192_{'causal' if causal else 'noncausal'}"
        for label, kw in (("two_kernel", {}), ("single_pass", {"single_pass": True}),
                          ("single_pass_deterministic", {"single_pass": True, "deterministic": True})):
            b = time_ms(lambda: ea.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=causal,
                                            softmax_scale=w.scale, dq=g[0], dk=g[1], dv=g[2], **kw), stream)
            rec(f"{name}_bwd_{label}", w, None, b, backward=label)
        del t, o, lse, g
        torch.cuda.empty_cache()
    w = workloads.mla_192_128()
    r = dense(w)
    rec("mla_192_128_B2_H32_N8192_causal", w, r["fwd"], r[False])
    w = workloads.bwd_d128_N16384()
    r = dense(w, modes=(False, True))
    rec("bwd_d128_B2_H16_N16384_causal", w, r["fwd"], r[False])
    rec("bwd_d128_B2_H16_N16384_causal_deterministic", w, None, r[True], deterministic=True)
    for causal in (False, True):  # short queries against long keys: the forward splits its keys across CTAs
        w = workloads.Workload(f"short_q{'_causal' if causal else ''}", 1, 16, 512, 32768, 128, 128, causal, seed=0)
        r = dense(w)
        rec(f"dense_d128_B1_H16_Nq512_Nk32768_{'causal' if causal else 'noncausal'}", w, r["fwd"], r[False],
            kv_split=True)

    w = workloads.varlen_32seq()
    t = workloads.make_varlen(w, device=dev)
    cu, L = t["cu_seqlens"], max(w.varlen_lengths)
    o, lse = ea.attn_fwd_varlen(t["q"], t["k"], t["v"], cu, cu, L, L, causal=True, softmax_scale=w.scale)
    f = time_ms(lambda: ea.attn_fwd_varlen(t["q"], t["k"], t["v"], cu, cu, L, L, causal=True, softmax_scale=w.scale,
                                           out=o, lse=lse), stream)
    g = tuple(torch.empty_like(t[n]) for n in ("q", "k", "v"))
    b = time_ms(lambda: ea.attn_bwd_varlen(t["q"], t["k"], t["v"], o, lse, t["do"], cu, cu, L, L, causal=True,
                                           softmax_scale=w.scale, dq=g[0], dk=g[1], dv=g[2]), stream)
    rec("varlen_32seq_H32_d128_causal", w, f, b, tokens=sum(w.varlen_lengths))
    del t, o, lse, g
    torch.cuda.empty_cache()
    ea.attn_get_device_status()
    return out


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_gpu(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    import exact_attention_bf16_gb300 as ea
    import workloads

    w = workloads.Workload("bench", WORKLOAD["batch"], WORKLOAD["heads"], WORKLOAD["seqlen"], WORKLOAD["seqlen"],
                           WORKLOAD["d_qk"], WORKLOAD["d_v"], False, seed=rank)
    t = workloads.make_dense(w, device=dev)
    q, k, v, do = t["q"], t["k"], t["v"], t["do"]
    B, N, H = w.batch, w.seqlen_q, w.heads
    o = {c: torch.empty_like(q) for c in (False, True)}
    lse = {c: torch.empty((B, H, N), dtype=torch.float32, device=dev) for c in (False, True)}
    grads = {c: tuple(torch.empty_like(x) for x in (q, k, v)) for c in (False, True)}
    stream = torch.cuda.current_stream(dev)

    def passes(record=None):
        for causal in (False, True):
            if record is not None:
                record[("fwd", causal)][0].record(stream)
            ea.attn_fwd(q, k, v, causal=causal, softmax_scale=w.scale, out=o[causal], lse=lse[causal])
            phase = None
            if record is not None:
                record[("fwd", causal)][1].record(stream)
                record[("bwd", causal)][0].record(stream)
                phase = record[("phases", causal)]
            dq, dk, dv = grads[causal]
            ea.attn_bwd(q, k, v, o[causal], lse[causal], do, causal=causal, softmax_scale=w.scale, dq=dq, dk=dk,
                        dv=dv, phase_events=phase)
            if record is not None:
                record[("bwd", causal)][1].record(stream)

    launches_per_step = 2 * (1 + 3)  # per mask: forward kernel; preprocess, dK/dV and dQ kernels
    flops = step_flops(w)
    total_flops = sum(flops.values())

    for _ in range(args.warmup):
        passes()
    torch.cuda.synchronize(dev)
    ea.attn_get_device_status()

    # ---- device-timed region -------------------------------------------------
    per_pass = {key: [] for key in flops}
    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize(dev)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        evs = []
        for _ in range(args.steps):
            d = {key: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for key in flops}
            for c in (False, True):
                d[("phases", c)] = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            evs.append(d)
        ev0.record(stream)
        for s in range(args.steps):
            passes(evs[s])
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
    elapsed_ms = ev0.elapsed_time(ev1)
    # per-kernel durations: forward (one launch per pass); backward phases from the library's events
    per_kernel = {"attn_fwd_kernel": [], "bwd_preprocess_kernel": [], "dkdv_wide_kernel": [], "dq_kernel": []}
    kernel_flops = {"attn_fwd_kernel": [], "bwd_preprocess_kernel": [], "dkdv_wide_kernel": [], "dq_kernel": []}
    for s in range(args.steps):
        for key in flops:
            a, b = evs[s][key]
            per_pass[key].append(a.elapsed_time(b))
        for c in (False, True):
            ph = evs[s][("phases", c)]
            b0 = evs[s][("bwd", c)][0]
            per_kernel["attn_fwd_kernel"].append(evs[s][("fwd", c)][0].elapsed_time(evs[s][("fwd", c)][1]))
            per_kernel["bwd_preprocess_kernel"].append(b0.elapsed_time(ph[0]))
            per_kernel["dkdv_wide_kernel"].append(ph[0].elapsed_time(ph[1]))
            per_kernel["dq_kernel"].append(ph[1].elapsed_time(ph[2]))
            pairs = w.batch * w.heads * (N * N / 2.0 if c else float(N) * N)
            kernel_flops["attn_fwd_kernel"].append(2 * pairs * (w.d_qk + w.d_v))
            kernel_flops["bwd_preprocess_kernel"].append(0.0)
            kernel_flops["dkdv_wide_kernel"].append(2 * pairs * (2 * w.d_qk + 2 * w.d_v))  # S^T, dP^T, dV, dK
            kernel_flops["dq_kernel"].append(2 * pairs * (2 * w.d_qk + w.d_v))        # S, dP, dQ
    ea.attn_get_device_status()
    elapsed_ms = reduce_max(elapsed_ms, dev)
    value = world * total_flops * args.steps / (elapsed_ms * 1e-3) / 1e12

    breakdown = {}
    for (direction, causal), ms in per_pass.items():
        med = statistics.median(ms)
        breakdown[f"{direction}_{'causal' if causal else 'noncausal'}"] = {
            "ms": med, "tflops": flops[(direction, causal)] / (med * 1e-3) / 1e12}

    # ---- end to end through the public API with host buffers ------------------
    # Every step copies its inputs (Q, K, V, dO) from pinned host memory to the
    # device, runs the forward and the backward for both masks through the
    # public API, and copies every output (O, LSE, dQ, dK, dV of both masks)
    # back to pinned host memory. Steps are pipelined over two device buffer
    # sets, with copies on their own streams (in and out), so one step's copies
    # overlap its neighbours' compute; all copies of all timed steps lie inside
    # the timed region.
    host_in = {n: t[n].cpu().pin_memory() for n in ("q", "k", "v", "do")}
    nbuf = 2
    dev_in = [{n: torch.empty_like(t[n]) for n in host_in} for _ in range(nbuf)]
    dev_out = [{c: [torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device=dev),
                    torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)] for c in (False, True)}
               for _ in range(nbuf)]
    host_out = [{c: [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in dev_out[i][c]] for c in (False, True)}
                for i in range(nbuf)]
    h2d = sum(x.numel() * x.element_size() for x in host_in.values())
    d2h = sum(x.numel() * x.element_size() for c in (False, True) for x in host_out[0][c])
    # Several copy streams per direction, each moving ~32 MB pieces, keep more than
    # one copy engine busy on the host link.
    n_cs = 4
    s_in = [torch.cuda.Stream(dev) for _ in range(n_cs)]
    s_out = [torch.cuda.Stream(dev) for _ in range(n_cs)]
    ev_in = [[torch.cuda.Event() for _ in range(n_cs)] for _ in range(nbuf)]
    ev_cmp = [torch.cuda.Event() for _ in range(nbuf)]
    ev_out = [[torch.cuda.Event() for _ in range(n_cs)] for _ in range(nbuf)]
    piece = 32 << 20

    def pieces(dst, src):
        d, sv = dst.view(-1), src.view(-1)
        step = max(1, piece // dst.element_size())
        return [(d[a:a + step], sv[a:a + step]) for a in range(0, d.numel(), step)]

    def e2e_step(kstep):
        i = kstep % nbuf
        jobs = [pc for n in host_in for pc in pieces(dev_in[i][n], host_in[n])]
        for c in range(n_cs):
            s_in[c].wait_event(ev_cmp[i])  # buffer i's inputs were last read by step kstep - 2
            with torch.cuda.stream(s_in[c]):
                for dst, src in jobs[c::n_cs]:
                    dst.copy_(src, non_blocking=True)
                ev_in[i][c].record(s_in[c])
            stream.wait_event(ev_in[i][c])
            stream.wait_event(ev_out[i][c])  # buffer i's outputs of step kstep - 2 are back on the host
        qi, ki, vi, doi = (dev_in[i][n] for n in ("q", "k", "v", "do"))
        for causal in (False, True):
            oo, ll, dq_, dk_, dv_ = dev_out[i][causal]
            ea.attn_fwd(qi, ki, vi, causal=causal, softmax_scale=w.scale, out=oo, lse=ll, stream=stream)
            ea.attn_bwd(qi, ki, vi, oo, ll, doi, causal=causal, softmax_scale=w.scale, dq=dq_, dk=dk_, dv=dv_,
                        stream=stream)
        ev_cmp[i].record(stream)
        jobs = [pc for causal in (False, True) for dst, src in zip(host_out[i][causal], dev_out[i][causal])
                for pc in pieces(dst, src)]
        for c in range(n_cs):
            s_out[c].wait_event(ev_cmp[i])
            with torch.cuda.stream(s_out[c]):
                for dst, src in jobs[c::n_cs]:
                    dst.copy_(src, non_blocking=True)
                ev_out[i][c].record(s_out[c])

    for kstep in range(max(2, args.warmup)):
        e2e_step(kstep)
    torch.cuda.synchronize(dev)
    barrier()
    e_steps = max(4, args.steps // 2)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for c in range(n_cs):
        s_in[c].wait_event(a)
        s_out[c].wait_event(a)
    for kstep in range(e_steps):
        e2e_step(kstep)
    for i in range(nbuf):
        for c in range(n_cs):
            stream.wait_event(ev_out[i][c])
    b.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(a.elapsed_time(b), dev)
    e2e_value = world * total_flops * e_steps / (e2e_ms * 1e-3) / 1e12
    # the last step's results, as read back, must match the device-resident run
    assert torch.equal(host_out[(e_steps - 1) % nbuf][True][1], lse[True].cpu()), "end-to-end LSE differs"

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    # ---- roofline of the dominant kernel (largest share of the step) -----------
    peaks, peak_kind = measured_peaks()
    totals = {k: sum(v) for k, v in per_kernel.items()}
    dom = max(totals, key=totals.get)
    n_launch = len(per_kernel[dom])
    dom_ms = totals[dom] / n_launch
    dom_flops = sum(kernel_flops[dom]) / n_launch
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    # The timed region lasts well under a second at full clock, so the burst
    # figure (a cuBLAS bf16 GEMM timed alone) is the matching denominator.
    peak = peaks.get("bf16_tflops", peaks.get("bf16_tflops_sustained"))
    src_sha = kernel_sources_sha(dom) if dom in KERNEL_SOURCES else None
    rec = KERNEL_TRAFFIC_NCU.get(dom, {})
    traffic = rec.get("bytes_per_launch") if rec.get("source_sha") == src_sha else None
    step_ms = sum(totals.values()) / args.steps
    roofline = {"kernel": f"{dom} d=128 (mean over non-causal and causal launches)", "bound": "tensor",
                "achieved": achieved, "peak": peak, "unit": UNIT, "frac": achieved / peak,
                "peak_kind": f"{peak_kind} bf16 burst (the timed region is short and runs at full clock)",
                "frac_of_nominal_2250": achieved / NOMINAL_PEAK_TFLOPS, "traffic": traffic,
                "algorithmic_flops_per_launch": dom_flops, "ms_per_launch": dom_ms,
                "share_of_step": totals[dom] / args.steps / step_ms,
                "kernels": {k: {"ms_per_launch": totals[k] / len(per_kernel[k]),
                                "share": totals[k] / args.steps / step_ms,
                                "tflops": (sum(kernel_flops[k]) / totals[k] / 1e9) if kernel_flops[k][0] else None}
                            for k in per_kernel}}

    configs = None if args.no_configs else measure_configs(ea, dev, stream)

    # ---- CPU baseline: the oracle on a bounded sample -------------------------
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cv, cdt, cfl = oracle_sample(WORKLOAD["seqlen"], n_pairs=4)
        cpu = {"value": cv, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": f"fp64 numpy oracle, forward + backward, non-causal and causal, 4 of the 64 (batch, head) "
                         f"units of the workload (N=8192, d=128): {cfl / 1e12:.3f} TFLOP in {cdt:.1f} s"}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_dict(),
        "pct_of_nominal_peak": 100.0 * value / (world * NOMINAL_PEAK_TFLOPS),
        "breakdown": breakdown,
        "configs": configs,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_case(args):
    """A few launches of one pass on a small workload (B=2, H=16, N=8192, d_qk =
    --dqk, d_v = min(d_qk, 128); Q, K, V, O of 67 to 100 MB each, larger than L2
    together) for profiler captures."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import exact_attention_bf16_gb300 as ea
    import workloads
    w = workloads.Workload("case", 2, 16, 8192, 8192, args.dqk, min(args.dqk, 128), args.causal, seed=0)
    t = workloads.make_dense(w, device="cuda")
    q, k, v, kw = t["q"], t["k"], t["v"], {}
    if args.e4m3:  # the E4M3 forward: codes of x / descale, descale = max|x| / 448
        for n in ("q", "k", "v"):
            kw[f"{n}_descale"] = float(t[n].abs().max()) / 448.0
        q, k, v = ((t[n].float() / kw[f"{n}_descale"]).to(torch.float8_e4m3fn) for n in ("q", "k", "v"))
    o, lse = ea.attn_fwd(t["q"], t["k"], t["v"], causal=w.causal)
    for _ in range(4):
        if args.case == "fwd":
            ea.attn_fwd(q, k, v, causal=w.causal, out=o, lse=lse, exp2_emu_period=args.emu, cta_pair=args.cta_pair,
                        **kw)
        else:
            ea.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=w.causal, cta_pair=args.cta_pair,
                        single_pass=args.single_pass)
    torch.cuda.synchronize()
    ea.attn_get_device_status()
    print(f"case {args.case} d_qk={args.dqk} causal={int(args.causal)} emu={args.emu} pair={int(args.cta_pair)} "
          f"e4m3={int(args.e4m3)} single_pass={int(args.single_pass)} done")
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", choices=["fwd", "bwd"], help="run a small profiling case and exit")
    ap.add_argument("--causal", action="store_true", help="causal mask for --case")
    ap.add_argument("--dqk", type=int, default=128, choices=[64, 128, 192], help="head dim of Q/K for --case")
    ap.add_argument("--emu", type=int, default=0, choices=[0, 4, 8], help="exp2 emulation period for --case fwd")
    ap.add_argument("--cta-pair", action="store_true", help="two-SM kernel for --case fwd / bwd (d = 128)")
    ap.add_argument("--e4m3", action="store_true", help="E4M3 inputs for --case fwd (d = 128)")
    ap.add_argument("--single-pass", action="store_true", help="single-pass backward for --case bwd (d = 64)")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-configuration lines")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.case:
        return run_case(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
