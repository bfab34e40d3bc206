"""Benchmark of the MoBA forward pass on GB300.

One step = one full forward (key pooling, gate + top-k, regroup, attention over
the selected past blocks, attention over the own block + merge) over one batch
of seeded synthetic inputs resident in HBM.  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload train32k] [--topk 3]

Under torchrun (N > 1) every rank runs the same per-GPU workload on its own
GPU with its own seed (weak scaling; the heads / sequences of different ranks
are independent, so there is no data-path collective); rank 0 prints the
whole-job throughput over the slowest rank's time.  `--impl reference` times
the CPU oracle on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoBA fwd tokens/s and effective TFLOP/s (% of BF16 peak) at 32K–1M tokens"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------
# work accounting (exact for the selection rule: past blocks are always full)
# ---------------------------------------------------------------------------

def issued_pairs(seqlens, block_size: int, topk: int):
    """(current-block pairs, past-block pairs) of (query, key) with key <= query
    that the forward attends to, summed over sequences, per head."""
    cur = past = 0
    for L in seqlens:
        n = (L + block_size - 1) // block_size
        for c in range(n):
            r = min(block_size, L - c * block_size)
            cur += r * (r + 1) // 2
            past += r * min(topk - 1, c) * block_size
    return cur, past


def hbm_bytes(w, topk: int):
    """Algorithmic HBM bytes of the pooling and gate kernels per forward."""
    total, H, D = w.total, w.H, w.D
    nb = sum((L + w.block_size - 1) // w.block_size for L in w.seqlens)
    pool = total * H * D * 2 + nb * H * D * 4
    gate = total * H * D * 2 + total * H * topk * 4
    return {"kpool": pool, "gate": gate}


# DRAM bytes (read + write) per launch of the dominant kernel, from one ncu
# capture of the command that produces the default line (the capture and its
# command are summarised under profiles/).  A figure is reported only while
# the kernel's sources hash to what was captured.
TRAFFIC_SOURCES = ("long_context_sparse_moba_gb300/csrc/moba_attn_tc.cu",
                   "long_context_sparse_moba_gb300/csrc/moba_ptx.cuh",
                   "long_context_sparse_moba_gb300/csrc/moba_internal.cuh")
MEASURED_TRAFFIC = {
    # (workload, topk, phase): (bytes per launch, sources_sha256() of the code measured)
    ("train32k", 3, "attn_past"): (1033480704 + 541106176,
                                   "5be34810902585958f7f2d11f2b1eb7214bd60bf842fa529a2923ffc30f1854e"),
}


def code_only(text: str) -> str:
    """Source text without comments and blank lines: what the compiler sees."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def sources_sha256() -> str:
    """Hash of the kernel sources' code (comments excluded), so that measured
    counters stay attached to the code they were taken on."""
    import hashlib
    h = hashlib.sha256()
    for rel in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()


def measured_traffic(workload: str, topk: int, phase: str):
    ent = MEASURED_TRAFFIC.get((workload, topk, phase))
    if ent is None or ent[1] != sources_sha256():
        return None
    return ent[0]


# ---- multi-rank host logic (one process per GPU, weak scaling) ----
def dist_env():
    """(world size, rank, local rank) from the launcher's environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_workload(w, rank: int):
    """The workload a rank times: same shapes, its own seed (independent
    sequences / heads, so the ranks never exchange data)."""
    from long_context_sparse_moba_gb300 import workloads
    return workloads.Workload(**{**w.__dict__, "seed": w.seed + 1000 * rank})


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The slowest rank's value (a MAX all-reduce; a no-op on one rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Tokens per second of the whole job: every rank's tokens over the slowest
    rank's step time."""
    return tokens_per_rank * world / (ms_per_step * 1e-3)


def decode_bench(ops, torch, dev, H, D, bs, topk, B=8, S=32768, steps=50):
    """One decode step of B sequences with S-token caches (the workload's heads,
    head size, block size and top-k): time per step, tokens/s and the
    algorithmic bytes (q, the pooled keys of the past blocks, the selected
    blocks' K and V, out, lse) over the time, against HBM."""
    g = torch.Generator(device=dev).manual_seed(77)
    kc = torch.randn(B, S, H, D, generator=g, device=dev, dtype=torch.bfloat16)
    vc = torch.randn(B, S, H, D, generator=g, device=dev, dtype=torch.bfloat16)
    q = torch.randn(B, H, D, generator=g, device=dev, dtype=torch.bfloat16)
    kbar = ops.kpool(kc, bs)
    lens = torch.full((B,), S, dtype=torch.int32, device=dev)
    ws = torch.empty(ops.decode_workspace_size(B, H, D, topk), dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty(B, H, dtype=torch.float32, device=dev)
    idx = torch.empty(B, H, topk, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(5):
        ops.decode_fwd(q, kc, vc, kbar, lens, bs, topk, out=out, lse=lse, idx=idx, workspace=ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        ops.decode_fwd(q, kc, vc, kbar, lens, bs, topk, out=out, lse=lse, idx=idx, workspace=ws)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    assert ops.get_status() == ops.MOBA_OK
    ci = (S - 1) // bs
    kv_keys = min(topk - 1, ci) * bs + (S - ci * bs)
    nbytes = B * H * (D * 2 + ci * D * 4 + kv_keys * D * 2 * 2 + D * 2 + 4)
    del kc, vc
    return {"B": B, "cache_len": S, "topk": topk, "ms_per_step": ms,
            "tokens_per_s": B / (ms * 1e-3), "gbs": nbytes / (ms * 1e-3) / 1e9,
            "bytes_per_step": nbytes}


def backward_bench(ops, torch, w, inp, topk, out, lse, flops_fwd, steps=10):
    """The backward pass (dq, dk, dv for a seeded upstream gradient) after the
    timed forward: time per call and its issued tensor-core work, five
    products per (query, key) pair against the forward's two, over the time.
    A training step keeps the forward's selection beside lse (``idx_out``),
    and the call takes it back (``idx_in``); the time of the call that
    recomputes the selection is reported beside it."""
    from long_context_sparse_moba_gb300 import workloads
    dev = inp.q.device
    dout = workloads.make_grad(w, device=dev)
    dq, dk, dv = (torch.empty_like(inp.q) for _ in range(3))
    ws = idx = None
    if not w.varlen:
        ws = torch.empty(ops.bwd_workspace_size(w.B, w.H, w.S, w.D, w.block_size, topk),
                         dtype=torch.uint8, device=dev)
        idx = torch.empty(w.B, w.S, w.H, topk, dtype=torch.int32, device=dev)
        out, lse = ops.attn_fwd(inp.q, inp.k, inp.v, w.block_size, topk, idx_out=idx)
        cu = None
    else:
        cu = torch.tensor(inp.cu_seqlens, dtype=torch.int32, device=dev)

    def call(saved):
        if w.varlen:
            ops.attn_bwd_varlen(inp.q, inp.k, inp.v, out, lse, dout, cu, w.S, w.block_size, topk)
        else:
            ops.attn_bwd(inp.q, inp.k, inp.v, out, lse, dout, w.block_size, topk, dq=dq, dk=dk,
                         dv=dv, workspace=ws, idx_in=idx if saved else None)

    def timed(saved):
        for _ in range(3):
            call(saved)
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            call(saved)
        e1.record(stream)
        torch.cuda.synchronize()
        assert ops.get_status() == ops.MOBA_OK
        return e0.elapsed_time(e1) / steps

    saved = idx is not None
    ms = timed(saved)
    flops = 2.5 * flops_fwd
    res = {"topk": topk, "ms_per_step": ms, "tokens_per_s": w.total / (ms * 1e-3),
           "issued_flops": flops, "effective_tflops": flops / (ms * 1e-3) / 1e12,
           "steps": steps,
           "selection": "the forward's (idx_out -> idx_in)" if saved else "recomputed"}
    if saved:
        res["ms_per_step_recomputing_selection"] = timed(False)
    return res


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------

def oracle_rows_rate(w, topk, host, kbar, n_rows, seed):
    import oracle
    tok, head = __import__("long_context_sparse_moba_gb300.workloads",
                           fromlist=["sample_rows"]).sample_rows(w, n_rows, seed=seed)
    q, k, v = host
    t0 = time.perf_counter()
    oracle.moba_rows(q, k, v, w.cu_seqlens(), w.H, w.D, w.block_size, topk, tok, head, kbar=kbar)
    return len(tok), time.perf_counter() - t0


def cpu_oracle_setup(w, inp):
    import oracle
    oracle.build()
    host = tuple(x.reshape(-1, w.H, w.D).cpu() for x in (inp.q, inp.k, inp.v))
    t0 = time.perf_counter()
    kbar = oracle.kpool(host[1], inp.cu_seqlens, w.H, w.D, w.block_size)
    t_pool = time.perf_counter() - t0
    return host, kbar, t_pool


def cpu_baseline(w, inp, topk, budget_s=12.0):
    """Oracle throughput on a bounded seeded sample of query rows; the pooling
    of the whole key tensor is charged pro rata to the sampled rows."""
    import oracle
    host, kbar, t_pool = cpu_oracle_setup(w, inp)
    n0, t0 = oracle_rows_rate(w, topk, host, kbar, 512, seed=77)
    n = int(min(w.total * w.H, max(512, n0 * budget_s / max(t0, 1e-6))))
    n, t = oracle_rows_rate(w, topk, host, kbar, n, seed=78)
    frac = n / (w.total * w.H)
    secs = t + t_pool * frac
    tokens = n / w.H
    return {"value": tokens / secs, "unit": "tokens/s", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{n} seeded (token, head) rows of the {w.name} workload (top-k {topk}) in "
                      f"{t:.1f} s plus key pooling of all blocks ({t_pool:.1f} s) charged pro rata "
                      f"({frac:.3%})"}


def run_reference(args, w, topk):
    """--impl reference: the CPU oracle, timed on the host cores."""
    import oracle
    from long_context_sparse_moba_gb300 import workloads
    inp = workloads.make_inputs(w, device="cpu")
    host, kbar, t_pool = cpu_oracle_setup(w, inp)
    n0, t0 = oracle_rows_rate(w, topk, host, kbar, 256, seed=90)
    rows = int(min(w.total * w.H, max(64, n0 * 0.25 / max(t0, 1e-6))))
    frac = rows / (w.total * w.H)
    for s in range(args.warmup):
        oracle_rows_rate(w, topk, host, kbar, rows, seed=100 + s)
    times = []
    for s in range(args.steps):
        _, t = oracle_rows_rate(w, topk, host, kbar, rows, seed=1000 + s)
        times.append(t + t_pool * frac)
    secs = sum(times)
    tokens = rows / w.H * args.steps
    value = tokens / secs
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, topk),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.max_threads(),
                             "kind": "oracle",
                             "sample": f"{rows} seeded (token, head) rows per step plus key "
                                       f"pooling charged pro rata ({frac:.3%})"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def config_of(w, topk):
    return {"workload": w.name, "B": w.B, "S": w.S, "H": w.H, "D": w.D,
            "block_size": w.block_size, "topk": topk, "tokens": w.total,
            "l2": "inputs larger than L2 (q, k, v %.0f MB)" % (3 * w.total * w.H * w.D * 2 / 1e6)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def phase_work(w, topk):
    """Algorithmic work of each timed phase: (bound, amount) -- HBM bytes for
    pooling and gate, issued tensor FLOPs for the two attention kernels."""
    cur, past = issued_pairs(w.seqlens, w.block_size, topk)
    hbm = hbm_bytes(w, topk)
    work = {"attn_past": ("tensor", 4 * w.D * past * w.H),
            "attn_current": ("tensor", 4 * w.D * cur * w.H)}
    n_max = (w.S + w.block_size - 1) // w.block_size
    if 1 < topk < n_max:  # pooling and gate run only when some row is scored
        work.update(kpool=("hbm", hbm["kpool"]), gate=("hbm", hbm["gate"]))
    if past == 0:
        del work["attn_past"]
    return work


def roofline_of(w, topk, per_call, peaks, peak_src):
    """Per-phase rates and the dominant kernel's roofline entry.  Tensor work
    is divided by the burst bf16 peak: every timed loop here lasts well under a
    second."""
    work = phase_work(w, topk)
    total_phase = sum(per_call.values())
    phases = {}
    for name, ms in per_call.items():
        ent = {"ms": ms, "share": ms / total_phase if total_phase > 0 else None}
        if name in work and ms > 0:
            kind, amount = work[name]
            if kind == "hbm":
                ent["gbs"] = amount / (ms * 1e-3) / 1e9
                ent["frac_hbm"] = ent["gbs"] / peaks["hbm_gbs"]
            else:
                ent["tflops"] = amount / (ms * 1e-3) / 1e12
                ent["frac_bf16"] = ent["tflops"] / peaks["bf16_tflops"]
        phases[name] = ent
    dom = max((n for n in per_call if n in work and per_call[n] > 0), key=lambda n: per_call[n])
    kind, amount = work[dom]
    dms = per_call[dom]
    if kind == "hbm":
        achieved, peak, unit, key = amount / (dms * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s", "hbm_gbs"
    else:
        achieved, peak, unit, key = (amount / (dms * 1e-3) / 1e12, peaks["bf16_tflops"], "TFLOP/s",
                                     "bf16_tflops")
    roofline = {"kernel": dom, "bound": kind, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "traffic": measured_traffic(w.name, topk, dom),
                "peak_source": f"{peak_src} ({key}, burst)"}
    return phases, roofline


class Forward:
    """One workload's inputs resident on the GPU and a forward step through
    the C ABI (caller workspace, so the timed step allocates nothing)."""

    def __init__(self, ops, torch, w, dev, **opts):
        from long_context_sparse_moba_gb300 import workloads
        self.ops, self.torch, self.w, self.dev = ops, torch, w, dev
        self.opts = opts  # per-call options of every step
        self.inp = workloads.make_inputs(w, device=dev)
        H, D = w.H, w.D
        if w.varlen:
            self.cu = torch.tensor(self.inp.cu_seqlens, dtype=torch.int32, device=dev)
            self.lse = torch.empty(H, w.total, dtype=torch.float32, device=dev)
        else:
            self.cu = None
            self.lse = torch.empty(w.B, H, w.S, dtype=torch.float32, device=dev)
        self.out = torch.empty_like(self.inp.q)
        self.ws = None
        self.ws_topk = None

    def workspace(self, topk):
        w, ops = self.w, self.ops
        if self.ws_topk != topk:
            if w.varlen:
                nb = ops.varlen_workspace_size(w.B, w.total, w.S, w.H, w.D, w.block_size, topk)
            else:
                nb = ops.workspace_size(w.B, w.H, w.S, w.D, w.block_size, topk)
            self.ws = None
            self.ws = self.torch.empty(max(nb, 256), dtype=self.torch.uint8, device=self.dev)
            self.ws_topk = topk
        return self.ws

    def step(self, topk, **kw):
        w, inp = self.w, self.inp
        ws = self.workspace(topk)
        kw = {**self.opts, **kw}
        if w.varlen:
            self.ops.attn_fwd_varlen(inp.q, inp.k, inp.v, self.cu, w.S, w.block_size, topk,
                                     out=self.out, lse=self.lse, workspace=ws, **kw)
        else:
            self.ops.attn_fwd(inp.q, inp.k, inp.v, w.block_size, topk, out=self.out,
                              lse=self.lse, workspace=ws, **kw)

    def time(self, topk, steps, warmup, phases=True, barrier=None):
        """(ms per step over `steps` forward calls timed with CUDA events on the
        launch stream, {phase: mean ms}, kernels launched in the timed loop)."""
        torch, ops = self.torch, self.ops
        for _ in range(warmup):
            self.step(topk)
        torch.cuda.synchronize()
        assert ops.get_status() == ops.MOBA_OK
        stream = torch.cuda.current_stream()
        evs = [ops.phase_events(stream) for _ in range(steps)] if phases else None
        torch.cuda.synchronize()
        if barrier:
            barrier()
        launches0 = ops.launch_count()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for s in range(steps):
            self.step(topk, phase_events=evs[s] if phases else None)
        e1.record(stream)
        torch.cuda.synchronize()
        if barrier:
            barrier()
        launches = ops.launch_count() - launches0
        ms = e0.elapsed_time(e1) / steps
        per_call = None
        if phases:
            per_call = {n: 0.0 for n in ops.PHASES}
            for ev in evs:
                for n, v in ops.phase_ms(ev).items():
                    per_call[n] += v / steps
        assert ops.get_status() == ops.MOBA_OK
        return ms, per_call, launches


def workload_entry(fw, topk, steps, warmup, peaks, peak_src):
    """Measured sub-object of the bench line for one (workload, top-k)."""
    w = fw.w
    ms, per_call, launches = fw.time(topk, steps, warmup)
    cur, past = issued_pairs(w.seqlens, w.block_size, topk)
    flops = 4 * w.D * (cur + past) * w.H
    tfl = flops / (ms * 1e-3) / 1e12
    phases, roofline = roofline_of(w, topk, per_call, peaks, peak_src)
    n_max = (w.S + w.block_size - 1) // w.block_size
    dcur, dpast = issued_pairs(w.seqlens, w.block_size, n_max)
    return {"config": config_of(w, topk), "steps": steps, "warmup": warmup,
            "ms_per_step": ms, "tokens_per_s": w.total / (ms * 1e-3),
            "issued_flops_per_step": flops, "effective_tflops": tfl,
            "frac_of_bf16_peak": tfl / peaks["bf16_tflops"],
            "sparsity_vs_dense_causal": 1.0 - (cur + past) / (dcur + dpast),
            "phases": phases, "roofline": roofline, "gpu_launches": launches}


def near_tie_report(w, fw, topk, n_rows=4096, seed=4242):
    """Selections the forward used (its idx_out), checked against the oracle's
    on a seeded row sample: rows whose last kept and first dropped past blocks
    score within 1e-5 are counted as near ties; any other difference is a
    mismatch.  Part of the CPU-baseline leg (the oracle runs on the host)."""
    import oracle
    from long_context_sparse_moba_gb300 import workloads
    torch, ops = fw.torch, fw.ops
    shape = (w.total, w.H, topk) if w.varlen else (w.B, w.S, w.H, topk)
    idx = torch.empty(shape, dtype=torch.int32, device=fw.dev)
    fw.step(topk, idx_out=idx)
    torch.cuda.synchronize()
    tok, head = workloads.sample_rows(w, n_rows, seed=seed)
    gi = idx.reshape(w.total, w.H, topk).cpu().numpy()[tok, head]
    host = tuple(x.reshape(-1, w.H, w.D).cpu() for x in (fw.inp.q, fw.inp.k, fw.inp.v))
    ref = oracle.moba_rows(*host, w.cu_seqlens(), w.H, w.D, w.block_size, topk, tok, head)
    near = ref["gap"] < 1e-5
    differ = (gi != ref["idx"]).any(axis=1)
    return {"workload": w.name, "topk": topk, "sampled_rows": int(len(tok)),
            "near_tie_rows": int(near.sum()), "near_tie_rows_selected_differently":
            int((near & differ).sum()), "mismatches_outside_near_ties": int((differ & ~near).sum()),
            "tie_gap": 1e-5}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="train32k")
    ap.add_argument("--topk", type=int, default=None)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-range", action="store_true",
                    help="skip the other workloads of the metric's range (128K, 1M, varlen)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from long_context_sparse_moba_gb300 import workloads
    w = workloads.WORKLOADS[args.workload]
    topk = args.topk if args.topk is not None else w.topks[0]

    world, rank, local = dist_env()

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, w, topk)
        return

    import torch
    import torch.distributed as dist
    from long_context_sparse_moba_gb300 import build as _build
    from long_context_sparse_moba_gb300 import ops

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0 or world == 1:
        _build.build()
    if world > 1:
        dist.barrier()
    ops.lib()
    barrier = dist.barrier if world > 1 else None

    dev = torch.device("cuda", local)
    wr = rank_workload(w, rank)
    fw = Forward(ops, torch, wr, dev)
    inp = fw.inp
    q, k, v = inp.q, inp.k, inp.v
    bs, H, D = w.block_size, w.H, w.D
    peaks, peak_src = load_peaks()

    # ---------------- the headline: timed steps of the workload ----------------
    for _ in range(args.warmup):
        fw.step(topk)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ms_per_step, per_call, launches = fw.time(topk, args.steps, 0, barrier=barrier)
    clk = clocks.stop()
    status = ops.get_status()
    ms_per_step = max_over_ranks(ms_per_step, world, dev)

    # dense comparison: same kernels with top-k = number of blocks
    dense = None
    n_max = (w.S + bs - 1) // bs
    if not args.no_dense and topk < n_max:
        dms, _, _ = fw.time(n_max, 3, 1, phases=False)
        dcur, dpast = issued_pairs(w.seqlens, bs, n_max)
        dfl = 4 * D * (dcur + dpast) * H
        dense = {"topk": n_max, "ms_per_step": dms,
                 "effective_tflops": dfl / (dms * 1e-3) / 1e12,
                 "frac_of_bf16_peak": dfl / (dms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                 "sparse_speedup": dms / ms_per_step}
        fw.workspace(topk)

    decode = None
    if not args.no_decode and rank == 0 and not w.varlen:
        decode = decode_bench(ops, torch, dev, H, D, bs, topk)
        decode["frac_hbm"] = decode["gbs"] / peaks["hbm_gbs"]

    # end to end through the public API with pinned host buffers
    e2e = None
    if not args.no_e2e:
        out, lse = fw.out, fw.lse
        hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))
        esteps = max(4, min(args.steps, 20))
        stream = torch.cuda.current_stream()
        if not wr.varlen:
            # moba_attn_fwd_host: each call copies its step's q, k, v in and
            # out, lse back itself; consecutive calls alternate two streams
            # (each with its own device scratch and host results), so one
            # call's copies run beside the other's kernels
            qB, qS = q.shape[0], q.shape[1]
            size = ops.host_scratch_size(qB, H, qS, D, bs, topk)
            streams = [torch.cuda.Stream(device=dev) for _ in range(2)]
            scratch = [torch.empty(size, dtype=torch.uint8, device=dev) for _ in range(2)]
            hout = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
            hlse = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]

            def e2e_step(n):
                ops.attn_fwd_host(hq, hk, hv, bs, topk, hout[n % 2], hlse[n % 2], scratch[n % 2],
                                  stream=streams[n % 2])
            overlap = "two streams: one call's host copies beside the other's kernels"
        else:
            hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
            hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
            streams = [stream]

            def e2e_step(n):
                q.copy_(hq, non_blocking=True)
                k.copy_(hk, non_blocking=True)
                v.copy_(hv, non_blocking=True)
                fw.step(topk)
                hout.copy_(out, non_blocking=True)
                hlse.copy_(lse, non_blocking=True)
            overlap = "none: copies and kernels in order on one stream"

        e2e_step(0)
        e2e_step(1)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for s_ in streams:
            s_.wait_event(e0)
        for n in range(esteps):
            e2e_step(n)
        for s_ in streams:
            stream.wait_stream(s_)
        e1.record(stream)
        torch.cuda.synchronize()
        assert ops.get_status() == ops.MOBA_OK
        ems = max_over_ranks(e0.elapsed_time(e1) / esteps, world, dev)
        e2e = {"value": whole_job_rate(wr.total, world, ems), "unit": "tokens/s",
               "h2d_bytes_per_step": 3 * q.numel() * 2,
               "d2h_bytes_per_step": out.numel() * 2 + lse.numel() * 4,
               "ms_per_step": ems, "steps": esteps, "overlap": overlap}
        del hq, hk, hv, hout, hlse

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    cur, past = issued_pairs(w.seqlens, bs, topk)
    flops = 4 * D * (cur + past) * H
    tflops = flops / (ms_per_step * 1e-3) / 1e12
    backward = None
    if not args.no_backward:
        rc_, rp_ = issued_pairs(wr.seqlens, bs, topk)
        backward = backward_bench(ops, torch, wr, inp, topk, fw.out, fw.lse,
                                  4 * D * (rc_ + rp_) * H)
        backward["frac_bf16"] = backward["effective_tflops"] / peaks["bf16_tflops"]
    phases, roofline = roofline_of(w, topk, per_call, peaks, peak_src)

    cpu = near = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(w, inp, topk)
        near = [near_tie_report(w, fw, topk)]

    # ---------------- the rest of the metric's range (32K to 1M) ----------------
    rng = {}
    if not args.no_range and world == 1:
        fw_keep = fw
        for name, steps in (("long128k", 20), ("prefill1m", 10)):
            if name == w.name:
                continue
            fw = None
            torch.cuda.empty_cache()
            fo = Forward(ops, torch, workloads.WORKLOADS[name], dev)
            t = workloads.WORKLOADS[name].topks[0]
            rng[name] = workload_entry(fo, t, steps, 3, peaks, peak_src)
            if not args.no_cpu_baseline:
                near.append(near_tie_report(fo.w, fo, t))
            del fo
        # the adaptive schedule against the block-major one on inputs whose
        # 256-row tiles agree on their past blocks (the adaptive schedule is the
        # default everywhere above)
        for name, steps in (("coherent32k", 20), ("coherent128k", 10)):
            torch.cuda.empty_cache()
            fo = Forward(ops, torch, workloads.WORKLOADS[name], dev)
            t = fo.w.topks[0]
            ent = {"adaptive": workload_entry(fo, t, steps, 3, peaks, peak_src)}
            fo.opts = {"schedule": ops.SCHEDULE_BLOCK_MAJOR}
            ent["block_major"] = workload_entry(fo, t, steps, 3, peaks, peak_src)
            ent["speedup"] = ent["block_major"]["ms_per_step"] / ent["adaptive"]["ms_per_step"]
            rng[name] = ent
            del fo
        if w.name != "varlen":
            torch.cuda.empty_cache()
            fo = Forward(ops, torch, workloads.WORKLOADS["varlen"], dev)
            rng["varlen"] = {str(t): workload_entry(fo, t, 20, 3, peaks, peak_src)
                             for t in fo.w.topks}
            if not args.no_cpu_baseline:
                near.append(near_tie_report(fo.w, fo, 3))
            del fo
        fw = fw_keep

    line = {"metric": METRIC, "value": whole_job_rate(w.total, world, ms_per_step), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_of(w, topk),
            "effective_tflops": tflops * world,
            "frac_of_bf16_peak": tflops / peaks["bf16_tflops"],
            "issued_flops_per_step": flops,
            "sparsity_vs_dense_causal": None,
            "roofline": roofline, "phases": phases, "dense": dense, "decode": decode,
            "backward": backward, "range": rng or None, "near_ties": near, "e2e": e2e,
            "cpu_baseline": cpu, "gpu_launches": launches, "clocks": clk,
            "device_status": ops.status_string(status)}
    dcur, dpast = issued_pairs(w.seqlens, bs, n_max)
    line["sparsity_vs_dense_causal"] = 1.0 - (cur + past) / (dcur + dpast)
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
