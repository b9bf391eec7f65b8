"""Benchmark of the sparse latent attention hot path on GB300.

One step = the whole hot path over one batch: the fp8 round trip of the step's new KV rows into
the ring, the window index rows, and sparse_attn over [ring | compressed rows] (all through the
C ABI of libdsattn).  The metric is gathered (token, head, valid row) units per second.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 4] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same workload on its own GPU (weak scaling, no data
path collective); rank 0 prints one JSON line with value = units of all ranks / max time.
`--impl reference` times the CPU oracle (plain C, all host cores) on a bounded sample of the
same workload; under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from sparse_latent_attention_attn_gb300 import workloads as wl  # noqa: E402

METRIC = "decode sparse_attn gathered (token·head·row)/s; % of tensor/HBM roofline"
UNIT = "(token·head·row)/s"
DEFAULT_CONFIG = 4
L2_BYTES = 129 * 1024 * 1024
SLEEP_CYCLES = 40_000_000      # ~20 ms of device time: long enough for the host to enqueue a run
ATTN_KERNEL_SOURCES = ["sparse_latent_attention_attn_gb300/csrc/sparse_attn_tc.cu",
                       "sparse_latent_attention_attn_gb300/csrc/sparse_attn_ot.cu",
                       "sparse_latent_attention_attn_gb300/csrc/sparse_attn_ot.cuh",
                       "sparse_latent_attention_attn_gb300/csrc/attn_split.cuh",
                       "sparse_latent_attention_attn_gb300/csrc/ptx.cuh",
                       "sparse_latent_attention_attn_gb300/csrc/common.cuh"]
PROFILE_SUMMARY = "profiles/sparse_attn_{workload}.txt"
INDEXER_KERNEL_SOURCES = ["sparse_latent_attention_attn_gb300/csrc/indexer.cu",
                          "sparse_latent_attention_attn_gb300/csrc/ptx.cuh",
                          "sparse_latent_attention_attn_gb300/csrc/common.cuh"]


# ----------------------------------------------------------------------------------------------
# distributed plumbing (one process per GPU; no collective on the data path)
# ----------------------------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def aggregate(units_local: float, seconds_local: float, world: int, device=None):
    """Whole-job units and the slowest rank's time (max over ranks), via two all-reduces."""
    if world == 1:
        return units_local, seconds_local
    t = torch.tensor([units_local], dtype=torch.float64, device=device)
    s = torch.tensor([seconds_local], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    torch.distributed.all_reduce(s, op=torch.distributed.ReduceOp.MAX)
    return float(t.item()), float(s.item())


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


# ----------------------------------------------------------------------------------------------
# peaks, clocks, profile summary
# ----------------------------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.count(",") >= 9]
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[2]))
                smax = float(r[3])
            except ValueError:
                continue
            for name, val in zip(names, r[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def _code_tokens(text: str) -> str:
    """The source without comments and whitespace: what the compiler sees, so a summary taken on
    the code stays valid across comment and layout edits."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return re.sub(r"\s+", "", text)


def kernel_source_hash(sources=None) -> str:
    h = hashlib.sha256()
    for rel in (ATTN_KERNEL_SOURCES if sources is None else sources):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_tokens(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, launches_units: float, summary: str = PROFILE_SUMMARY, sources=None):
    """dram bytes per launch from the committed ncu summary, if it was taken on this kernel source."""
    path = os.path.join(ROOT, summary.format(workload=workload))
    if not os.path.exists(path):
        return None
    src_hash, traffic = None, None
    with open(path) as f:
        for line in f:
            if line.startswith("kernel_source_sha256_16:"):
                src_hash = line.split(":", 1)[1].strip()
            if line.startswith("dram_bytes_per_launch:"):
                traffic = float(line.split(":", 1)[1].strip())
    if src_hash != kernel_source_hash(sources):
        return None
    return traffic


# ----------------------------------------------------------------------------------------------
# one set of step inputs on the device
# ----------------------------------------------------------------------------------------------

class StepSet:
    def __init__(self, w: wl.Workload, device, seed: int, kv_mode: str = "bf16", pairs: bool = False):
        from sparse_latent_attention_attn_gb300 import dsattn
        self.w = w
        self.fp8 = kv_mode == "fp8"
        self.pairs = pairs
        inp = wl.make_step_inputs(w, device=device, seed=seed)
        self.q, self.kv, self.sink = inp.q, inp.kv, inp.sink
        self.cidx = inp.cidx
        self.idx = torch.empty((w.b, w.m, w.topk), dtype=torch.int32, device=device)
        self.idx[..., w.win_cols:] = inp.cidx
        self.o = torch.empty_like(inp.q)
        if w.decode:
            dsattn.kv_quant_ring_write(inp.hist, self.kv[:, : w.window], w.start_pos - w.window, w.window)
            self.new_kv = inp.new_kv
            self.ring = self.kv[:, : w.window]
        else:
            self.new_kv = None
            self.ring = torch.zeros((w.b, w.window, w.d), dtype=torch.bfloat16, device=device)
        del inp
        if self.fp8:
            # the fp8 row store of the whole kv (window ring in its leading rows, then the
            # compressed rows, all kept quantised); self.kv becomes its bf16 decode (the round trip)
            self.codes, self.exps = dsattn.kv_quantize_fp8(self.kv)
            dsattn.kv_quant_ring_write(self.kv, None, 0, 1)
        need = (dsattn.sparse_attn_prefill_workspace_bytes(w.b, w.m, w.h, w.d, w.topk) if pairs
                else dsattn.sparse_attn_workspace_bytes(w.b, w.m, w.h, w.d, w.topk))
        self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        # library kernels per step: ring write, window rows, sparse_attn (+ combine when tokens are cut)
        self.attn_kernel = dsattn.KERNEL_CLUSTER
        if pairs:   # ring write, window rows, the pair union, attention, and the combine when pairs are cut
            union = (w.b * ((w.m + 1) // 2) * 2 * w.topk * 4 + 255) // 256 * 256
            self.launches = 4 + (1 if need > union else 0)
        elif self.fp8:
            self.launches = 3 + (1 if need > 0 else 0)
        else:
            n_attn, self.attn_kernel = dsattn.sparse_attn_launches(w.b, w.m, w.h, w.d, w.topk)
            self.launches = 2 + n_attn

    def attend(self, ev=None):
        """sparse_attn alone on the step's inputs; events (start, end) around it when given."""
        from sparse_latent_attention_attn_gb300 import dsattn
        if ev is not None:
            ev[0].record()
        self._attn(dsattn)
        if ev is not None:
            ev[1].record()

    def _attn(self, dsattn):
        if self.pairs:
            dsattn.sparse_attn_prefill(self.q, self.kv, self.sink, self.idx, self.w.scale, o=self.o, workspace=self.ws)
        elif self.fp8:
            dsattn.sparse_attn_fp8kv(self.q, self.codes, self.exps, self.sink, self.idx, self.w.scale, o=self.o,
                                     workspace=self.ws)
        else:
            dsattn.sparse_attn(self.q, self.kv, self.sink, self.idx, self.w.scale, o=self.o, workspace=self.ws)

    def run(self, ev_attn=None):
        """The whole step; events (start, end) bracket the sparse_attn launch when given."""
        from sparse_latent_attention_attn_gb300 import dsattn
        w = self.w
        if w.decode and self.fp8:
            dsattn.kv_quant_ring_write_fp8(self.new_kv, self.codes, self.exps, w.start_pos, w.window)
            dsattn.window_topk_idxs(self.idx, w.b, 1, w.start_pos, w.window)
        elif w.decode:
            dsattn.kv_quant_ring_write(self.new_kv, self.ring, w.start_pos, w.window)
            dsattn.window_topk_idxs(self.idx, w.b, 1, w.start_pos, w.window)
        else:
            dsattn.kv_quant_ring_write(self.kv[:, : w.s], self.ring, 0, w.window)
            dsattn.window_topk_idxs(self.idx, w.b, w.s, 0, w.window)
        if ev_attn is not None:
            ev_attn[0].record()
        self._attn(dsattn)
        if ev_attn is not None:
            ev_attn[1].record()

    def counts(self):
        """units, algorithmic bytes and flops of one sparse_attn launch (idx as the step leaves it)."""
        w = self.w
        valid = int((self.idx >= 0).sum().item())
        units = valid * w.h
        row_bytes = (w.d + w.d // 32) if self.fp8 else w.d * 2    # codes + exponents, or bf16
        bytes_ = valid * row_bytes + 2 * w.b * w.m * w.h * w.d * 2 + self.idx.numel() * 4 + w.h * 4
        flops = 4 * w.d * units
        return units, bytes_, flops

    def io_bytes(self):
        """Bytes a step takes from and gives back to the host in the end-to-end measurement."""
        w = self.w
        h2d = self.q.numel() * 2 + self.cidx.numel() * 4
        h2d += (self.new_kv.numel() * 2) if w.decode else (w.b * w.s * w.d * 2)
        return h2d, self.o.numel() * 2


# ----------------------------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# ----------------------------------------------------------------------------------------------

class OracleSample:
    """The oracle (plain C, all host cores) on the host copy of a workload's inputs.

    Inputs are generated and copied to the host once; `time(n)` runs the oracle on the first n
    sequences (decode) or n evenly spaced query tokens (prefill) and returns (seconds, units)."""

    def __init__(self, w: wl.Workload, sset: StepSet | None, device, max_items: int):
        import oracle
        oracle.build()
        self.oracle = oracle
        self.w = w
        self.cores = os.cpu_count() or 1
        if sset is None:
            inp = wl.make_step_inputs(w, device=device)
            idx = torch.empty((w.b, w.m, w.topk), dtype=torch.int32, device=device)
            idx[..., w.win_cols:] = inp.cidx
            q, kv, sink = inp.q, inp.kv, inp.sink
        else:
            idx, q, kv, sink = sset.idx, sset.q, sset.kv, sset.sink
        # window columns as the oracle computes them
        win = oracle.window_topk_idxs(w.s if not w.decode else 1, w.start_pos, w.window)
        self.limit = w.b if w.decode else w.m
        keep = min(self.limit, max(1, max_items))
        if w.decode:
            seqs = torch.arange(keep, device=q.device)
            self.q = wl.bits(q.index_select(0, seqs))
            self.kv = wl.bits(kv.index_select(0, seqs))
            self.idx = idx[:keep].cpu().numpy()
        else:
            self.q, self.kv = wl.bits(q), wl.bits(kv)
            self.idx = idx.cpu().numpy()
        self.idx[..., : w.win_cols] = win[None]
        self.sink = sink.cpu().numpy()
        self.keep = keep

    def time(self, n: int):
        w, o = self.w, self.oracle
        n = max(1, min(n, self.keep))
        if w.decode:
            ib = np.ascontiguousarray(self.idx[:n])
            t0 = time.perf_counter()
            o.sparse_attn(np.ascontiguousarray(self.q[:n]), np.ascontiguousarray(self.kv[:n]), self.sink, ib,
                          w.scale, nthreads=self.cores)
            dt = time.perf_counter() - t0
            units = int((ib >= 0).sum()) * w.h
        else:
            toks = np.linspace(0, w.m - 1, n).astype(np.int64)
            t0 = time.perf_counter()
            o.sparse_attn(self.q, self.kv, self.sink, self.idx, w.scale, tokens=toks, nthreads=self.cores)
            dt = time.perf_counter() - t0
            units = int((self.idx[0, toks] >= 0).sum()) * w.h
        return dt, units

    def size_for(self, budget_s: float) -> int:
        """Items whose oracle run takes about budget_s (measured on a first small run)."""
        n = min(self.keep, self.cores)
        dt, _ = self.time(n)
        if dt < budget_s / 4 and n < self.keep:
            n = int(min(self.keep, max(n + 1, n * budget_s / max(dt, 1e-3) * 0.8)))
        return n

    def describe(self, n: int, units: int, dt: float) -> str:
        what = "sequences" if self.w.decode else "query tokens"
        return (f"{n} of {self.limit} {what} of {self.w.name} ({units} units, {dt:.2f} s wall, plain C, "
                f"{self.cores} threads)")


def oracle_sample_rate(w: wl.Workload, sset: StepSet | None, budget_s: float, device):
    """cpu_baseline: the oracle timed on a bounded sample (about budget_s of host work)."""
    cores = os.cpu_count() or 1
    smp = OracleSample(w, sset, device, max_items=max(cores, 4 * cores))
    n = smp.size_for(budget_s)
    dt, units = smp.time(n)
    return {"value": units / dt, "unit": UNIT, "cores": smp.cores, "kind": "oracle",
            "sample": smp.describe(n, units, dt), "_units": units, "_seconds": dt}


def public(d):
    return None if d is None else {k: v for k, v in d.items() if not k.startswith("_")}


# ----------------------------------------------------------------------------------------------
# arms
# ----------------------------------------------------------------------------------------------

def workload_config(w: wl.Workload, nsets: int):
    return {"workload": f"{w.name}: b={w.b} h={w.h} d={w.d} window={w.window} start_pos={w.start_pos} "
                        f"queries/seq={w.m} compressed={w.topk_comp} of {w.n_comp} rows, "
                        f"{w.neg_frac:.0%} of them -1",
            "global_batch": w.b, "seq_len": w.m, "topk": w.topk, "heads": w.h, "head_dim": w.d,
            "parallelism": "replicas (one independent batch per GPU)",
            "l2": f"{nsets} rotating input sets; each step's gathered rows exceed or rotate past the "
                  f"{L2_BYTES >> 20} MiB L2"}


def run_reference(args):
    """The reference arm: the oracle, as it stands, on the host cores (rank 0 only).

    Each of the warm-up and timed steps runs the oracle on the same bounded sample of the
    workload, sized so that the whole run takes about --ref-budget seconds of host work."""
    rank, world, local = dist_env()
    if rank != 0:
        return 0
    w = wl.WORKLOADS[args.config]
    device = "cuda" if torch.cuda.is_available() else "cpu"
    cores = os.cpu_count() or 1
    nsteps = args.warmup + args.steps
    smp = OracleSample(w, None, device, max_items=4 * cores)
    n = smp.size_for(max(0.05, args.ref_budget / max(1, nsteps)))
    total_units, total_s = 0, 0.0
    for k in range(nsteps):
        dt, units = smp.time(n)
        if k >= args.warmup:
            total_units += units
            total_s += dt
    value = total_units / total_s if total_s else 0.0
    per_step = total_units // max(1, args.steps)
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": 1e3 * total_s / max(1, args.steps), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded, N(0,1))",
           "config": workload_config(w, 1),
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": smp.cores, "kind": "oracle",
                            "sample": "each step: " + smp.describe(n, per_step, total_s / max(1, args.steps))},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)
    return 0


def run_indexer(args):
    """The Indexer step of a workload (its scores and top-k) timed alone: CUDA events around K
    calls on the launching stream after W warm-ups, two input sets alternating so consecutive
    calls read different keys.  Unit: one (query, visible compressed position) pair scored."""
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist_init(world, "nccl")
    from sparse_latent_attention_attn_gb300 import dsattn
    iw = wl.INDEXER_WORKLOADS[args.config]
    peaks = load_peaks()
    kk = min(iw.topk, iw.Tv)
    sets = []
    for k_ in range(2):
        q, k, w = wl.indexer_inputs(iw, device=device, seed=iw.seed + 7919 * k_ + 104729 * rank)
        idx = torch.empty((iw.b, iw.s, kk), dtype=torch.int32, device=device)
        ws = torch.empty(dsattn.indexer_workspace_bytes(iw.b, iw.s, iw.start_pos, iw.ratio), dtype=torch.uint8,
                         device=device)
        sets.append((q, k, w, idx, ws))

    def call(st):
        q, k, w, idx, ws = st
        dsattn.indexer_topk(q, k, w, iw.start_pos, iw.ratio, iw.topk, iw.offset, idx=idx, workspace=ws)

    for j in range(args.warmup):
        call(sets[j % 2])
    torch.cuda.synchronize()
    dsattn.device_status()
    lens = [min((iw.start_pos + i + 1) // iw.ratio, iw.Tv) for i in range(iw.s)]
    units = iw.b * sum(lens)                                   # (query, visible position) pairs
    flops = 2 * iw.H * iw.D * units
    key_bytes = iw.b * iw.Tv * iw.D * 2                        # every key row read once per call
    alg_bytes = key_bytes + iw.b * iw.s * (iw.H * iw.D * 2 + iw.H * 4 + kk * 4)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    torch.cuda._sleep(SLEEP_CYCLES)
    for j in range(args.steps):
        ev[j][0].record()
        call(sets[j % 2])
        ev[j][1].record()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    status = dsattn.device_status()
    per = [a.elapsed_time(b) / 1e3 for a, b in ev]
    elapsed = sum(per)
    units_all, slowest = aggregate(float(units) * args.steps, elapsed, world, device)
    if rank == 0:
        t = statistics.mean(per)
        t_hbm = alg_bytes / (peaks["hbm_gbs"] * 1e9)
        t_tc = flops / (peaks["bf16_tflops"] * 1e12)
        if t_hbm >= t_tc:
            roof = {"bound": "hbm", "achieved": alg_bytes / t / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
        else:
            roof = {"bound": "tensor", "achieved": flops / t / 1e12, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
        roof["frac"] = roof["achieved"] / roof["peak"]
        roof.update({"traffic": profiled_traffic(iw.name, 1, "profiles/{workload}.txt", INDEXER_KERNEL_SOURCES),
                     "kernel_source_sha256_16": kernel_source_hash(INDEXER_KERNEL_SOURCES),
                     "peak_source": peaks["source"], "kernel": "indexer scores + select",
                     "kernel_ms": t * 1e3, "roofline_ms": max(t_hbm, t_tc) * 1e3, "algorithmic_bytes": alg_bytes,
                     "algorithmic_flops": flops})
        out = {"metric": "Indexer (query·visible position)/s scored and selected", "value": units_all / slowest,
               "unit": "(query·position)/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
               "ms_per_step": 1e3 * slowest / args.steps, "higher_is_better": True, "scaling": "weak",
               "vs_baseline": None, "dtype": "bf16 q/k, f32 weights and scores",
               "data": "synthetic (seeded, N(0,1) bf16 q/k, N(0,1)/sqrt(D H) weights)",
               "config": {"workload": f"{iw.name}: b={iw.b} s={iw.s} H={iw.H} D={iw.D} start_pos={iw.start_pos} "
                                      f"ratio={iw.ratio} topk={iw.topk} ({iw.Tv} positions)",
                          "l2": "two input sets alternating; decode keys exceed the L2"},
               "roofline": roof, "clocks": clk, "device_status": status, "gpu_launches": 2 * args.steps}
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_ours(args):
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist_init(world, "nccl")
    from sparse_latent_attention_attn_gb300 import dsattn
    w = wl.WORKLOADS[args.config]
    if args.batch:   # smaller batch of the same workload (profiling captures)
        w = dataclasses.replace(w, b=args.batch, name=f"{w.name}[b={args.batch}]")
    if args.kv == "fp8":
        if not w.decode or w.d != 512:
            print(json.dumps({"error": "--kv fp8 needs a decode workload with head_dim 512"}))
            return 1
        w = dataclasses.replace(w, name=f"{w.name}_fp8kv")
    peaks = load_peaks()

    # enough independent input sets that the gathered rows of consecutive steps miss in L2
    per_set_bytes = w.b * w.m * w.topk * w.d * 2
    nsets = args.sets or max(1, min(24, -(-4 * L2_BYTES // max(per_set_bytes, 1))))
    if w.n_comp * w.b * w.d * 2 > 4 * L2_BYTES:
        nsets = args.sets or 2
    if args.prefill_pairs and w.decode:
        print(json.dumps({"error": "--prefill-pairs needs the prefill workload"}))
        return 1
    sets = [StepSet(w, device, seed=w.seed + 7919 * k + 104729 * rank, kv_mode=args.kv, pairs=args.prefill_pairs)
            for k in range(nsets)]
    torch.cuda.synchronize()

    # one CUDA graph per input set holds a whole step (the three library calls); replaying graphs
    # is how a serving loop drives the path, and it keeps host launch latency out of the timing
    for sset in sets:
        sset.run()
    torch.cuda.synchronize()
    graphs = []
    for sset in sets:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            sset.run()
        graphs.append(g)
    torch.cuda.synchronize()

    # warm-up
    for k in range(args.warmup):
        graphs[k % nsets].replay()
    torch.cuda.synchronize()
    units, alg_bytes, flops = sets[0].counts()
    dsattn.device_status()

    # timed region: exactly K steps, barrier + synchronize on both sides; a device-side sleep
    # before the start event lets the host enqueue the replays ahead of the device
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    torch.cuda._sleep(max(SLEEP_CYCLES, 200_000 * args.steps))
    start.record()
    for k in range(args.steps):
        graphs[k % nsets].replay()
    end.record()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    elapsed_s = start.elapsed_time(end) / 1e3
    status = dsattn.device_status()
    units_all, slowest_s = aggregate(float(units) * args.steps, elapsed_s, world, device)
    value = units_all / slowest_s

    # the sparse_attn launch alone (kernel + combine), CUDA events on its stream around every
    # launch, after a device sleep so the events bracket device time only
    ev_attn = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    torch.cuda.synchronize()
    torch.cuda._sleep(max(SLEEP_CYCLES, 200_000 * args.steps))
    for k in range(args.steps):
        sets[k % nsets].attend(ev_attn[k])
    torch.cuda.synchronize()
    attn_ms = [a.elapsed_time(b) for a, b in ev_attn]

    # end to end through the public API: host inputs in, host output out, every step.  Steps are
    # pipelined the way a serving loop runs them: step i's inputs go up (copy stream) and step
    # i - 1's output comes down (second copy stream) while step i - 1 / i compute, alternating
    # between the resident input sets, with events ordering each set's reuse.  Every step still
    # moves its own inputs and output inside the timed region.
    h2d, d2h = sets[0].io_bytes()
    e2e = None
    if args.e2e_steps > 0:
        # three sets in flight (one uploading, one computing, one downloading); a set beyond the
        # timed-loop sets is made for it when needed
        pipe = list(sets[:3])
        while len(pipe) < 3:
            pipe.append(StepSet(w, device, seed=w.seed + 7919 * len(pipe) + 104729 * rank, kv_mode=args.kv,
                                pairs=args.prefill_pairs))
        host = []
        for st_ in pipe:
            host.append({"q": st_.q.cpu().pin_memory(), "c": st_.cidx.cpu().pin_memory(),
                         "new": (st_.new_kv.cpu() if w.decode else st_.kv[:, : w.s].cpu()).pin_memory(),
                         "o": torch.empty(st_.o.shape, dtype=st_.o.dtype).pin_memory()})
        for st_ in pipe:
            st_.run()
        torch.cuda.synchronize()
        s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        nb = len(pipe)
        in_done = [torch.cuda.Event() for _ in range(nb)]
        cmp_done = [torch.cuda.Event() for _ in range(nb)]
        out_done = [torch.cuda.Event() for _ in range(nb)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        e0.record(s_in)
        for i in range(args.e2e_steps):
            k = i % nb
            st_, hb = pipe[k], host[k]
            with torch.cuda.stream(s_in):
                if i >= nb:
                    s_in.wait_event(cmp_done[k])         # the set's previous step has read its inputs
                st_.q.copy_(hb["q"], non_blocking=True)
                st_.idx[..., w.win_cols:].copy_(hb["c"], non_blocking=True)
                if w.decode:
                    st_.new_kv.copy_(hb["new"], non_blocking=True)
                else:
                    st_.kv[:, : w.s].copy_(hb["new"], non_blocking=True)
                in_done[k].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(in_done[k])
                if i >= nb:
                    s_cmp.wait_event(out_done[k])        # the set's previous output is on the host
                st_.run()
                cmp_done[k].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(cmp_done[k])
                hb["o"].copy_(st_.o, non_blocking=True)
                out_done[k].record(s_out)
        e1.record(s_out)
        torch.cuda.synchronize()
        # each set got the same inputs every step and the kernel is deterministic, so a download
        # that raced its step would show here
        for st_, hb in zip(pipe[: min(nb, args.e2e_steps)], host):
            if not torch.equal(hb["o"], st_.o.cpu()):
                raise RuntimeError("end-to-end pipeline: a host output differs from its device output")
        e2e_units, e2e_s = aggregate(float(units) * args.e2e_steps, e0.elapsed_time(e1) / 1e3, world, device)
        e2e = {"value": e2e_units / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "pipelined_sets": nb}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_sample_rate(w, sets[0], args.cpu_budget, device)

    if rank == 0:
        attn_s = statistics.mean(attn_ms) / 1e3
        t_hbm = alg_bytes / (peaks["hbm_gbs"] * 1e9)
        t_tc = flops / (peaks["bf16_tflops"] * 1e12)
        if t_hbm >= t_tc:
            roof = {"bound": "hbm", "achieved": alg_bytes / attn_s / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
        else:
            roof = {"bound": "tensor", "achieved": flops / attn_s / 1e12, "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s"}
        roof["frac"] = roof["achieved"] / roof["peak"]
        # the capture matching this run: the prefill pairs and the fp8 row store (whose workload
        # name ends in _fp8kv) have their own
        profile_name = w.name + ("_pairs" if args.prefill_pairs else "")
        roof["traffic"] = profiled_traffic(profile_name, 1)
        roof["peak_source"] = peaks["source"]
        roof["kernel"] = ("sparse_attn_ot_kernel (one CTA per work range, transposed accumulator; tokens cut "
                          "across CTAs merge inside a cluster or in a combine kernel)"
                          if sets[0].attn_kernel == dsattn.KERNEL_ONE_CTA else
                          "sparse_attn_tc_kernel (2-CTA cluster, d split) + combine when tokens are cut")
        roof["kernel_source_sha256_16"] = kernel_source_hash()
        roof["kernel_ms"] = attn_s * 1e3
        roof["roofline_ms"] = max(t_hbm, t_tc) * 1e3
        roof["algorithmic_bytes"] = alg_bytes
        roof["algorithmic_flops"] = flops
        out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
               "warmup": args.warmup, "ms_per_step": 1e3 * slowest_s / args.steps, "higher_is_better": True,
               "scaling": "weak", "vs_baseline": None,
               "dtype": ("bf16 q/o, kv as e4m3 codes + per-32 power-of-two exponents, f32 accumulate"
                         if args.kv == "fp8" else "bf16 in/out, f32 accumulate"),
               "data": "synthetic (seeded, N(0,1) bf16 q/kv, N(0,1) f32 sink)"
                       + ("; kv rows stored quantised (fp8 row store)" if args.kv == "fp8" else ""),
               "config": workload_config(w, nsets), "roofline": roof, "cpu_baseline": public(cpu), "e2e": e2e,
               "gpu_launches": sets[0].launches * args.steps, "clocks": clk, "device_status": status,
               "units_per_step": units}
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sets", type=int, default=0, help="input sets to rotate through (0 = automatic)")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (profiling captures)")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--path", choices=["attn", "indexer"], default="attn",
                    help="attn: the sparse_attn step (the bench line); indexer: the Indexer step of --config 2-4")
    ap.add_argument("--prefill-pairs", action="store_true",
                    help="prefill workload: neighbouring queries share one gather (ds_sparse_attn_prefill)")
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="kv rows as bf16, or as the fp8 row store (decode, head_dim 512)")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget", type=float, default=60.0,
                    help="seconds of host work for the whole --impl reference run")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.path == "indexer":
        return run_indexer(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
