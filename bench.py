#!/usr/bin/env python3
"""Throughput of causal + document-masked GQA attention, forward + backward,
for emulated context-parallel ranks on GB300.

One step = the whole hot path for every emulated rank of the workload:
plan (CP position map + block-mask builder), forward (O, LSE), backward
(Delta, dK/dV, dQ), inputs already resident in HBM.  The metric counts only
unmasked (query, key) pairs: FLOPs = sum over ranks and samples of
Hq * pairs * (4*D forward + 10*D backward).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 8b]
    python bench.py --sweep-causal [--steps K]   # throughput vs sequence length
    python bench.py --impl reference ...   # the float64 oracle on host cores

Under torchrun (N > 1) the emulated CP ranks of the workload are dealt to the
processes (rank r of the workload to process r mod N, each process holding
the full K/V), the natural partition of the path: no data-path collective.
When there are more processes than emulated ranks, further copies of the
workload (inputs re-drawn from a shifted seed) fill them.  The step time is
the max over processes.  Rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from document_masked_gqa_gb300 import workloads as wl  # noqa: E402

METRIC = "doc-masked GQA attn fwd+bwd TFLOP/s (unmasked FLOPs), % of GB300 bf16 peak"
UNIT = "TFLOP/s"
# GB300 dense bf16: NVIDIA's HGX B300 figure of 36 PFLOP/s bf16 for 8 GPUs is
# quoted with 2:4 sparsity, i.e. 4.5 PFLOP/s sparse and 2.25 dense per GPU
DATASHEET_BF16_TFLOPS = 2250.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20
CPU_BASELINE_TARGET_S = 15.0  # seconds of host work the bounded oracle sample aims at
PLAN_SORT_MAX = 2048  # launch orders up to this many units are sorted inside the scan kernel


def kernels_per_rank_step(w) -> int:
    """Kernels one rank's step launches: the planner's four (positions,
    block classes, scans + launch orders + the dK/dV work list, lists) plus
    one per launch order too long for the in-block sort (and, for the key
    tiles, one more that lays out the uncut dK/dV work list), the forward's
    two (V to fp16, attention) and the backward's two (dQ with Delta, dK/dV;
    cut dK/dV lists are summed inside the dK/dV kernel)."""
    g = w.n_heads // w.n_kv_heads
    nq = w.batch * ((w.seq_len // w.cp_size) // (128 // g))
    nk = w.batch * (w.seq_len // 128)
    return 4 + int(nq > PLAN_SORT_MAX) + 2 * int(nk > PLAN_SORT_MAX) + 2 + 2


# ------------------------------------------------------------------ counting

def local_positions(seq_len: int, cp_size: int, rank: int) -> np.ndarray:
    c = seq_len // (2 * cp_size)
    a, b = rank, 2 * cp_size - 1 - rank
    return np.concatenate([np.arange(a * c, (a + 1) * c), np.arange(b * c, (b + 1) * c)])


def pairs_per_sample(cu: np.ndarray, batch: int, seq_len: int, cp_size: int,
                     rank: int) -> np.ndarray:
    """Allowed (query, key) pairs of one rank per sample and head."""
    qpos = local_positions(seq_len, cp_size, rank)
    cu = np.asarray(cu, dtype=np.int64)
    out = []
    for b in range(batch):
        g = b * seq_len + qpos
        d = np.searchsorted(cu, g, side="right") - 1
        start = cu[d] - b * seq_len
        out.append(int((qpos - start + 1).sum()))
    return np.asarray(out, dtype=np.int64)


def flops_of(w: wl.Workload, cu, ranks, heads=None, fwd=4, bwd=10) -> float:
    h = w.n_heads if heads is None else heads
    tot = 0
    for r in ranks:
        tot += int(pairs_per_sample(cu, w.batch, w.seq_len, w.cp_size, r).sum())
    return float(h) * tot * (fwd + bwd) * w.head_dim


# ---------------------------------------------------------- distributed bits

def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def delta_bytes(w: wl.Workload) -> int:
    """Algorithmic bytes of one rank's Delta preprocess: reads O (fp32) and dO
    (bf16), writes Delta (fp32), per query row and head."""
    return w.batch * w.local_len * w.n_heads * (6 * w.head_dim + 4)


def plan_bytes(w: wl.Workload, n_docs: int, listed_pairs: int) -> int:
    """Algorithmic bytes of one rank's planner: reads cu_doc_lens; writes the
    position map, document starts (queries) and ends (keys), chunk order,
    tile classes (1 byte per tile pair), row / column counts and pointers,
    the row and column lists (`listed_pairs` non-skipped tile pairs each) and
    the two launch orders."""
    g = w.n_heads // w.n_kv_heads
    nqt = w.local_len // (128 // g)
    nkt = w.seq_len // 128
    b = w.batch
    return (4 * (n_docs + 1) + 4 * w.local_len + 4 * b * w.local_len + 4 * b * w.seq_len
            + 4 * 2 * w.cp_size + b * nqt * nkt
            + 4 * (2 * b * nqt + 1) + 4 * (2 * b * nkt + 1)
            + 4 * 2 * listed_pairs + 4 * (b * nqt + b * nkt))


def host_description() -> dict:
    """CPU model and numpy's BLAS backend of the host the oracle runs on."""
    out = {"cpu_model": None, "blas": None}
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for key in ("model name", "Model", "CPU part"):
            m = re.search(rf"^{key}\s*:\s*(.+)$", info, flags=re.M)
            if m:
                out["cpu_model"] = m.group(1).strip() if key != "CPU part" else f"arm part {m.group(1).strip()}"
                break
    except OSError:
        pass
    try:
        blas = np.show_config(mode="dicts")["Build Dependencies"]["blas"]
        out["blas"] = f"{blas.get('name')} {blas.get('version')}"
    except Exception:  # older numpy: no dict form
        pass
    return out


def copy_workload(w: wl.Workload, copy: int) -> wl.Workload:
    """Copy `copy` of a workload: the same shape, inputs drawn from the seed
    shifted by 7919 per copy (copy 0 is the workload itself)."""
    return dataclasses.replace(w, seed=w.seed + 7919 * copy) if copy else w


def assign_units(world: int, ranks) -> tuple:
    """Work units of an N-process run and the share of each process.  The
    job is ceil(N / R) copies of the workload (R emulated CP ranks); its
    (copy, rank) units are dealt round-robin to the processes, so with
    N <= R the emulated ranks of one workload are split across processes
    (each holds the full K/V: the partition the path has), and with N > R
    whole further copies fill the extra processes.  Returns (shares, copies)
    with shares[p] the (copy, rank) list of process p."""
    ranks = list(ranks)
    copies = -(-world // len(ranks))
    units = [(c, r) for c in range(copies) for r in ranks]
    return [units[p::world] for p in range(world)], copies


def scaling_kind(world: int, copies: int) -> str:
    """'strong' when one copy of the workload is split over several
    processes, else 'weak' (fixed work per process as N grows)."""
    return "strong" if (world > 1 and copies == 1) else "weak"


def algorithmic_bytes(w: wl.Workload, kernel: str) -> int:
    """Bytes one launch of an attention kernel must move at least: every
    input read once and every output written once (q, dO, dQ bf16; O fp32;
    K, V bf16 (the forward reads V's fp16 copy, same size); dK, dV fp32;
    LSE, Delta fp32), whole tensors.  The dQ kernel also computes Delta
    from O and dO."""
    rows = w.batch * w.local_len * w.n_heads
    qsz = rows * w.head_dim * 2                                   # bf16 [B, Lq, Hq, D]
    kvsz = w.batch * w.seq_len * w.n_kv_heads * w.head_dim * 2    # bf16 [B, S, Hkv, D]
    stat = rows * 4                                               # fp32 [B, Hq, Lq]
    if kernel == "fwd":
        return qsz + 2 * kvsz + 2 * qsz + stat                    # q, k, v; o fp32, lse
    if kernel == "dkdv":
        return 2 * qsz + 2 * kvsz + 2 * stat + 2 * 2 * kvsz       # q, dO, k, v, lse, Delta; dk, dv fp32
    if kernel == "dq":
        # q, dO, k, v, lse, O (fp32) in; dq, Delta out (the kernel computes Delta)
        return 2 * qsz + 2 * kvsz + stat + 2 * qsz + qsz + stat
    raise ValueError(kernel)


def reduce_max(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world == 1:
        return
    import torch
    import torch.distributed as dist
    t = torch.zeros(1, device=device)
    dist.all_reduce(t)


# ------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of this GPU's clocks and throttle reasons."""
    FIELDS = ("pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus_id = (bus_id or "").lower()
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        rows = self.rows
        if self.bus_id:
            mine = [r for r in rows if self.bus_id.endswith(r[0].lower()[-12:]) or
                    r[0].lower().endswith(self.bus_id[-12:])]
            rows = mine or rows
        if not rows:
            return None
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = sorted({names[i] for r in rows for i in range(1, 5)
                          if r[4 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ helpers

def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


def _code_only(text: str) -> str:
    """C/C++/CUDA source without comments and with whitespace collapsed, so
    that an edit to a comment does not count as a change of the kernels."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "document_masked_gqa_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str) -> float | None:
    """DRAM bytes per launch from the committed ncu summary of this kernel
    and workload, if it was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", f"traffic_{kernel}_{workload}.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if "=" in line and not line.startswith("#"):
                    k, v = line.split("=", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_sha") != kernel_source_hash():
            return None
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# ------------------------------------------------------------- CPU oracle

def oracle_sample_step(w: wl.Workload, inputs: dict, cu, rows=None, threads=None):
    """One bounded sample of the workload on the float64 oracle: sample 0,
    the query heads of K/V head 0, rank ranks[0], the given local rows (all
    when None; dK/dV then from those rows alone); fwd + bwd on `threads`
    host threads (default: every core).  Returns (counted FLOPs of the
    sample, threads)."""
    from oracle import attention as oa
    from oracle import cp as ocp
    r = w.ranks[0]
    g = w.group
    q = ocp.gather_local(inputs["q"][:1, :, :g], w.seq_len, w.cp_size, r)
    do = ocp.gather_local(inputs["do"][:1, :, :g], w.seq_len, w.cp_size, r)
    k = inputs["k"][:1, :, :1]
    v = inputs["v"][:1, :, :1]
    cu0 = np.asarray([x for x in cu if x <= w.seq_len], dtype=np.int64)
    threads = threads or (os.cpu_count() or 1)
    oa.attention(q, k, v, cu0, w.cp_size, r, do_local=do, rows=rows, threads=threads,
                 kv_grads_from_rows=True)
    return float(g) * sample_pairs(w, cu0, rows) * 14 * w.head_dim, threads


def sample_pairs(w: wl.Workload, cu0, rows=None) -> int:
    """Allowed pairs of the sample's rows (sample 0, rank ranks[0]), per head."""
    qpos = local_positions(w.seq_len, w.cp_size, w.ranks[0])
    sel = qpos if rows is None else qpos[np.asarray(rows)]
    d = np.searchsorted(cu0, sel, side="right") - 1
    return int((sel - cu0[d] + 1).sum())


def oracle_sample_rows(w: wl.Workload, inputs: dict, cu, target_s: float):
    """Rows of the bounded oracle sample: the last local rows (the rank's
    heaviest, at the end of its second chunk), grown from 64 by trial runs
    until one takes about `target_s` / 2 seconds or more.  None = all."""
    n = min(64, w.local_len)
    while n < w.local_len:
        rows = np.arange(w.local_len - n, w.local_len)
        t0 = time.perf_counter()
        oracle_sample_step(w, inputs, cu, rows=rows)
        dt = time.perf_counter() - t0
        if dt >= target_s / 2:
            return rows
        n = min(w.local_len, n * max(2, min(8, int(target_s / max(dt, 1e-3)))))
    return None


def sample_text(w: wl.Workload, rows) -> str:
    what = (f"all {w.local_len} local rows" if rows is None else
            f"local rows {rows[0]}-{rows[-1]} (dK/dV from those rows)")
    return (f"sample 0, query heads 0-{w.group - 1} (K/V head 0), rank {w.ranks[0]}, "
            f"{what}, fwd+bwd, float64 numpy")


def run_reference(args, w: wl.Workload):
    rank, world, _ = dist_info()
    if rank != 0:
        return 0
    cu = wl.cu_doc_lens(w)
    inputs = wl.tensors(w)
    budget = float(os.environ.get("DMA_REF_BUDGET_S", "150"))
    steps_total = args.steps + args.warmup
    # size the sample so that the whole run stays within the budget
    rows = oracle_sample_rows(w, inputs, cu, budget / steps_total)
    sample = sample_text(w, rows)
    times = []
    for i in range(steps_total):
        t0 = time.perf_counter()
        flops, threads = oracle_sample_step(w, inputs, cu, rows=rows)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    sec = sum(times) / len(times)
    value = flops / sec / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample, "threads": threads,
                         "cores_available": os.cpu_count(), **host_description()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(w: wl.Workload) -> dict:
    docs = {"uniform": f"uniform [{w.doc_lo}, {w.doc_hi}]",
            "loguniform": f"log-uniform [{w.doc_lo}, {w.doc_hi}] per sample",
            "single": "one document per sample"}.get(w.doc_dist, w.doc_dist)
    return {"workload": w.name, "seq_len": w.seq_len, "cp_size": w.cp_size,
            "ranks": list(w.ranks), "batch": w.batch, "n_heads": w.n_heads,
            "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "docs": docs,
            "q_prescale": w.q_prescale, "seed": w.seed,
            "l2": "flushed between steps (256 MiB write, outside the timed events)",
            "flops": "unmasked pairs x Hq x (4D fwd + 10D bwd)"}


# --------------------------------------------------------------- GPU arm

def run_gpu(args, w: wl.Workload):
    import torch

    import document_masked_gqa_gb300 as dma

    rank, world, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    shares, copies = assign_units(world, w.ranks)
    stream = torch.cuda.current_stream(dev)

    # every unit of the whole job, for the FLOP count; this process's own
    copy_of = {c: copy_workload(w, c) for c in range(copies)}
    cu_of = {c: wl.cu_doc_lens(copy_of[c]) for c in range(copies)}
    flops_job = sum(flops_of(copy_of[c], cu_of[c], (r,)) for sh in shares for c, r in sh)
    mine = shares[rank]
    inputs_of = {c: wl.tensors(copy_of[c]) for c in sorted({c for c, _ in mine})}
    dev_of = {}
    for c, inp in inputs_of.items():
        dev_of[c] = {"cu": torch.from_numpy(cu_of[c]).to(dev), "k": inp["k"].to(dev),
                     "v": inp["v"].to(dev)}
    units = []
    for c, r in mine:
        D = dev_of[c]
        need = dma.dma_plan_workspace_bytes(w.batch, w.seq_len, w.cp_size, w.n_heads,
                                            w.n_kv_heads, w.head_dim)
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
        plan = dma.dma_plan(D["cu"], w.batch, w.seq_len, w.cp_size, r, w.n_heads, w.n_kv_heads,
                            w.head_dim, workspace=ws)
        q = dma.dma_cp_gather(plan, inputs_of[c]["q"].to(dev))
        do = dma.dma_cp_gather(plan, inputs_of[c]["do"].to(dev))
        o, lse = dma.dma_attn_fwd(plan, q, D["k"], D["v"])
        dq, dk, dv = dma.dma_attn_bwd(plan, q, D["k"], D["v"], o, lse, do)
        pairs = int(pairs_per_sample(cu_of[c], w.batch, w.seq_len, w.cp_size, r).sum())
        units.append(dict(c=c, r=r, ws=ws, q=q, do=do, o=o, lse=lse, dq=dq, dk=dk, dv=dv,
                          k=D["k"], v=D["v"], cu=D["cu"], pairs=pairs))
    torch.cuda.synchronize(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    names = ("plan", "fwd", "dq", "dkdv")

    def step(record: bool):
        evs = []
        for U in units:
            e = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] \
                if record else None
            if record:
                e[0].record(stream)
            plan = dma.dma_plan(U["cu"], w.batch, w.seq_len, w.cp_size, U["r"], w.n_heads,
                                w.n_kv_heads, w.head_dim, workspace=U["ws"])
            U["plan"] = plan
            if record:
                e[1].record(stream)
            dma.dma_attn_fwd(plan, U["q"], U["k"], U["v"], U["o"], U["lse"])
            if record:
                e[2].record(stream)
            # the backward: dQ with Delta in one kernel, then dK/dV
            dma.dma_attn_bwd_dq_delta(plan, U["q"], U["k"], U["v"], U["o"], U["lse"], U["do"],
                                      U["dq"])
            if record:
                e[3].record(stream)
            dma.dma_attn_bwd_dkdv(plan, U["q"], U["k"], U["v"], U["lse"], U["do"], U["dk"],
                                  U["dv"])
            if record:
                e[4].record(stream)
            evs.append(e)
        return evs

    for _ in range(args.warmup):
        step(False)
        flush.zero_()
    torch.cuda.synchronize(dev)
    for U in units:
        st = dma.dma_plan_check(U["plan"])
        if st != 0:
            raise RuntimeError(f"plan status {st}: {dma.status_str(st)}")

    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id if hasattr(
            torch.cuda.get_device_properties(dev), "pci_bus_id") else None
    except Exception:
        bus = None
    sampler = ClockSampler(bus)
    sampler.start()
    time.sleep(0.3)

    barrier(world, dev)
    torch.cuda.synchronize(dev)
    step_pairs = []
    all_evs = []
    for _ in range(args.steps):
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        evs = step(True)
        s1.record(stream)
        step_pairs.append((s0, s1))
        all_evs.append(evs)
        flush.zero_()  # L2 flush between steps, outside the step's events
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    clocks = sampler.stop()

    ms_steps = [a.elapsed_time(b) for a, b in step_pairs]
    ms_local = sum(ms_steps) / len(ms_steps)
    # per unit and kernel: mean ms per launch
    per_unit = []
    for ui, U in enumerate(units):
        km = {n: 0.0 for n in names}
        for evs in all_evs:
            e = evs[ui]
            for i, n in enumerate(names):
                km[n] += e[i].elapsed_time(e[i + 1])
        km = {n: km[n] / args.steps for n in names}
        per_unit.append({"copy": U["c"], "rank": U["r"], "pairs_per_head": U["pairs"],
                         "process": rank, "ms": {n: round(km[n], 5) for n in names},
                         "ms_total": round(sum(km.values()), 5)})
    kms = {n: sum(u["ms"][n] for u in per_unit) / len(per_unit) for n in names}
    for U in units:
        st = dma.dma_plan_check(U["plan"])
        if st != 0:
            raise RuntimeError(f"plan status {st}: {dma.status_str(st)}")
    if world > 1:
        import torch.distributed as dist
        gathered = [None] * world
        dist.all_gather_object(gathered, per_unit)
        per_unit_all = [u for part in gathered for u in part]
    else:
        per_unit_all = per_unit

    ms = reduce_max(ms_local, world, dev)
    value = flops_job / (ms * 1e-3) / 1e12

    # roofline of the dominant kernel (largest share of the step), on this
    # process's launches
    algo = {"fwd": 4, "dkdv": 8, "dq": 6}  # contractions over D per pair and head, x D
    dom = max(("fwd", "dkdv", "dq"), key=lambda n: kms[n])
    mean_pairs = sum(U["pairs"] for U in units) / len(units)
    algo_flops = w.n_heads * mean_pairs * algo[dom] * w.head_dim
    achieved = algo_flops / (kms[dom] * 1e-3) / 1e12
    peaks = measured_peaks()
    peak = peaks.get("bf16_tflops")
    peak_src = "measured burst (MEASURED_PEAKS.json bf16_tflops)"
    if not peak:
        peak, peak_src = FALLBACK_BF16_TFLOPS, "fallback"
    hbm_peak = peaks.get("hbm_gbs")
    abytes = algorithmic_bytes(w, dom)
    traffic = profiled_traffic(dom, w.name)
    roof = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
            "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": peak_src,
            "traffic": traffic, "algorithmic_flops_per_launch": algo_flops,
            "algorithmic_bytes": abytes,
            "traffic_over_algorithmic": (traffic / abytes) if traffic else None,
            # the same launch against the HBM roofline (the second bound that
            # matters where masks leave little work per byte)
            "hbm_achieved_gbs": abytes / (kms[dom] * 1e-3) / 1e9,
            "hbm_frac": (abytes / (kms[dom] * 1e-3) / 1e9 / hbm_peak) if hbm_peak else None,
            "kernel_ms": {n: round(kms[n], 5) for n in names}}

    # the HBM-bound part against the measured copy bandwidth: the planner
    # (latency-bound: a handful of small launches).  Delta is computed inside
    # the dQ kernel, whose O reads count in its algorithmic bytes.
    hbm = {"peak_gbs": hbm_peak, "peak_source": "measured copy (MEASURED_PEAKS.json hbm_gbs)"}
    try:
        listed = [int(dma.plan_arrays(U["plan"])["row_ptr"][-1]) for U in units]
        n_docs = len(cu_of[units[0]["c"]]) - 1
        pb = sum(plan_bytes(w, n_docs, n) for n in listed) / len(listed)
        hbm["plan"] = {"bytes": pb, "ms": kms["plan"], "gbs": pb / (kms["plan"] * 1e-3) / 1e9,
                       "note": "latency-bound: one memset and four small launches"}
    except Exception as exc:  # the line is printed regardless
        hbm["plan"] = {"error": str(exc)[:120]}
    if hbm_peak and "gbs" in hbm["plan"]:
        hbm["plan"]["frac"] = hbm["plan"]["gbs"] / hbm_peak
    # the same step counted without the backward's recompute (4D + 8D per pair)
    flops_mfu = sum(flops_of(copy_of[c], cu_of[c], (r,), fwd=4, bwd=8)
                    for sh in shares for c, r in sh)
    mfu_value = flops_mfu / (ms * 1e-3) / 1e12
    mfu = {"value": mfu_value, "unit": UNIT, "count": "4D fwd + 8D bwd per pair and head",
           "pct_of_measured_peak": 100.0 * mfu_value / world / peak}

    # end to end through the public API: pinned host inputs -> device -> step ->
    # results back to pinned host memory, every step
    e2e = run_e2e(args, w, dma, dev, mine, copy_of, cu_of, inputs_of, flops_job, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        inputs = inputs_of[0]
        rows = oracle_sample_rows(w, inputs, cu_of[0], CPU_BASELINE_TARGET_S)
        t0 = time.perf_counter()
        fl, threads = oracle_sample_step(w, inputs, cu_of[0], rows=rows)
        dt = time.perf_counter() - t0
        cpu = {"value": fl / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
               "threads": threads, "cores_available": os.cpu_count(), **host_description(),
               "sample": f"{sample_text(w, rows)}, {dt:.1f} s"}

    if rank == 0:
        slowest = max(per_unit_all, key=lambda u: u["ms_total"])
        fastest = min(per_unit_all, key=lambda u: u["ms_total"])
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": scaling_kind(world, copies),
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(config_of(w), copies=copies,
                           units_per_process=[[list(u) for u in sh] for sh in shares]),
            "pct_of_measured_peak": 100.0 * value / world / peak,
            "pct_of_datasheet_peak": 100.0 * value / world / DATASHEET_BF16_TFLOPS,
            "roofline": roof, "mfu_style": mfu, "hbm": hbm, "cpu_baseline": cpu, "e2e": e2e,
            "per_rank": per_unit_all,
            "rank_imbalance": {"slowest_over_fastest": slowest["ms_total"] / fastest["ms_total"],
                               "slowest": [slowest["copy"], slowest["rank"]],
                               "fastest": [fastest["copy"], fastest["rank"]]},
            "gpu_launches": kernels_per_rank_step(w) * len(units) * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_e2e(args, w, dma, dev, mine, copy_of, cu_of, inputs_of, flops_job, world):
    import torch
    steps = max(3, min(args.steps, 20))
    per = []
    host_kv = {}
    for c in sorted(inputs_of):
        host_kv[c] = {"k": inputs_of[c]["k"].pin_memory(), "v": inputs_of[c]["v"].pin_memory(),
                      "cu": torch.from_numpy(cu_of[c]).pin_memory()}
    for c, r in mine:
        pos = torch.from_numpy(local_positions(w.seq_len, w.cp_size, r))
        h_q = inputs_of[c]["q"][:, pos].contiguous().pin_memory()
        h_do = inputs_of[c]["do"][:, pos].contiguous().pin_memory()
        h_k = host_kv[c]["k"]
        outs = {"o": torch.empty(h_q.shape, dtype=torch.float32).pin_memory(),
                "lse": torch.empty(w.batch, w.n_heads, w.local_len).pin_memory(),
                "dq": torch.empty_like(h_q).pin_memory(),
                "dk": torch.empty(h_k.shape, dtype=torch.float32).pin_memory(),
                "dv": torch.empty(h_k.shape, dtype=torch.float32).pin_memory()}
        per.append((c, r, h_q, h_do, outs))
    h2d = sum(t.nbytes for kv in host_kv.values() for t in kv.values()) + \
        sum(p[2].nbytes + p[3].nbytes for p in per)
    d2h = sum(sum(t.nbytes for t in p[4].values()) for p in per)

    # Within a step the copies overlap the compute: inputs come in on one
    # stream (dO after q, k, v, so that the forward starts first), the
    # results go out on another as soon as the kernel producing them is
    # done (O and LSE during the backward).  A step starts only after the
    # previous one has finished, so every step pays for its own copies.
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    stream = torch.cuda.Stream(dev)  # compute; the binding launches on the current stream

    def one():
        s_in.wait_stream(stream)
        with torch.cuda.stream(s_in):
            kv = {c: {n: t.to(dev, non_blocking=True) for n, t in hk.items()}
                  for c, hk in host_kv.items()}
            qs = [h_q.to(dev, non_blocking=True) for _, _, h_q, _, _ in per]
            ev_qkv = torch.cuda.Event()
            ev_qkv.record(s_in)
            dos = [h_do.to(dev, non_blocking=True) for _, _, _, h_do, _ in per]
            ev_do = torch.cuda.Event()
            ev_do.record(s_in)
        for t in [t for d in kv.values() for t in d.values()] + qs + dos:
            t.record_stream(stream)
        stream.wait_event(ev_qkv)
        fwd_out = []
        for (c, r, h_q, h_do, outs), q in zip(per, qs):
            plan = dma.dma_plan(kv[c]["cu"], w.batch, w.seq_len, w.cp_size, r, w.n_heads,
                                w.n_kv_heads, w.head_dim)
            o, lse = dma.dma_attn_fwd(plan, q, kv[c]["k"], kv[c]["v"])
            ev = torch.cuda.Event()
            ev.record(stream)
            s_out.wait_event(ev)
            with torch.cuda.stream(s_out):
                outs["o"].copy_(o, non_blocking=True)
                outs["lse"].copy_(lse, non_blocking=True)
            o.record_stream(s_out)
            lse.record_stream(s_out)
            fwd_out.append((plan, o, lse))
        stream.wait_event(ev_do)
        for (c, r, h_q, h_do, outs), q, do, (plan, o, lse) in zip(per, qs, dos, fwd_out):
            dq, dk, dv = dma.dma_attn_bwd(plan, q, kv[c]["k"], kv[c]["v"], o, lse, do)
            ev = torch.cuda.Event()
            ev.record(stream)
            s_out.wait_event(ev)
            with torch.cuda.stream(s_out):
                outs["dq"].copy_(dq, non_blocking=True)
                outs["dk"].copy_(dk, non_blocking=True)
                outs["dv"].copy_(dv, non_blocking=True)
            for t in (dq, dk, dv):
                t.record_stream(s_out)
        stream.wait_stream(s_out)

    with torch.cuda.stream(stream):
        for _ in range(2):
            one()
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    # three timed runs of `steps` steps each; the median run is reported
    # (host-side variation between runs has been seen to move this leg by
    # tens of percent while the device-side step time stays put)
    runs = []
    for _ in range(3):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(steps):
                one()
            b.record(stream)
        torch.cuda.synchronize(dev)
        runs.append(a.elapsed_time(b) / steps)
    ms = reduce_max(sorted(runs)[1], world, dev)
    return {"value": flops_job / (ms * 1e-3) / 1e12, "unit": UNIT,
            "ms_per_step": ms, "steps": steps, "runs_ms_per_step": [round(x, 4) for x in runs],
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


SWEEP_LENGTHS = (8192, 16384, 32768, 65536, 131072)


def run_sweep(args) -> int:
    """Throughput against sequence length on one GPU: CP = 1, batch 1, the
    405B shard's heads (Hq = 16, Hkv = 1, D = 128), plain causal (one
    document) and document-masked (log-uniform lengths in [1024,
    min(65536, S/2)]) at 8K ... 128K.  One JSON line per configuration; `rel` = its TFLOP/s over
    the 128K causal value, the kind of curve the pages' Figure 11 draws as
    relative HFU.  Inputs resident, L2 flushed between steps, CUDA events
    around each step (plan, forward, backward)."""
    import torch
    import document_masked_gqa_gb300 as dma
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    peak = measured_peaks().get("bf16_tflops") or FALLBACK_BF16_TFLOPS
    lines = []
    for mask in ("causal", "docs"):
        for n, s_len in enumerate(SWEEP_LENGTHS):
            if mask == "causal":
                w = wl.custom(f"sweep-causal-{s_len}", s_len, 1, 1, 16, 1, 128, "single",
                              seed=2000 + n)
            else:
                w = wl.custom(f"sweep-docs-{s_len}", s_len, 1, 1, 16, 1, 128, "loguniform",
                              1024, min(65536, s_len // 2), seed=2100 + n)
            cu_np = wl.cu_doc_lens(w)
            inp = {k: v.to(dev) for k, v in wl.tensors(w).items()}
            cu = torch.from_numpy(cu_np).to(dev)
            need = dma.dma_plan_workspace_bytes(w.batch, w.seq_len, 1, w.n_heads, w.n_kv_heads,
                                                w.head_dim)
            ws = torch.empty(need, dtype=torch.uint8, device=dev)
            out = {}

            def step():
                plan = dma.dma_plan(cu, w.batch, w.seq_len, 1, 0, w.n_heads, w.n_kv_heads,
                                    w.head_dim, workspace=ws)
                if not out:
                    o, lse = dma.dma_attn_fwd(plan, inp["q"], inp["k"], inp["v"])
                    dq, dk, dv = dma.dma_attn_bwd(plan, inp["q"], inp["k"], inp["v"], o, lse,
                                                  inp["do"])
                    out.update(o=o, lse=lse, dq=dq, dk=dk, dv=dv)
                else:
                    dma.dma_attn_fwd(plan, inp["q"], inp["k"], inp["v"], out["o"], out["lse"])
                    dma.dma_attn_bwd(plan, inp["q"], inp["k"], inp["v"], out["o"], out["lse"],
                                     inp["do"], out["dq"], out["dk"], out["dv"])
                return plan

            for _ in range(args.warmup):
                step()
                flush.zero_()
            torch.cuda.synchronize(dev)
            times = []
            for _ in range(args.steps):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                plan = step()
                b.record(stream)
                flush.zero_()
                times.append((a, b))
            torch.cuda.synchronize(dev)
            st = dma.dma_plan_check(plan)
            if st != 0:
                raise RuntimeError(f"plan status {st}: {dma.status_str(st)}")
            ms = sum(a.elapsed_time(b) for a, b in times) / len(times)
            tf = flops_of(w, cu_np, (0,)) / (ms * 1e-3) / 1e12
            lines.append({"sweep": "causal-vs-docs", "mask": mask, "seq_len": s_len,
                          "docs": len(cu_np) - 1, "ms_per_step": ms, "tflops": tf,
                          "pct_of_measured_peak": 100.0 * tf / peak})
            del inp, out, ws
            torch.cuda.empty_cache()
    ref = [x["tflops"] for x in lines if x["mask"] == "causal" and x["seq_len"] == SWEEP_LENGTHS[-1]]
    for x in lines:
        x["rel"] = x["tflops"] / ref[0] if ref else None
        print(json.dumps(x), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--workload", default="8b", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep-causal", action="store_true",
                    help="throughput against sequence length, causal vs document-masked")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.sweep_causal:
        return run_sweep(args)
    w = wl.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_gpu(args, w)


if __name__ == "__main__":
    sys.exit(main())
