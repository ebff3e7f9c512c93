#!/usr/bin/env python
"""Benchmark of one DeFT tree-attention decode step on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl deft|reference]

A step is one pass of the whole hot path (phase-1 partial attention over all
chunks + phase-2 LSE merge) on one synthetic tree whose KV cache and queries
are already resident in HBM.  The default workload is the shared-prefix
few-shot decode tree (4096-token prefix, 32 branches of 256 tokens, one
query per branch tip, 32 query / 32 KV heads, head_dim 128, bf16); other
shapes via --config 1..6.  The L2 cache is flushed between timed steps,
outside the timed events: a 2 x L2 memset, then a read of another 2 x L2
buffer, so that the step starts with a cold L2 that holds no dirty lines
(their write-back would otherwise land inside the timed region).

Prints one JSON line (rank 0).  `value` is microseconds per step (lower is
better); for N > 1 the ranks run independent replicas and `value` is the
whole job's time per step (max over ranks of the timed region / (K * N)).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "tree-attention µs/step; achieved HBM GB/s vs unique-KV-bytes roofline"
SPEC_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", type=int, default=2)
    ap.add_argument("--chunk-target", type=int, default=256)
    ap.add_argument("--impl", choices=["deft", "reference"], default="deft")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the naive, e2e, CPU-baseline and per-workload legs")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the per-workload entries (configs 1-7) of the line")
    ap.add_argument("--shard", choices=["replicas", "heads"], default="replicas",
                    help="N > 1: independent replicas of the step, or one step split by KV head")
    ap.add_argument("--tensor-pack", type=int, default=-1,
                    help="plan with DEFT_PLAN_TENSOR_PACK (1), without (0), or when head_dim is 128 (-1)")
    ap.add_argument("--step-flags", type=int, default=0,
                    help="deft_tree_attn_ex flags for the timed step (4: merge in a separate launch)")
    ap.add_argument("--profile-case", default=None, choices=sorted(PROFILE_CASES),
                    help="run a few steps of a small named case for an ncu capture, print nothing else")
    ap.add_argument("--range", action="store_true",
                    help="with --profile-case: bracket one more step with cudaProfilerStart/Stop "
                         "(ncu --replay-mode range --profile-from-start off)")
    return ap.parse_args()


# Small seeded cases of the benchmark workloads' shapes, for ncu captures that
# must stay small (a few hundred MB on the device).
PROFILE_CASES = {
    # 3 requests x (4000-token prefix + 64-node token tree), 32/32 heads: tensor-core launch, 64 rows
    "speculative_3req": lambda: W.speculative_forest(requests=3),
    # 32 independent 2048-token sequences, GQA 32/8: CUDA-core launch, 4 rows
    "control_32x2048": lambda: W.imbalance_tree(control=True, leaves=32),
    # the few-shot tree (4096-token prefix + 32 x 256)
    "few_shot": lambda: W.config(2),
    # the reasoning tree (4 levels, 128 queries, GQA 32/8)
    "reasoning": lambda: W.config(4),
    # the imbalance shape with 64 leaves: the 32768-token prefix at 256 rows (two 128-row
    # blocks reading the same KV), 64 leaves of 64-8192 tokens
    "imbalance_64leaves": lambda: W.imbalance_tree(leaves=64),
}


def run_profile_case(args):
    """A few steps of a named case on cuda:0 (the capture target); with
    --range one more step bracketed for ncu's range replay."""
    import torch
    import shared_prefix_kv_deft_gb300 as deft
    spec = PROFILE_CASES[args.profile_case]()
    lay = W.paged_layout(spec)
    t = W.make_tensors(spec, lay, device="cuda")
    npo = torch.from_numpy(lay.node_page_off).cuda()
    pid = torch.from_numpy(lay.page_id).cuda()
    plan = deft.Plan(spec.parent, spec.node_len, spec.query_node, args.chunk_target, spec.gqa_group,
                     tensor_pack=tensor_pack(args, spec))
    plan.upload()
    bufs = deft.alloc_buffers(plan, spec.num_queries, spec.num_q_heads, spec.head_dim)

    def step():
        deft.deft_tree_attn(t.q, t.k_pages, t.v_pages, npo, pid, plan, bufs=bufs, flags=args.step_flags)
    for _ in range(max(1, args.steps)):
        step()
    torch.cuda.synchronize()
    if args.range:
        torch.cuda.profiler.start()
        step()
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
    if plan.step_status() != 0:
        raise RuntimeError("a kernel reported a failed wait")
    print("ok", spec.name)
    return 0


def tensor_pack(args, spec) -> bool:
    """Tensor-packed plans for head_dim 128 (the tcgen05 path) unless told."""
    return bool(args.tensor_pack) if args.tensor_pack >= 0 else spec.head_dim == 128


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", FALLBACK_HBM_GBS)), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# Algorithmic bytes (no re-reads counted): what one launch must move at least.
# ---------------------------------------------------------------------------

def algorithmic_bytes(plan, spec, family="tree"):
    """Per-launch algorithmic bytes, keyed like the trace records."""
    d, Hq, Hkv = spec.head_dim, spec.num_q_heads, spec.num_kv_heads
    kv_tok = 2 * Hkv * d * 2                      # K + V bytes of one token, all KV heads
    part_row = (d + 1) * 4                        # one fp32 partial (o and lse)
    pre = "" if family == "tree" else "naive_"
    seg_off = plan.get(pre + "chunk_seg_off")
    seg_len = plan.get(pre + "seg_tok_len")
    tok = np.add.reduceat(seg_len, seg_off[:-1]) if len(seg_len) else np.zeros(0, np.int64)
    G = spec.gqa_group
    out = {}
    if family == "tree":
        fams = {(0, 0): plan.get("fma_items").reshape(-1, 3),
                (1, 0): plan.get("mma_items").reshape(-1, 3),
                (0, 1): plan.get("fallback_items").reshape(-1, 3)}
    else:
        fams = {(0, 0): np.zeros((0, 3), np.int32)}
    for (kern, fb), items in fams.items():
        if len(items) == 0:
            continue
        rows = (items[:, 2] - items[:, 1]) * G
        if kern == 1:
            b = (((rows + 1) // 2 + 15) // 16) - 1          # column bucket (16 (b + 1) per warpgroup)
        else:
            b = np.select([rows <= 1, rows <= 2, rows <= 4, rows <= 8], [0, 1, 2, 3], 4)
        groups = {int(x): b == x for x in np.unique(b)}
        groups[-1] = np.ones(len(items), bool)             # every bucket (one launch for all)
        for bucket, sel in groups.items():
            chunks = np.unique(items[sel, 0])
            kv = int(tok[chunks].sum()) * kv_tok
            q = int(rows[sel].sum()) * Hkv * d * 2
            part = int(rows[sel].sum()) * Hkv * part_row
            out[(kern, bucket, fb)] = {"kv": kv, "q": q, "partials": part, "total": kv + q + part}
    return out


def phase2_bytes(plan, spec, family="tree"):
    d, Hq = spec.head_dim, spec.num_q_heads
    slots = plan.stats["num_slots" if family == "tree" else "naive_num_slots"]
    Q = spec.num_queries
    return slots * Hq * (d + 1) * 4 + Q * Hq * (d * 2 + 4) + (Q + 1 + slots) * 4


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix=f"deft_clocks_rank{device_index}_", suffix=".csv")
        os.close(fd)
        sel = []
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES")
            sel = ["-i", vis.split(",")[device_index] if vis else str(device_index)]
        self.sel = sel
        self.cmd = ["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                    "-lms", "50"]

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(self.cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()
        try:
            os.unlink(self.path)
        except OSError:
            pass

    def summary(self, t0: float, t1: float):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[2].split()[0]), float(parts[3].split()[0]),
                             parts[4], parts[6:10]))
            except (ValueError, IndexError):
                continue
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        window = "timed region"
        if not inside:
            inside, window = rows, "whole run (timed region shorter than the sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[4]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside), "window": window, "gpu": " ".join(self.sel)}


# ---------------------------------------------------------------------------
# ncu summary (committed under profiles/) for the roofline's traffic figure
# ---------------------------------------------------------------------------

# Sources that decide what the phase-1 kernels read and write: the kernels,
# their launch shapes and the planner (not the C-ABI glue).
HOST_GLUE = ("capi.cu", "noalloc.cu")


def strip_comments(src: str) -> str:
    """C/C++ source without its comments and blank lines (string and
    character literals kept), so that a change to comments alone leaves the
    source hash, and the counters recorded against it, as they were."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(l.rstrip() for l in "".join(out).split("\n") if l.strip())


def kernel_source_hash():
    """Hash of the kernel, launch and planner sources (comments left out)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "shared_prefix_kv_deft_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h", ".cpp")) and f not in HOST_GLUE:
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                h.update(strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, cfg: int):
    """DRAM bytes per launch from profiles/ncu_traffic.json, or None when no
    capture exists for this kernel/workload or the sources changed since."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    ent = d.get(f"config{cfg}", {}).get(kernel)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# Reference arm: the fp64 CPU oracle on the host cores
# ---------------------------------------------------------------------------

def host_inputs(spec, layout, t):
    return (W.bf16_bits(t.q), W.bf16_bits(t.k_pages), W.bf16_bits(t.v_pages))


def oracle_step(oracle, spec, layout, bits, subset, threads=0):
    return oracle.tree_attn(bits[0], bits[1], bits[2], layout.node_page_off, layout.page_id,
                            layout.page_size, spec.parent, spec.node_len, spec.query_node,
                            spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                            1.0 / math.sqrt(spec.head_dim), query_subset=subset,
                            query_pos=spec.query_pos, threads=threads)


def time_oracle(oracle, spec, layout, bits, budget_s, threads=0):
    """us per full step of the oracle on `threads` host threads (0: all),
    timed on a sample of queries sized to about `budget_s` seconds."""
    Q = spec.num_queries
    # Calibrate on one query, then size the sample to the budget.
    t0 = time.perf_counter()
    oracle_step(oracle, spec, layout, bits, [0], threads)
    per_q = max(time.perf_counter() - t0, 1e-6)
    nq = int(max(1, min(Q, budget_s / 2 / per_q)))
    subset = np.linspace(0, Q - 1, nq).astype(np.int32)
    reps, spent = 0, 0.0
    while spent < budget_s / 2 and reps < 50:
        t0 = time.perf_counter()
        oracle_step(oracle, spec, layout, bits, subset, threads)
        spent += time.perf_counter() - t0
        reps += 1
    return spent / reps * (Q / nq) * 1e6, f"{nq} of {Q} queries x all {spec.num_q_heads} heads, " \
                                           f"{reps} run(s), scaled to the full step"


def cpu_baseline(spec, layout, bits, budget_s=12.0, single_thread=True):
    """Time the oracle, as it stands, on a bounded sample of the workload: on
    all host threads (the value) and on one thread."""
    import oracle
    oracle.load()
    us, sample = time_oracle(oracle, spec, layout, bits, budget_s)
    out = {"value": us, "unit": "us/step", "cores": oracle.max_threads(), "kind": "oracle", "sample": sample}
    if single_thread:
        us1, sample1 = time_oracle(oracle, spec, layout, bits, budget_s / 2, threads=1)
        out["single_thread"] = {"value": us1, "unit": "us/step", "cores": 1, "sample": sample1}
    return out


def max_over_ranks(x: float, pg, device) -> float:
    """The largest of every rank's x (x itself without a process group)."""
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_us_per_step(slowest_ms_per_step: float, world: int) -> float:
    """Whole-job time per step: `world` replicas each finish a step in the
    slowest rank's time, so the job completes `world` steps in that time."""
    return slowest_ms_per_step * 1e3 / world


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    spec = W.config(args.config)
    layout = W.paged_layout(spec)
    t = W.make_tensors(spec, layout, device="cpu")
    bits = host_inputs(spec, layout, t)
    import oracle
    oracle.load()
    Q = spec.num_queries
    t0 = time.perf_counter()
    oracle_step(oracle, spec, layout, bits, [0])
    per_q = max(time.perf_counter() - t0, 1e-6)
    # Each step is a bounded sample sized so that the whole run takes a few minutes.
    total_budget = 150.0
    per_step = total_budget / max(1, args.steps + args.warmup)
    nq = int(max(1, min(Q, per_step / per_q)))
    subset = np.linspace(0, Q - 1, nq).astype(np.int32)
    for _ in range(args.warmup):
        oracle_step(oracle, spec, layout, bits, subset)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(oracle, spec, layout, bits, subset)
        times.append(time.perf_counter() - t0)
    us = statistics.mean(times) * (Q / nq) * 1e6
    line = {"impl": "reference", "metric": METRIC, "value": us, "unit": "us/step",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": spec.name, "global_batch": Q, "parallelism": "host cores"},
            "cpu_baseline": {"value": us, "unit": "us/step", "cores": oracle.max_threads(),
                             "kind": "oracle",
                             "sample": f"{nq} of {Q} queries x all heads per step, scaled"},
            "e2e": {"value": us, "unit": "us/step", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def head_shard(num_q_heads: int, num_kv_heads: int, rank: int, world: int):
    """KV heads [k0, k1) and their query heads [q0, q1) of rank `rank` when a
    step is split by KV head over `world` devices (whole GQA groups, no
    exchange: every query head reads only its own KV head)."""
    if num_kv_heads % world:
        raise ValueError(f"{num_kv_heads} KV heads do not split over {world} ranks")
    G = num_q_heads // num_kv_heads
    per = num_kv_heads // world
    k0, k1 = rank * per, (rank + 1) * per
    return k0 * G, k1 * G, k0, k1


class Runner:
    """One workload on one device: inputs resident in HBM, a plan, buffers,
    and the timing legs of the benchmark."""

    def __init__(self, deft, torch, dev, spec, args, pg=None, shard=None):
        self.deft, self.torch, self.dev, self.args, self.pg = deft, torch, dev, args, pg
        if shard is not None:
            # This rank's KV heads and their query heads, the same tree and plan.
            q0, q1, k0, k1 = shard
            spec = dataclasses.replace(spec, name=spec.name + f"_kvheads{k0}-{k1}", num_q_heads=q1 - q0,
                                       num_kv_heads=k1 - k0)
        self.spec = spec
        self.layout = W.paged_layout(spec)
        self.t = W.make_tensors(spec, self.layout, device=dev)
        self.npo = torch.from_numpy(self.layout.node_page_off).to(dev)
        self.pid = torch.from_numpy(self.layout.page_id).to(dev)
        self.tp = tensor_pack(args, spec)
        self.plan = deft.Plan(spec.parent, spec.node_len, spec.query_node, args.chunk_target, spec.gqa_group,
                              query_pos=spec.query_pos, tensor_pack=self.tp)
        self.plan.upload()
        self.bufs = deft.alloc_buffers(self.plan, spec.num_queries, spec.num_q_heads, spec.head_dim, dev)
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
        self.flush_rd = torch.zeros(2 * l2 // 8, dtype=torch.int64, device=dev)
        self.stream = torch.cuda.current_stream(dev)

    def flush_l2(self):
        self.flush.zero_()
        self.flush_rd.sum()

    def step(self):
        t = self.t
        self.deft.deft_tree_attn(t.q, t.k_pages, t.v_pages, self.npo, self.pid, self.plan, bufs=self.bufs,
                                 flags=self.args.step_flags)

    def naive_step(self):
        t = self.t
        self.deft.deft_naive_attn(t.q, t.k_pages, t.v_pages, self.npo, self.pid, self.plan, bufs=self.bufs)

    def barrier(self):
        self.torch.cuda.synchronize(self.dev)
        if self.pg is not None:
            self.pg.barrier()

    def timed(self, fn, n, trace=False):
        """n steps, each after an L2 flush outside its events; ms per step."""
        torch, deft = self.torch, self.deft
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        if trace:
            deft.trace_read()
            deft.trace_enable(True)
        self.barrier()
        w0 = time.time()
        for i in range(n):
            self.flush_l2()
            starts[i].record(self.stream)
            fn()
            ends[i].record(self.stream)
        self.barrier()
        w1 = time.time()
        recs = []
        if trace:
            deft.trace_enable(False)
            recs = deft.trace_read()
        return [s.elapsed_time(e) for s, e in zip(starts, ends)], recs, w0, w1

    def warm(self, n):
        for _ in range(n):
            self.flush_l2()
            self.step()
        self.torch.cuda.synchronize(self.dev)

    def kernels(self, recs, steps):
        """Per-kernel durations (library event trace) and algorithmic bytes."""
        spec, plan = self.spec, self.plan
        alg = algorithmic_bytes(plan, spec)
        p2 = phase2_bytes(plan, spec)
        # A CUDA-core launch whose item count is not its bucket's covers every bucket.
        fma_items = plan.get("fma_items").reshape(-1, 3)
        rows = (fma_items[:, 2] - fma_items[:, 1]) * spec.gqa_group
        fb = np.select([rows <= 1, rows <= 2, rows <= 4, rows <= 8], [0, 1, 2, 3], 4)
        # Likewise a tensor-core launch whose item count is not its width's
        # (the planner ran both widths as one launch).
        mma_items = plan.get("mma_items").reshape(-1, 3)
        mrows = (mma_items[:, 2] - mma_items[:, 1]) * spec.gqa_group
        mb = (((mrows + 1) // 2 + 15) // 16) - 1
        out = {}
        for r in recs:
            if r["kernel"] == "phase2_merge":
                key, ab = "phase2_merge", p2
            else:
                kk = 1 if r["kernel"] == "phase1_mma" else 0
                key = f'{r["kernel"]}[bucket={r["bucket"]}{",fallback" if r["fallback"] else ""}]'
                b = r["bucket"]
                if kk == 0 and not r["fallback"] and int((fb == b).sum()) != r["items"]:
                    b = -1
                if kk == 1 and int((mb == b).sum()) != r["items"]:
                    b = -1
                ab = alg.get((kk, b, r["fallback"]), {}).get("total", 0)
            k = out.setdefault(key, {"launches": 0, "total_ms": 0.0, "alg_bytes": ab, "items": r["items"]})
            k["launches"] += 1
            k["total_ms"] += r["ms"]
        tot = sum(k["total_ms"] for k in out.values()) or 1.0
        for k in out.values():
            k["avg_us"] = k["total_ms"] / k["launches"] * 1e3
            k["share"] = k["total_ms"] / tot
            k["achieved_gbs"] = k["alg_bytes"] / (k["avg_us"] * 1e-6) / 1e9 if k["avg_us"] else None
        return out

    def unique_kv(self):
        s = self.spec
        return self.plan.stats["unique_tokens"] * 2 * s.num_kv_heads * s.head_dim * 2

    def naive_kv(self):
        s = self.spec
        return self.plan.stats["naive_tokens"] * 2 * s.num_kv_heads * s.head_dim * 2

    def naive_leg(self, n):
        for _ in range(3):
            self.naive_step()
        nms, _, _, _ = self.timed(self.naive_step, n)
        return statistics.mean(nms) * 1e3

    def e2e_leg(self, n):
        """End to end through the public API, as a decode loop runs it: the
        tree planned afresh every step (tree-only, rebuilt into the loop's
        plan so that its device copy and staging buffer are reused), the plan
        uploaded, then one deft_tree_attn_host call (through a HostStep
        bound to the loop's buffers once, as a decode loop holds them): Q
        copied from pinned host memory, the step run, out + lse copied back
        to pinned host memory."""
        torch, deft, spec, t, a = self.torch, self.deft, self.spec, self.t, self.args
        q_host = t.q.cpu().pin_memory()
        out_host = torch.empty(self.bufs.out.shape, dtype=self.bufs.out.dtype).pin_memory()
        lse_host = torch.empty(self.bufs.lse.shape, dtype=self.bufs.lse.dtype).pin_memory()
        q_dev = torch.empty_like(t.q)
        times = []
        p = deft.Plan(spec.parent, spec.node_len, spec.query_node, a.chunk_target, spec.gqa_group,
                      query_pos=spec.query_pos, naive=False, tensor_pack=self.tp)
        step = deft.HostStep(q_host, q_dev, t.k_pages, t.v_pages, self.npo, self.pid, p, self.bufs, out_host,
                             lse_host)
        for i in range(n + 3):
            self.barrier()
            t0 = time.perf_counter()
            p.rebuild(spec.parent, spec.node_len, spec.query_node, a.chunk_target, spec.gqa_group,
                      query_pos=spec.query_pos, naive=False, tensor_pack=self.tp)
            p.upload()
            step()
            torch.cuda.synchronize(self.dev)
            if i >= 3:
                times.append(time.perf_counter() - t0)
        plan_bytes = p.stats["device_bytes"]
        del step, p
        return (statistics.mean(times) * 1e6, int(q_host.numel() * 2 + plan_bytes),
                int(out_host.numel() * out_host.element_size() + lse_host.numel() * 4))

    def graph_leg(self, n):
        """The same step captured once into a CUDA graph and replayed."""
        torch = self.torch
        try:
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream(self.dev)
            side.wait_stream(self.stream)
            with torch.cuda.stream(side):
                self.step()
            self.stream.wait_stream(side)
            torch.cuda.synchronize(self.dev)
            with torch.cuda.graph(g):
                self.step()
            for _ in range(3):
                self.flush_l2()
                g.replay()
            gms, _, _, _ = self.timed(g.replay, n)
            return {"us_per_step": statistics.mean(gms) * 1e3, "us_per_step_median": statistics.median(gms) * 1e3,
                    "steps": n}
        except Exception as e:   # report, do not fail the bench line
            return {"error": str(e).splitlines()[0][:200]}


def roofline_of(kernels, ms_per_step, unique_kv, hbm_peak, peak_kind, cfg):
    """Whole step against the unique-KV roofline, and the dominant kernel's
    own fraction (its event window overlaps the other phase-1 launches, which
    share the SMs with it: an SM-share-limited figure)."""
    dom_name = max(kernels, key=lambda n: kernels[n]["total_ms"]) if kernels else None
    dom = kernels.get(dom_name, {})
    step_gbs = unique_kv / (ms_per_step * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": dom_name, "achieved": dom.get("achieved_gbs"), "peak": hbm_peak,
            "unit": "GB/s", "frac": (dom.get("achieved_gbs") or 0) / hbm_peak,
            "traffic": ncu_traffic(dom_name, cfg) if dom_name else None,
            "peak_source": f"{peak_kind} HBM copy bandwidth",
            "alg_bytes_per_launch": dom.get("alg_bytes"), "avg_launch_us": dom.get("avg_us"),
            "kernel_frac_note": "the dominant launch's algorithmic bytes over its own event window; the "
                                "phase-1 launches run concurrently and share the SMs, so this is an "
                                "SM-share-limited figure, not the chip's",
            "whole_step": {"achieved": step_gbs, "peak": hbm_peak, "unit": "GB/s", "frac": step_gbs / hbm_peak,
                           "bytes": "unique KV bytes per step / step time"}}


def measure_config(deft, torch, dev, cfg, args, hbm_peak, peak_kind, steps, warmup, oracle_budget):
    """The sweep entry of one workload: device time, whole-step roofline,
    dominant kernel, naive form, e2e and the oracle on the host cores."""
    r = Runner(deft, torch, dev, W.config(cfg), args)
    r.warm(warmup)
    ms, _, _, _ = r.timed(r.step, steps)
    _, recs, _, _ = r.timed(r.step, max(3, steps // 4), trace=True)
    kernels = r.kernels(recs, steps)
    med = statistics.median(ms)
    roof = roofline_of(kernels, med, r.unique_kv(), hbm_peak, peak_kind, cfg)
    e2e_us, _, _ = r.e2e_leg(max(3, steps // 4))
    entry = {"workload": r.spec.name, "chunk_target": args.chunk_target, "tensor_pack": r.tp,
             "us_per_step_median": med * 1e3, "us_per_step_p10": float(np.percentile(ms, 10)) * 1e3,
             "us_per_step_p90": float(np.percentile(ms, 90)) * 1e3, "steps": steps,
             "unique_kv_bytes": r.unique_kv(), "frac_of_measured_hbm": roof["whole_step"]["frac"],
             "whole_step_roofline": roof["whole_step"],
             "dominant_kernel": {"name": roof["kernel"], "avg_us": roof["avg_launch_us"],
                                 "frac_sm_share_limited": roof["frac"],
                                 "alg_bytes_per_launch": roof["alg_bytes_per_launch"],
                                 "dram_bytes_per_launch": roof["traffic"]},
             "naive_us_per_step": r.naive_leg(max(3, steps // 2)), "e2e_us_per_step": e2e_us}
    if oracle_budget > 0:
        cb = cpu_baseline(r.spec, r.layout, host_inputs(r.spec, r.layout, r.t), budget_s=oracle_budget,
                          single_thread=False)
        entry["oracle_us_per_step"] = cb["value"]
        entry["oracle_cores"] = cb["cores"]
    del r
    torch.cuda.empty_cache()
    return entry


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.profile_case:
        return run_profile_case(args)

    import torch
    import shared_prefix_kv_deft_gb300 as deft
    deft.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    spec = W.config(args.config)
    shard = head_shard(spec.num_q_heads, spec.num_kv_heads, rank, world) \
        if args.shard == "heads" and world > 1 else None
    run = Runner(deft, torch, dev, spec, args, pg=pg, shard=shard)
    spec = run.spec
    run.warm(args.warmup)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    ms, _, w0, w1 = run.timed(run.step, args.steps)          # timed region: the value
    clocks = sampler.summary(w0, w1)
    sampler.stop()
    _, recs, _, _ = run.timed(run.step, args.steps, trace=True)  # per-kernel durations
    elapsed = max_over_ranks(sum(ms), pg, dev)
    ms_per_step = elapsed / args.steps
    # Replicas: the job finishes `world` steps in the slowest rank's time.
    # Head shards: the ranks share one step, done when the slowest is.
    value_us = job_us_per_step(ms_per_step, world) if shard is None else ms_per_step * 1e3

    st = run.plan.stats
    d, Hq, Hkv, Q = spec.head_dim, spec.num_q_heads, spec.num_kv_heads, spec.num_queries
    hbm_peak, peak_kind = measured_peaks()
    kernels = run.kernels(recs, args.steps)
    per_step = len(recs) // max(1, args.steps)
    roofline = roofline_of(kernels, ms_per_step, run.unique_kv(), hbm_peak, peak_kind, args.config)
    step_gbs = roofline["whole_step"]["achieved"]

    line = {
        "metric": METRIC, "value": value_us, "unit": "us/step", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": False, "scaling": "weak" if shard is None else "strong",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 Q/K/V, random-init; no dataset)",
        "config": {"workload": spec.name, "config_index": args.config, "global_batch": Q * (1 if shard else world),
                   "seq_len": int(max(1, st["naive_tokens"] // max(1, Q))),
                   "parallelism": ("single GPU" if world == 1 else
                                   f"kv-head shards x{world}" if shard else f"replicas x{world}"),
                   "chunk_target": args.chunk_target, "tensor_pack": run.tp,
                   "l2": "flushed between timed steps (2 x L2 memset, then 2 x L2 read: cold, clean)",
                   "q_heads": Hq, "kv_heads": Hkv, "head_dim": d},
        "us_per_step_median": statistics.median(ms) * 1e3,
        "us_per_step_p10": float(np.percentile(ms, 10)) * 1e3,
        "us_per_step_p90": float(np.percentile(ms, 90)) * 1e3,
        "unique_kv_bytes": run.unique_kv(), "naive_kv_bytes": run.naive_kv(),
        "achieved_gbs_vs_unique_kv": step_gbs,
        "frac_of_measured_hbm": step_gbs / hbm_peak, "frac_of_spec_8tbs": step_gbs / SPEC_HBM_GBS,
        "roofline": roofline, "kernels": kernels,
        "gpu_launches": per_step * args.steps,
        "clocks": clocks,
        "plan": {k: st[k] for k in ("num_chunks", "num_segments", "num_slots", "num_fma_items",
                                    "num_mma_items", "num_fallback_items", "max_chunk_tokens",
                                    "num_merge_queries")},
    }

    if not args.no_extras:
        line["cuda_graph"] = run.graph_leg(args.steps)
        nk = max(3, min(args.steps, 200))
        nus = run.naive_leg(nk)
        line["naive"] = {"us_per_step": nus, "steps": nk, "kv_bytes": run.naive_kv(),
                         "speedup_of_tree": nus / (ms_per_step * 1e3)}
        e2e_us, h2d, d2h = run.e2e_leg(max(3, min(args.steps, 200)))
        e2e_us = max_over_ranks(e2e_us, pg, dev)
        line["e2e"] = {"value": job_us_per_step(e2e_us * 1e-3, world) if shard is None else e2e_us,
                       "unit": "us/step", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "includes": "host planning (rebuilt into the loop's plan) + plan upload + one "
                                   "deft_tree_attn_host call (Q H2D, step, out/lse D2H)",
                       "steps": max(3, min(args.steps, 200))}
        if rank == 0 and world == 1:
            line["cpu_baseline"] = cpu_baseline(spec, run.layout, host_inputs(spec, run.layout, run.t))
        del run
        torch.cuda.empty_cache()
        # Every workload, measured in the same process (rank 0 alone).
        if rank == 0 and world == 1 and not args.no_sweep:
            sweep = {}
            for cfg in range(1, 8):
                big = cfg in (5, 6)
                sweep[str(cfg)] = measure_config(deft, torch, dev, cfg, args, hbm_peak, peak_kind,
                                                 steps=min(args.steps, 40 if big else 200),
                                                 warmup=3, oracle_budget=2.0 if big else 3.0)
            line["configs"] = sweep
    if rank == 0:
        print(json.dumps(line))
    if pg is not None:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
