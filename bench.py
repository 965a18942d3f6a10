#!/usr/bin/env python3
"""Benchmark of the paged-KV decode hot path on GB300.

One step = one pass of the hot path over one batch: the new token of every
sequence is written into its slot, then paged decode attention runs over the
whole context (pa_decode_append; the context split across CTAs and merged by
log-sum-exp). The scatter alone (pa_reshape_and_cache) is timed as a
component. The default workload is the
Qwen3-8B-shaped layer: 16 sequences x 4,164 tokens, 32 query / 8 KV heads,
head_dim 128, bf16, blocks of 16 scattered over a 38,348-block pool.

Prints ONE JSON line (rank 0). ``value`` is KV GB/s: the bytes of K and V a
decode step must read (valid tokens only) divided by the device time per step,
with inputs resident in HBM. Two batches alternate so that consecutive steps
read disjoint 273 MB sets (L2 is 129 MB). ``e2e`` is the wall-clock rate of
the same steps with every step's inputs copied from pinned host memory and
its output copied back and read on the host: each step is one CUDA graph
captured from the public call, the upload of the next step's inputs and the
download of the previous step's output on a second stream beside its kernels;
the host reads each output two steps later.

``--impl reference`` times the oracle (fp64 CPU) on the host cores instead,
one bounded sample of the workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

HBM_NOMINAL_GBS = 8000.0
GRAPH_STEPS = 20          # steps captured per CUDA graph in the timed loop
E2E_DEPTH = 3             # e2e steps in flight before the host reads a step's output
E2E_MIN_STEPS = 2000      # e2e is timed over at least this many steps (the pipeline's fill and
E2E_MAX_STEPS = 20000     #   drain would dominate a short run), and at most this many
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# workload description
# ---------------------------------------------------------------------------
def build_workload(config: str, rank: int, copies: int, block_size: int = 16, layout: str = "paged"):
    """The workload's batch (``copies`` disjoint batches) and its description.
    ``layout`` "contiguous" gives the same lengths in a contiguous cache of
    one maximum-length reservation per sequence (the unpaged baseline)."""
    if layout == "contiguous":
        nb = per_batch(config)
        if config == "qwen3":
            lens, hq, L = [workloads.QWEN3_TOKENS] * (nb * copies), 32, workloads.QWEN3_TOKENS
        elif config == "long":
            lens, hq, L = [workloads.LONG_TOKENS] * (nb * copies), 64, workloads.LONG_TOKENS
        elif config == "gqa_uniform":
            lens, hq, L = [workloads.GQA_UNIFORM_TOKENS] * (nb * copies), 32, workloads.GQA_UNIFORM_TOKENS
        else:
            lens, hq, L = workloads.gqa_lengths(nb * copies), 32, 4096
        desc = "%s, contiguous cache: %d seqs x %d reserved rows (lengths as the paged workload), Hq %d, Hkv 8, D 128, bf16" % (
            config, nb, L, hq)
        return workloads.contiguous(config, lens, hq, 8, 128, L), desc
    if config == "qwen3":
        return workloads.qwen3(num_seqs=16, copies=copies, block_size=block_size), \
            "qwen3-8b layer: 16 seqs x 4164 tokens, Hq 32, Hkv 8, D 128, bf16, block %d, pool %d blocks" % (
                block_size, workloads.QWEN3_POOL_BLOCKS * 16 // block_size)
    if config == "long":
        return workloads.long_context(block_size=block_size, num_seqs=4, copies=copies), \
            "long context: 4 seqs x 32768 tokens, Hq 64, Hkv 8, D 128, bf16, block %d" % block_size
    if config == "gqa_uniform":
        return workloads.gqa_uniform(num_seqs=64 * copies, num_blocks=20000 * copies * 16 // block_size,
                                     block_size=block_size), \
            "llama gqa, uniform: 64 seqs x 2304 tokens, Hq 32, Hkv 8, D 128, bf16, block %d" % block_size
    if config == "gqa":
        return workloads.gqa(num_seqs=64 * copies, num_blocks=20000 * copies * 16 // block_size,
                             block_size=block_size), \
            "llama gqa: 64 seqs, len U[512,4096], Hq 32, Hkv 8, D 128, bf16, block %d" % block_size
    raise SystemExit(f"unknown config {config}")


def workload_config(desc: str, kv_per_step: int) -> dict:
    """``config`` of the JSON line: what the workload is, the same for both
    arms (how each arm runs it goes elsewhere in the line)."""
    return {"workload": desc,
            "l2": "inputs larger than L2 (129 MB): each step reads %.0f MB of K/V" % (kv_per_step / 1e6)}


def per_batch(config: str) -> int:
    return {"qwen3": 16, "long": 4, "gqa": 64, "gqa_uniform": 64}[config]


def kv_bytes(lens, hkv, d, elem) -> int:
    return int(sum(int(n) for n in lens)) * hkv * d * elem * 2


def decode_alg_bytes(lens, hq, hkv, d, bs, elem) -> int:
    """Algorithmic bytes of one decode launch: K/V of valid tokens, the query,
    the fp32 output, the block-table entries used (none for a contiguous
    cache, ``bs`` None) and the lengths."""
    B = len(lens)
    tbl = 0 if bs is None else sum(workloads.cdiv(int(n), bs) for n in lens) * 4
    return kv_bytes(lens, hkv, d, elem) + B * hq * d * elem + B * hq * d * 4 + tbl + B * 4


def max_over_ranks(values, device):
    """Element-wise maximum of per-rank timings over the process group (a
    barrier-free all-reduce; the only cross-rank traffic of the benchmark)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_gbs(world: int, bytes_per_rank_step: float, ms_per_step: float) -> float:
    """Whole-job throughput: every rank processes its own batch each step
    (weak scaling), and a step lasts as long as the slowest rank's."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


DECODE_SOURCES = ("decode_mma.cu", "device_common.cuh", "mma_tile.cuh")
BALANCED_SOURCES = ("decode_balanced.cu", "device_common.cuh", "mma_tile.cuh")


def decode_source_sha(files=DECODE_SOURCES) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "paged_kv_cache_121_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(config: str, files=DECODE_SOURCES):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"pa_decode_{config}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_tr or m_sha.group(1) != decode_source_sha(files):
        return None
    return float(m_tr.group(1))


# ---------------------------------------------------------------------------
# clocks sampled by nvidia-smi during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
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
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, line in self.lines:
            if not (t0 <= t <= t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id_for_smi(torch, local_rank: int) -> str:
    """Identifier nvidia-smi -i accepts for the GPU this process uses."""
    try:
        u = str(torch.cuda.get_device_properties(local_rank).uuid)
        if u and u != "None":
            return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [x for x in vis.split(",") if x.strip()]
    return ids[local_rank].strip() if local_rank < len(ids) else str(local_rank)


# ---------------------------------------------------------------------------
# oracle timing (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------
def oracle_units_time(batch, seqs, nthreads):
    import oracle
    q = batch.query[seqs]
    tables = batch.block_tables[seqs]
    lens = batch.context_lens[seqs]
    t = time.perf_counter()
    oracle.paged_attention(q, batch.k_cache, batch.v_cache, tables, lens, batch.scale,
                           nthreads=nthreads)
    return time.perf_counter() - t


def cpu_baseline(batch, nseq_batch, budget_s=10.0):
    """The oracle as it stands, on the host cores, over whole decode steps of
    the workload (all sequences of one batch) repeated for ~budget_s."""
    nthreads = os.cpu_count() or 1
    seqs = np.arange(nseq_batch)
    lens = batch.context_lens[seqs]
    elapsed, reps = 0.0, 0
    while elapsed < budget_s or reps == 0:
        elapsed += oracle_units_time(batch, seqs, nthreads)
        reps += 1
        if reps >= 1000:
            break
    kvb = kv_bytes(lens, batch.num_kv_heads, batch.head_dim, batch.elem_bytes) * reps
    # the same oracle on one thread, over a smaller sample (a quarter of the batch, twice)
    one = seqs[: max(1, nseq_batch // 4)]
    t1 = sum(oracle_units_time(batch, one, 1) for _ in range(2))
    kv1 = kv_bytes(batch.context_lens[one], batch.num_kv_heads, batch.head_dim, batch.elem_bytes) * 2
    return {"value": kvb / elapsed / 1e9, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
            "sample": f"{reps} full decode step(s) of the workload ({nseq_batch} sequences, fp64 C, "
                      f"OpenMP over (sequence, KV head)), {elapsed:.1f} s",
            "tokens_per_s": nseq_batch * reps / elapsed,
            "single_thread": {"value": kv1 / t1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": f"{len(one)} sequence(s) x 2, {t1:.1f} s"}}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    if args.config in ("cow", "swap"):
        print(json.dumps({"impl": "reference", "unavailable": "the oracle arm times the paged decode "
                          "workloads (qwen3, long, gqa)"}), flush=True)
        return 0
    batch, desc = build_workload(args.config, 0, 1, args.block_size)
    nb = per_batch(args.config)
    nthreads = os.cpu_count() or 1
    # size each step's sample (whole sequences) so the K + W steps fit ~120 s
    t1 = oracle_units_time(batch, np.arange(1), nthreads)
    budget = 120.0 / max(1, args.steps + args.warmup)
    per_step = int(max(1, min(nb, budget // max(t1, 1e-6))))
    order = np.arange(nb)
    for i in range(args.warmup):
        oracle_units_time(batch, order[(i * per_step + np.arange(per_step)) % nb], nthreads)
    total, kvb, seqs_done = 0.0, 0, 0
    for i in range(args.steps):
        seqs = order[(i * per_step + np.arange(per_step)) % nb]
        total += oracle_units_time(batch, seqs, nthreads)
        kvb += kv_bytes(batch.context_lens[seqs], batch.num_kv_heads, batch.head_dim, batch.elem_bytes)
        seqs_done += len(seqs)
    value = kvb / total / 1e9
    line = {
        "metric": ("paged decode attention KV GB/s (Qwen3-8B shape)" if args.config == "qwen3"
                   else "paged decode attention KV GB/s (%s workload)" % args.config),
        "value": value, "unit": "GB/s", "impl": "reference", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1), bf16-rounded)",
        "config": workload_config(desc, kv_bytes(batch.context_lens, batch.num_kv_heads, batch.head_dim,
                                                 batch.elem_bytes)),
        "sample": {"seqs_per_step": per_step, "of": nb},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
                         "sample": f"{per_step} sequence(s) of the batch per step"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "tokens_per_s": seqs_done / total,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# the CUDA arm
# ---------------------------------------------------------------------------
def long_context_line(torch, pa, stream, reps: int, peak: float, peak_kind: str) -> dict:
    """The long-context workload (4 x 32,768 tokens, Hq 64, Hkv 8, D 128, bf16,
    blocks of 16) timed as the headline is: GRAPH_STEPS launches per CUDA
    graph, two disjoint batches alternating, CUDA events on the launching
    stream. The decode alone (pa_decode) gives the roofline fraction; the
    whole step (pa_decode_append: the new tokens written, then the decode)
    is timed the same way."""
    copies = 2
    batch, desc = build_workload("long", 0, copies)
    nb = per_batch("long")
    hq, hkv, d, bs = batch.num_heads, batch.num_kv_heads, batch.head_dim, batch.block_size

    def dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    k_cache, v_cache = dev(batch.k_cache), dev(batch.v_cache)
    views = []
    for c in range(copies):
        sl = slice(c * nb, (c + 1) * nb)
        lens = batch.context_lens[sl]
        views.append({"query": dev(batch.query[sl]), "tables": dev(batch.block_tables[sl]), "lens": dev(lens),
                      "key": dev(batch.new_key[sl]), "value": dev(batch.new_value[sl]),
                      "max_len": int(lens.max()), "lens_h": lens,
                      "out": torch.empty((nb, hq, d), dtype=torch.float32, device="cuda")})
    ws_bytes = max(pa.pa_decode_workspace_size(nb, hq, hkv, d, bs, v["max_len"]) for v in views)
    workspace = torch.zeros(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    plan = pa.pa_decode_plan(nb, hq, hkv, d, bs, max(v["max_len"] for v in views), with_workspace=True)

    def decode(i):
        v = views[i % copies]
        pa.pa_decode(v["out"], v["query"], k_cache, v_cache, v["tables"], v["lens"], v["max_len"], batch.scale,
                     workspace=workspace)

    def step(i):
        v = views[i % copies]
        pa.pa_decode_append(v["out"], v["query"], v["key"], v["value"], k_cache, v_cache, v["tables"], v["lens"],
                            v["max_len"], batch.scale, workspace=workspace)

    def graph_of(fn):
        with torch.cuda.stream(stream):
            for i in range(3):
                fn(i)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for i in range(GRAPH_STEPS):
                fn(i)
        return g

    def per_launch_ms(g):
        with torch.cuda.stream(stream):
            g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / (reps * GRAPH_STEPS)

    decode_ms = per_launch_ms(graph_of(decode))
    step_ms = per_launch_ms(graph_of(step))
    if pa.pa_device_status() != 0:
        raise SystemExit("device status not clean after the long-context loops")
    alg = np.mean([decode_alg_bytes(v["lens_h"], hq, hkv, d, bs, batch.elem_bytes) for v in views])
    kvb = np.mean([kv_bytes(v["lens_h"], hkv, d, batch.elem_bytes) for v in views])
    achieved = alg / (decode_ms * 1e-3) / 1e9
    return {"workload": desc, "plan": plan, "decode_us": decode_ms * 1e3, "alg_bytes_per_launch": int(alg),
            "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
            "pct_of_8tbs": 100.0 * achieved / HBM_NOMINAL_GBS,
            "step_us": step_ms * 1e3, "step_kv_gbs": kvb / (step_ms * 1e-3) / 1e9,
            "launches": reps * GRAPH_STEPS * 2}


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import paged_kv_cache_121_gb300 as pa

    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    pa.load_library()

    copies = 2
    contig = args.layout == "contiguous"
    batch, desc = build_workload(args.config, rank, copies, args.block_size, args.layout)
    nb = per_batch(args.config)
    hq, hkv, d = batch.num_heads, batch.num_kv_heads, batch.head_dim
    bs = None if contig else batch.block_size
    elem = batch.elem_bytes
    headline = not contig and bs == 16

    def dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    if contig:
        # [B, L, Hkv, D]; the scatter sees it as a pool of one-token blocks
        L = batch.max_seq_len
        k_full, v_full = dev(batch.k), dev(batch.v)
        k_cache = k_full.view(batch.num_seqs * L, 1, hkv, d)
        v_cache = v_full.view(batch.num_seqs * L, 1, hkv, d)
        slots_all = np.arange(batch.num_seqs, dtype=np.int64) * L + batch.new_pos
    else:
        k_cache, v_cache = dev(batch.k_cache), dev(batch.v_cache)
        seq_all = np.arange(batch.num_seqs, dtype=np.int32)
        slots_all = pa.pa_compute_slot_mapping(batch.block_tables, seq_all, batch.new_pos, bs)
    views = []
    for c in range(copies):
        sl = slice(c * nb, (c + 1) * nb)
        lens = batch.context_lens[sl]
        views.append({
            "query": dev(batch.query[sl]),
            "tables": None if contig else dev(batch.block_tables[sl]),
            "k": k_full[sl] if contig else None, "v": v_full[sl] if contig else None,
            "lens": dev(lens), "key": dev(batch.new_key[sl]), "value": dev(batch.new_value[sl]),
            "slots": torch.from_numpy(slots_all[sl].copy()).cuda(),
            "max_len": int(lens.max()), "lens_h": lens,
            "out": torch.empty((nb, hq, d), dtype=torch.float32, device="cuda"),
        })
    ws_bytes = max(pa.pa_decode_workspace_size(nb, hq, hkv, d, 16 if contig else bs, v["max_len"])
                   for v in views)
    workspace = torch.zeros(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    plan = pa.pa_decode_plan(nb, hq, hkv, d, 16 if contig else bs, max(v["max_len"] for v in views),
                             with_workspace=True)

    def scatter(v):
        pa.pa_reshape_and_cache(v["key"], v["value"], k_cache, v_cache, v["slots"])

    def decode_into(out, v, query, lens, tables, stream=None):
        if contig:
            pa.pa_decode_contiguous(out, query, v["k"], v["v"], lens, v["max_len"], batch.scale,
                                    workspace=workspace, stream=stream)
        else:
            pa.pa_decode(out, query, k_cache, v_cache, tables, lens, v["max_len"], batch.scale,
                         workspace=workspace, stream=stream)

    def decode(v):
        decode_into(v["out"], v, v["query"], v["lens"], v["tables"])

    def step(i):
        v = views[i % copies]
        if contig:
            scatter(v)
            decode(v)
        else:   # one call: the new tokens written (by the decode kernel itself where it can), then the decode
            pa.pa_decode_append(v["out"], v["query"], v["key"], v["value"], k_cache, v_cache, v["tables"],
                                v["lens"], v["max_len"], batch.scale, workspace=workspace)

    for i in range(copies):
        step(i)
    torch.cuda.synchronize()
    if pa.pa_device_status() != 0:
        raise SystemExit("device status not clean after warm-up")
    if args.profile_steps:
        # a few eager steps and nothing else: the command ncu captures
        for i in range(args.profile_steps):
            step(i)
        torch.cuda.synchronize()
        print(json.dumps({"profile_steps": args.profile_steps, "config": desc,
                          "workspace_bytes": int(ws_bytes)}), flush=True)
        return 0

    # CUDA graphs: one graph per batch view, each holding one whole step
    stream = torch.cuda.Stream()
    step_graphs, decode_graphs = [], []
    with torch.cuda.stream(stream):
        for i in range(3):
            step(i)
        torch.cuda.synchronize()
        for c in range(copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                step(c)
            step_graphs.append(g)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                decode(views[c])
            decode_graphs.append(g)
        # GRAPH_STEPS consecutive steps (batches alternating) in one graph, as a
        # serving engine captures a whole forward pass; and the same for decode alone
        multi_step = torch.cuda.CUDAGraph()
        with torch.cuda.graph(multi_step, stream=stream, capture_error_mode="thread_local"):
            for i in range(GRAPH_STEPS):
                step(i)
        multi_decode = torch.cuda.CUDAGraph()
        with torch.cuda.graph(multi_decode, stream=stream, capture_error_mode="thread_local"):
            for i in range(GRAPH_STEPS):
                decode(views[i % copies])
    torch.cuda.synchronize()

    K, W = args.steps, args.warmup
    with torch.cuda.stream(stream):
        for i in range(W):
            step_graphs[i % copies].replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(gpu_id_for_smi(torch, local_rank))
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        # one more untimed graph of steps first, not waited for: the GPU is busy
        # with it while the timed graphs are submitted, so the start event is
        # followed at once by the K timed steps (no graph-launch latency inside
        # the window); the batches keep alternating across the boundary
        multi_step.replay()
        ev0.record(stream)
        for _ in range(K // GRAPH_STEPS):
            multi_step.replay()
        for i in range(K - K % GRAPH_STEPS, K):
            step_graphs[i % copies].replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.perf_counter()
    if world > 1:
        dist.barrier()
    ms_total = ev0.elapsed_time(ev1)
    steps_timed = K

    # the dominant kernel alone: decode-only graph replays, CUDA events on its stream
    dreps = max(5, min(K, 20000) // GRAPH_STEPS)
    with torch.cuda.stream(stream):
        multi_decode.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(dreps):
            multi_decode.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    decode_ms = e0.elapsed_time(e1) / (dreps * GRAPH_STEPS)
    scatter_ms, _ = time_graph(torch, stream, lambda i: scatter(views[i % copies]), dreps)

    # e2e through the public API, host buffers (pinned), copies inside the timed
    # region. Every step copies its inputs (query, new K/V, lengths, slots,
    # tables: one packed pinned buffer, one transfer) to the device, runs the
    # step's public call (pa_decode_append; for the contiguous layout the
    # scatter and pa_decode_contiguous), and copies the output back to pinned
    # host memory, where the host reads it. Each step is one CUDA graph
    # captured from those calls, as a serving engine captures its decode
    # step: on the step's stream the kernels of step i, and beside them, on a
    # second stream forked and joined inside the graph, the upload of step
    # i + 1's inputs and the download of step i - 1's output. E2E_DEPTH buffer
    # sets rotate; the host replays step i's graph, then waits for step i - 1's
    # graph and reads step i - 2's output (which that graph downloaded).
    def pack(arrays):
        offs, pos = [], 0
        for a in arrays:
            offs.append(pos)
            pos += (a.nbytes + 255) // 256 * 256
        buf = np.zeros(pos, np.uint8)
        for a, o in zip(arrays, offs):
            buf[o:o + a.nbytes] = np.ascontiguousarray(a).view(np.uint8).reshape(-1)
        return torch.from_numpy(buf).pin_memory(), offs

    def host_arrays(c):
        sl = slice(c * nb, (c + 1) * nb)
        arrs = [batch.query[sl], batch.new_key[sl], batch.new_value[sl], batch.context_lens[sl],
                slots_all[sl].astype(np.int64)]
        if not contig:
            arrs.append(batch.block_tables[sl])
        return arrs

    staged = [pack(host_arrays(c)) for c in range(copies)]
    h2d = staged[0][0].numel()
    kv_t = k_cache.dtype
    arr0 = host_arrays(0)
    offs0 = staged[0][1]
    s_e2e, s_copy = torch.cuda.Stream(), torch.cuda.Stream()

    def slot_buffers():
        stage = torch.empty(h2d, dtype=torch.uint8, device="cuda")

        def view(i, dtype, shape):
            o = offs0[i]
            n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
            return stage[o:o + n].view(dtype).view(shape)

        return {"stage": stage, "q": view(0, kv_t, arr0[0].shape), "k": view(1, kv_t, arr0[1].shape),
                "v": view(2, kv_t, arr0[2].shape), "lens": view(3, torch.int32, arr0[3].shape),
                "slots": view(4, torch.int64, arr0[4].shape),
                "tables": None if contig else view(5, torch.int32, arr0[5].shape),
                "out": torch.empty((nb, hq, d), dtype=torch.float32, device="cuda"),
                "h_out": torch.empty((nb, hq, d), dtype=torch.float32).pin_memory(),
                "done": torch.cuda.Event()}

    slots_e2e = [slot_buffers() for _ in range(E2E_DEPTH)]
    d2h = slots_e2e[0]["h_out"].numel() * 4
    period = E2E_DEPTH * copies // math.gcd(E2E_DEPTH, copies)   # graphs differ by (slot, batch)

    def step_kernels(sb, c):
        if contig:
            pa.pa_reshape_and_cache(sb["k"], sb["v"], k_cache, v_cache, sb["slots"])
            decode_into(sb["out"], views[c], sb["q"], sb["lens"], sb["tables"])
        else:
            pa.pa_decode_append(sb["out"], sb["q"], sb["k"], sb["v"], k_cache, v_cache, sb["tables"],
                                sb["lens"], views[c]["max_len"], batch.scale, workspace=workspace)

    def e2e_body(i):   # captured: step i's kernels, beside them step i + 1's upload and step i - 1's download
        cur, nxt, prv = (slots_e2e[(i + x) % E2E_DEPTH] for x in (0, 1, E2E_DEPTH - 1))
        fork, join = torch.cuda.Event(), torch.cuda.Event()
        fork.record(s_e2e)
        s_copy.wait_event(fork)
        with torch.cuda.stream(s_copy):
            nxt["stage"].copy_(staged[(i + 1) % copies][0], non_blocking=True)
            prv["h_out"].copy_(prv["out"], non_blocking=True)
            join.record(s_copy)
        step_kernels(cur, i % copies)
        s_e2e.wait_event(join)

    # warm-up outside any capture, then one graph per (slot, batch) pattern
    with torch.cuda.stream(s_e2e):
        for c in range(copies):
            slots_e2e[c % E2E_DEPTH]["stage"].copy_(staged[c][0])
        for i in range(period):
            e2e_body(i)
    torch.cuda.synchronize()
    e2e_graphs = []
    for i in range(period):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s_e2e, capture_error_mode="thread_local"):
            e2e_body(i)
        e2e_graphs.append(g)
    checksum = [0.0]

    def e2e_run(first, n):
        """Steps first .. first + n - 1; reads the outputs of steps first - 1 .. first + n - 2."""
        with torch.cuda.stream(s_e2e):
            for i in range(first, first + n):
                e2e_graphs[i % period].replay()
                slots_e2e[i % E2E_DEPTH]["done"].record(s_e2e)
                if i >= 1:
                    slots_e2e[(i - 1) % E2E_DEPTH]["done"].synchronize()
                    checksum[0] += float(slots_e2e[(i - 2) % E2E_DEPTH]["h_out"][0, 0, 0])   # step i - 2's result

    # prime the pipeline: the inputs of the first timed step are uploaded by the graph before it
    with torch.cuda.stream(s_e2e):
        slots_e2e[0]["stage"].copy_(staged[0][0])
    e2e_run(0, 2 * period)
    e2e_steps = min(max(K, E2E_MIN_STEPS), E2E_MAX_STEPS)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    e2e_run(2 * period, e2e_steps)
    e2e_s = time.perf_counter() - t0
    torch.cuda.synchronize()
    if pa.pa_device_status() != 0:
        raise SystemExit("device status not clean after the timed region")
    if not np.isfinite(checksum[0]):
        raise SystemExit("non-finite decode output in the e2e loop")
    peak, peak_kind = measured_peaks()
    # the second workload the roofline target names: long contexts, decode timed the same way
    long_ctx = (long_context_line(torch, pa, stream, dreps, peak, peak_kind)
                if headline and args.config == "qwen3" else None)
    t_end = time.perf_counter()
    time.sleep(0.15)
    sampler.stop()
    # clocks over every timed loop of the run (the K steps, the decode-only
    # loops and e2e); the K steps alone may be shorter than one sample
    clocks = sampler.summary(t_wall0 - 0.05, t_end + 0.05)
    clocks["timed_steps_samples"] = sampler.summary(t_wall0 - 0.05, t_wall1 + 0.05)["samples"]
    clocks["window"] = "timed steps, decode-only loops and e2e"

    # max over ranks
    ms_step = ms_total / steps_timed
    e2e_ms_step = e2e_s * 1e3 / e2e_steps
    if world > 1:
        ms_step, e2e_ms_step, decode_ms = max_over_ranks([ms_step, e2e_ms_step, decode_ms], "cuda")
        if long_ctx is not None:
            long_ctx["decode_us"], long_ctx["step_us"] = max_over_ranks(
                [long_ctx["decode_us"], long_ctx["step_us"]], "cuda")
            long_ctx["achieved"] = long_ctx["alg_bytes_per_launch"] / (long_ctx["decode_us"] * 1e-6) / 1e9
            long_ctx["frac"] = long_ctx["achieved"] / peak

    lens0 = views[0]["lens_h"]
    step_kv = kv_bytes(lens0, hkv, d, elem)          # per batch; both batches have equal totals for qwen3/long
    avg_kv = np.mean([kv_bytes(v["lens_h"], hkv, d, elem) for v in views])
    value = whole_job_gbs(world, avg_kv, ms_step)
    e2e_value = whole_job_gbs(world, avg_kv, e2e_ms_step)
    alg = np.mean([decode_alg_bytes(v["lens_h"], hq, hkv, d, bs, elem) for v in views])
    achieved = alg / (decode_ms * 1e-3) / 1e9
    traffic = profiled_traffic(args.config, BALANCED_SOURCES if plan.get("balanced") else DECODE_SOURCES) \
        if headline else None
    if not plan["tensor_cores"]:
        kernel = "decode_simt_kernel"
    elif contig:
        kernel = "decode_mma_kernel<128,16> (contiguous)"
    elif bs == 8:
        kernel = "decode_mma_kernel<128,16> (two blocks per tile)"
    elif bs < 8:
        kernel = "decode_mma_kernel<128,16> (one bulk copy per token row, %d blocks per tile)" % (16 // bs)
    elif plan.get("balanced"):
        kernel = "decode_balanced_kernel<128> (equal tile ranges per CTA) + balanced_merge_kernel<128>"
    else:
        kernel = "decode_mma_kernel<128,16>"
    decode_launches = plan["kernel_launches"]       # a wide split adds the merge kernel
    # the tensor-core kernels write the step's new tokens themselves; the CUDA-core one scatters first
    step_launches = decode_launches + (1 if contig or not plan["tensor_cores"] else 0)
    line = {
        "metric": ("decode attention KV GB/s, contiguous cache (unpaged baseline)" if contig
                   else "paged decode attention KV GB/s (Qwen3-8B shape)" if args.config == "qwen3"
                   else "paged decode attention KV GB/s (%s workload)" % args.config),
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": steps_timed, "warmup": W,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16",
        "data": ("synthetic (seeded N(0,1), bf16-rounded; one contiguous reservation per sequence)" if contig else
                 "synthetic (seeded N(0,1), bf16-rounded; block placement a seeded random permutation)"),
        "config": workload_config(desc, step_kv),
        "setup": {"graphs": "%d steps per CUDA graph" % GRAPH_STEPS,
                  "batches": "%d disjoint batches of the workload alternate, so consecutive steps read "
                             "disjoint memory" % copies,
                  "plan": plan,
                  "step": ("reshape_and_cache(%d tokens) + pa_decode_contiguous" % nb if contig else
                           "pa_decode_append: %d new tokens into their slots, then the decode" % nb)},
        "tokens_per_s": world * nb / (ms_step * 1e-3),
        "pct_of_8tbs": 100.0 * value / HBM_NOMINAL_GBS,
        "pct_of_measured_hbm": 100.0 * value / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": kernel, "peak_kind": peak_kind,
                     "decode_us": decode_ms * 1e3, "alg_bytes_per_launch": int(alg)},
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms_step, "steps": e2e_steps},
        "gpu_launches": step_launches * steps_timed,
        "components": {"reshape_and_cache_us": scatter_ms * 1e3,
                       "reshape_and_cache_gbs": nb * hkv * d * elem * 2 * 2 / (scatter_ms * 1e-3) / 1e9,
                       "reshape_and_cache_tokens": nb},
        "tokens_per_s_36_layers_attention_only": world * nb / (36 * ms_step * 1e-3),
    }
    if long_ctx is not None:
        line["long_context"] = long_ctx
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not contig:
        line["cpu_baseline"] = cpu_baseline(batch, nb, budget_s=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------
# copy-on-write workload: 64 sequences forked from one prefix
# ---------------------------------------------------------------------------
COW_COPIES = 6      # disjoint copies of the workload (6 x ~42 MB unique > L2)


def build_cow_state(torch, pa, copies: int, prefix_len: int):
    """The copy-on-write workload built through the library: per copy, one
    sequence is prefilled with the shared prefix, forked to 63 more, every
    sequence appends its suffix through the block manager (copy-on-write of
    the half-filled shared block by copy_blocks), and the decode token's slot
    is allocated. Returns the device caches and, per copy, the step's inputs."""
    case = workloads.shared_prefix(prefix_len=prefix_len)
    S, bs, hkv, d = len(case.suffix_lens), case.block_size, case.num_kv_heads, case.head_dim
    nblocks = case.num_blocks * copies
    k_cache = torch.zeros((nblocks, bs, hkv, d), dtype=torch.bfloat16, device="cuda")
    v_cache = torch.zeros_like(k_cache)
    bm = pa.BlockManager(nblocks, bs)

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)

    views, pairs_all = [], []
    for c in range(copies):
        base = c * S
        bm.allocate(base, prefix_len)
        slots = pa.pa_compute_slot_mapping(np.array([bm.block_table(base)], np.int32),
                                           np.zeros(prefix_len, np.int32), np.arange(prefix_len, dtype=np.int32), bs)
        pa.pa_reshape_and_cache(dev(case.prefix_key), dev(case.prefix_value), k_cache, v_cache,
                                torch.from_numpy(slots).cuda())
        for s_ in range(1, S):
            bm.fork(base, base + s_)
        pairs, slots, keys, vals, dec_slots = [], [], [], [], []
        for s_ in range(S):
            n = case.suffix_key[s_].shape[0]
            for t in range(n):
                slot, src, dst = bm.append_slot(base + s_)
                if src >= 0:
                    pairs.append((src, dst))
                if t < n - 1:
                    slots.append(slot)
                else:
                    dec_slots.append(slot)      # the decode token: written inside the timed step
            keys.append(case.suffix_key[s_][:-1])
            vals.append(case.suffix_value[s_][:-1])
        if pairs:
            pa.pa_copy_blocks(k_cache, v_cache, torch.from_numpy(np.array(pairs, np.int64)).cuda())
        if slots:
            pa.pa_reshape_and_cache(dev(np.concatenate(keys)), dev(np.concatenate(vals)), k_cache, v_cache,
                                    torch.from_numpy(np.array(slots, np.int64)).cuda())
        lens = np.array([bm.num_tokens(base + s_) for s_ in range(S)], np.int32)
        maxb = max(len(bm.block_table(base + s_)) for s_ in range(S))
        tables = np.zeros((S, maxb), np.int32)
        for s_ in range(S):
            t = bm.block_table(base + s_)
            tables[s_, :len(t)] = t
        dk = np.stack([case.suffix_key[s_][-1] for s_ in range(S)])
        dv = np.stack([case.suffix_value[s_][-1] for s_ in range(S)])
        views.append({"query": dev(case.query), "tables": torch.from_numpy(tables).cuda(),
                      "lens": torch.from_numpy(lens).cuda(), "lens_h": lens, "key": dev(dk), "value": dev(dv),
                      "slots": torch.from_numpy(np.array(dec_slots, np.int64)).cuda(),
                      "max_len": int(lens.max()), "shared": prefix_len // bs,
                      "out": torch.empty((S, case.num_heads, d), dtype=torch.float32, device="cuda"),
                      "host": {"query": case.query, "tables": tables, "lens": lens, "key": dk, "value": dv,
                               "slots": np.array(dec_slots, np.int64)}})
        pairs_all.append(np.array(pairs, np.int64).reshape(-1, 2))
    torch.cuda.synchronize()
    return case, k_cache, v_cache, views, pairs_all, bm.stats()


def time_graph(torch, stream, fn, reps: int):
    """Device time of one call of fn: a CUDA graph of GRAPH_STEPS calls
    replayed reps times, CUDA events on the graph's stream."""
    with torch.cuda.stream(stream):
        for i in range(3):
            fn(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        for i in range(GRAPH_STEPS):
            fn(i)
    with torch.cuda.stream(stream):
        g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (reps * GRAPH_STEPS), g


def run_cow(args, rank, world, local_rank):
    """Copy-on-write workload (64 sequences sharing a 2,064-token prefix in
    blocks of 32, suffixes U[0, 256]): a step scatters each sequence's decode
    token and runs one decode, plain (pa_decode: every sequence reads the
    prefix through its own table) or prefix-aware (pa_decode_shared_prefix:
    the 64 shared blocks read once)."""
    import torch
    import torch.distributed as dist

    import paged_kv_cache_121_gb300 as pa

    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    pa.load_library()
    prefix_len = 2064
    copies = args.copies or COW_COPIES
    case, k_cache, v_cache, views, pairs_all, stats = build_cow_state(torch, pa, copies, prefix_len)
    S, hq, hkv, d, bs = len(case.suffix_lens), case.num_heads, case.num_kv_heads, case.head_dim, case.block_size
    shared = prefix_len // bs
    aware = args.prefix_aware
    mcl = max(v["max_len"] for v in views)
    if aware:
        ws_bytes = pa.pa_decode_shared_prefix_workspace_size(S, hq, hkv, d, bs, mcl, shared)
    else:
        ws_bytes = pa.pa_decode_workspace_size(S, hq, hkv, d, bs, mcl)
    workspace = torch.zeros(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")

    def decode_into(out, v, query, lens, tables):
        if aware:
            pa.pa_decode_shared_prefix(out, query, k_cache, v_cache, tables, lens, v["max_len"], v["shared"],
                                       case.scale, workspace)
        else:
            pa.pa_decode(out, query, k_cache, v_cache, tables, lens, v["max_len"], case.scale,
                         workspace=workspace)

    def step(i):
        v = views[i % copies]
        pa.pa_reshape_and_cache(v["key"], v["value"], k_cache, v_cache, v["slots"])
        decode_into(v["out"], v, v["query"], v["lens"], v["tables"])

    def decode(i):
        v = views[i % copies]
        decode_into(v["out"], v, v["query"], v["lens"], v["tables"])

    # copy_blocks of one copy's copy-on-write pairs, into spare blocks (the
    # same bytes as the real copies, without undoing the suffixes written since)
    npairs = int(pairs_all[0].shape[0])
    scratch_pairs = pairs_all[0].copy()
    scratch_pairs[:, 1] = np.arange(k_cache.shape[0] - npairs, k_cache.shape[0])
    scratch_pairs_d = torch.from_numpy(scratch_pairs).cuda()

    stream = torch.cuda.Stream()
    K, W = args.steps, args.warmup
    with torch.cuda.stream(stream):
        for i in range(W):
            step(i)
    torch.cuda.synchronize()
    if pa.pa_device_status() != 0:
        raise SystemExit("device status not clean after warm-up")
    if args.profile_steps:
        for i in range(args.profile_steps):
            step(i)
        torch.cuda.synchronize()
        print(json.dumps({"profile_steps": args.profile_steps, "config": "cow", "prefix_aware": aware}), flush=True)
        return 0
    reps = max(5, K // GRAPH_STEPS)
    sampler = ClockSampler(gpu_id_for_smi(torch, local_rank))
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    t_wall0 = time.perf_counter()
    step_ms, _ = time_graph(torch, stream, step, reps)
    t_wall1 = time.perf_counter()
    time.sleep(0.15)
    sampler.stop()
    clocks = sampler.summary(t_wall0 - 0.05, t_wall1 + 0.05)
    decode_ms, _ = time_graph(torch, stream, decode, reps)
    scatter_ms, _ = time_graph(torch, stream, lambda i: pa.pa_reshape_and_cache(
        views[i % copies]["key"], views[i % copies]["value"], k_cache, v_cache, views[i % copies]["slots"]), reps)
    copy_ms, _ = time_graph(torch, stream, lambda i: pa.pa_copy_blocks(k_cache, v_cache, scratch_pairs_d), reps)
    if pa.pa_device_status() != 0:
        raise SystemExit("device status not clean after the timed region")

    # e2e through the public API: host inputs in, output out, every step
    h_in = []
    for v in views:
        h = v["host"]
        h_in.append({k: torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16 else
                                         np.ascontiguousarray(a)).pin_memory() for k, a in h.items()})
        h_in[-1]["out"] = torch.empty((S, hq, d), dtype=torch.float32).pin_memory()
    dq = torch.empty((S, hq, d), dtype=torch.bfloat16, device="cuda")
    dk = torch.empty((S, hkv, d), dtype=torch.bfloat16, device="cuda")
    dvv = torch.empty_like(dk)
    dl = torch.empty((S,), dtype=torch.int32, device="cuda")
    ds = torch.empty((S,), dtype=torch.int64, device="cuda")
    dts = [torch.empty_like(v["tables"]) for v in views]
    dout = torch.empty((S, hq, d), dtype=torch.float32, device="cuda")

    def e2e_step(i):
        h, v, dt = h_in[i % copies], views[i % copies], dts[i % copies]
        dq.view(torch.int16).copy_(h["query"], non_blocking=True)
        dk.view(torch.int16).copy_(h["key"], non_blocking=True)
        dvv.view(torch.int16).copy_(h["value"], non_blocking=True)
        dt.copy_(h["tables"], non_blocking=True)
        dl.copy_(h["lens"], non_blocking=True)
        ds.copy_(h["slots"], non_blocking=True)
        pa.pa_reshape_and_cache(dk, dvv, k_cache, v_cache, ds)
        decode_into(dout, v, dq, dl, dt)
        h["out"].copy_(dout, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        return float(h["out"][0, 0, 0])

    for i in range(3):
        e2e_step(i)
    e2e_steps = min(max(K, E2E_MIN_STEPS), E2E_MAX_STEPS)
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    e2e_ms = (time.perf_counter() - t0) * 1e3 / e2e_steps
    h2d = sum(h_in[0][k].numel() * h_in[0][k].element_size() for k in ("query", "tables", "lens", "key", "value", "slots"))
    d2h = S * hq * d * 4
    if world > 1:
        step_ms, decode_ms, e2e_ms = max_over_ranks([step_ms, decode_ms, e2e_ms], "cuda")

    lens0 = views[0]["lens_h"]
    logical = kv_bytes(lens0, hkv, d, 2)                                  # every sequence's whole context
    private_blocks = sum(workloads.cdiv(int(n), bs) - shared for n in lens0)
    unique = (shared + private_blocks) * bs * hkv * d * 2 * 2              # each block once
    alg = unique + S * hq * d * 2 + S * hq * d * 4 + tables_bytes(lens0, bs) + S * 4
    peak, peak_kind = measured_peaks()
    value = whole_job_gbs(world, logical, step_ms)
    line = {
        "metric": "decode attention KV GB/s, copy-on-write shared-prefix workload (logical bytes)",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": reps * GRAPH_STEPS, "warmup": W,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1), bf16-rounded; blocks placed by the block manager)",
        "config": {"workload": "cow: 64 seqs sharing a %d-token prefix, suffix U[0,256] + 1 decode token, "
                               "Hq 32, Hkv 8, D 128, bf16, block 32" % prefix_len,
                   "decode": "pa_decode_shared_prefix (%d shared blocks read once)" % shared if aware
                   else "pa_decode (each sequence reads the prefix through its table)",
                   "graphs": "%d steps per CUDA graph, %d copies of the workload alternate" % (GRAPH_STEPS, copies),
                   "l2": "inputs larger than L2: %d copies x %.0f MB unique" % (copies, unique / 1e6),
                   "cow_pairs_per_copy": npairs},
        "unique_kv_gbs": whole_job_gbs(world, unique, step_ms),
        "tokens_per_s": world * S / (step_ms * 1e-3),
        "roofline": {"bound": "hbm", "achieved": alg / (decode_ms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": alg / (decode_ms * 1e-3) / 1e9 / peak, "traffic": None,
                     "kernel": "prefix pass + decode + merge" if aware else "decode_mma_kernel<128,16>",
                     "peak_kind": peak_kind, "decode_us": decode_ms * 1e3, "alg_bytes_per_launch": int(alg),
                     "alg_bytes": "unique K/V bytes (each block once) + q + out + table + lengths"},
        "components": {
            "reshape_and_cache_us": scatter_ms * 1e3,
            "reshape_and_cache_gbs": S * hkv * d * 2 * 2 * 2 / (scatter_ms * 1e-3) / 1e9,
            "copy_blocks_us": copy_ms * 1e3,
            "copy_blocks_pairs": npairs,
            "copy_blocks_gbs": npairs * bs * hkv * d * 2 * 2 * 2 / (copy_ms * 1e-3) / 1e9,
        },
        "clocks": clocks,
        "e2e": {"value": whole_job_gbs(world, logical, e2e_ms), "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms, "steps": e2e_steps},
        "gpu_launches": (1 + (3 if aware else pa.pa_decode_plan(S, hq, hkv, d, bs, mcl)["kernel_launches"]))
                        * reps * GRAPH_STEPS,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_swap(args, rank, world, local_rank):
    """Swap of the Qwen3-8B layer's KV (16 sequences x 4,164 tokens, 261
    blocks of 16 each) to a page-locked CPU pool and back: one pa_swap_blocks
    launch per direction, against one copy call per block and cache (the
    many small transfers the pages describe), captured in a CUDA graph."""
    import torch
    import torch.distributed as dist

    import paged_kv_cache_121_gb300 as pa

    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    pa.load_library()
    batch = workloads.qwen3(num_seqs=16, copies=1)
    hkv, d, bs = batch.num_kv_heads, batch.head_dim, batch.block_size
    kd = torch.from_numpy(batch.k_cache.view(np.int16)).cuda().view(torch.bfloat16)
    vd = torch.from_numpy(batch.v_cache.view(np.int16)).cuda().view(torch.bfloat16)
    used = [batch.block_tables[i, :workloads.cdiv(int(n), bs)] for i, n in enumerate(batch.context_lens)]
    nblk = int(sum(len(u) for u in used))
    # the batch's placement: device block -> CPU block pairs, CPU ids 0..nblk-1
    out_pairs = np.stack([np.concatenate(used).astype(np.int64), np.arange(nblk, dtype=np.int64)], 1)
    in_pairs = out_pairs[:, ::-1].copy()
    hk = torch.empty((nblk, bs, hkv, d), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    po, pi = torch.from_numpy(out_pairs).cuda(), torch.from_numpy(in_pairs).cuda()
    moved = nblk * bs * hkv * d * 2 * 2                       # K and V bytes, one direction
    stream = torch.cuda.Stream()
    reps = max(3, args.steps // GRAPH_STEPS)

    def kernel_step(i):
        pa.pa_swap_blocks(hk, hv, kd, vd, po)
        pa.pa_swap_blocks(kd, vd, hk, hv, pi)

    def per_block_step(i):
        for g, h in out_pairs[:, :2].tolist():
            hk[h].copy_(kd[g], non_blocking=True)
            hv[h].copy_(vd[g], non_blocking=True)
        for g, h in out_pairs[:, :2].tolist():
            kd[g].copy_(hk[h], non_blocking=True)
            vd[g].copy_(hv[h], non_blocking=True)

    sampler = ClockSampler(gpu_id_for_smi(torch, local_rank))
    sampler.start()
    time.sleep(0.3)
    t0 = time.perf_counter()
    k_ms, _ = time_graph(torch, stream, kernel_step, reps)
    t1 = time.perf_counter()
    time.sleep(0.15)
    sampler.stop()
    clocks = sampler.summary(t0 - 0.05, t1 + 0.05)
    b_ms = time_graph_once(torch, stream, per_block_step, max(3, reps // 20))
    # the link's ceiling for the same bytes: one bulk copy per cache and direction
    kd_flat, vd_flat = kd[:nblk], vd[:nblk]

    def bulk_step(i):
        hk.copy_(kd_flat, non_blocking=True)
        hv.copy_(vd_flat, non_blocking=True)
        kd_flat.copy_(hk, non_blocking=True)
        vd_flat.copy_(hv, non_blocking=True)

    c_ms = time_graph_once(torch, stream, bulk_step, max(3, reps // 4))
    ok = torch.equal(kd.view(torch.int16).cpu(), torch.from_numpy(batch.k_cache.view(np.int16)))
    if world > 1:
        k_ms, b_ms, c_ms = max_over_ranks([k_ms, b_ms, c_ms], "cuda")
    line = {
        "metric": "KV swap GB/s (GPU -> page-locked CPU pool -> GPU, Qwen3-8B layer)",
        "value": whole_job_gbs(world, 2 * moved, k_ms), "unit": "GB/s", "n_gpus": world,
        "steps": reps * GRAPH_STEPS, "warmup": 3, "ms_per_step": k_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1), bf16-rounded)",
        "config": {"workload": "swap: 16 seqs x 4164 tokens, %d blocks of 16 (Hkv 8, D 128), out and back" % nblk,
                   "bytes_each_way": moved, "l2": "inputs larger than L2 (%.0f MB each way)" % (moved / 1e6)},
        "per_block_copies": {"ms_per_step": b_ms, "gbs": 2 * moved / (b_ms * 1e-3) / 1e9,
                             "calls_per_step": 4 * nblk},
        "bulk_copies": {"ms_per_step": c_ms, "gbs": 2 * moved / (c_ms * 1e-3) / 1e9, "calls_per_step": 4,
                        "note": "contiguous blocks copied in bulk: the link's ceiling, not a block swap"},
        "restored_bit_exact": bool(ok),
        "clocks": clocks,
        "gpu_launches": 2 * reps * GRAPH_STEPS,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def time_graph_once(torch, stream, fn, reps: int):
    """Device time of one call of fn captured alone in a CUDA graph."""
    with torch.cuda.stream(stream):
        fn(0)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        fn(0)
    with torch.cuda.stream(stream):
        g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def tables_bytes(lens, bs) -> int:
    return sum(workloads.cdiv(int(n), bs) for n in lens) * 4


def spawn_ranks(nproc: int) -> int:
    """``--gpus N`` run directly (not under a launcher): start this script on N
    local ranks, one process per GPU, through torch.distributed.run with the
    rendezvous on 127.0.0.1 and the same arguments; its exit status is the
    launcher's. Each rank times its own batch (weak scaling); rank 0 prints."""
    import socket
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=%d" % nproc,
           "--master-addr=127.0.0.1", "--master-port=%d" % port, os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=["qwen3", "long", "gqa", "gqa_uniform", "cow", "swap"], default="qwen3")
    ap.add_argument("--copies", type=int, default=0,
                    help="cow: disjoint copies of the workload held on the device (default %d)" % COW_COPIES)
    ap.add_argument("--prefix-aware", action="store_true",
                    help="cow: decode with pa_decode_shared_prefix (the shared blocks read once)")
    ap.add_argument("--layout", choices=["paged", "contiguous"], default="paged",
                    help="contiguous: the same lengths in one reservation per sequence, no block table")
    ap.add_argument("--block-size", type=int, default=16, choices=[1, 2, 4, 8, 16, 32, 64, 128],
                    help="tokens per block of the paged cache (the pool keeps its token count)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="run this many eager steps after the warm-up and exit (for ncu)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return spawn_ranks(args.gpus)
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.config == "cow":
        return run_cow(args, rank, world, local_rank)
    if args.config == "swap":
        return run_swap(args, rank, world, local_rank)
    return run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    sys.exit(main())
