"""Benchmark: GQA split-KV decode on GB300.

One step = one decode call over the workload (contiguous: ``gqa_decode``, the
split-KV partial pass with the in-kernel merge; paged: ``gqa_decode_paged``),
inputs resident in HBM.  The headline workload is the long-context single
sequence (S_kv = 2^20, h_q = 32, h_kv = 8, d_head = 128, ~4 GiB of f16 K+V).

Printed (rank 0, one JSON line): KV-cache read GB/s over the whole job
(bytes = K + V + Q + O per step, plus block tables and lengths when paged),
microseconds per step, the roofline of the kernel against the measured HBM
copy bandwidth, the same metric end to end from pinned host buffers, and the
CPU float64 oracle timed on the host cores as a reported baseline.

``--impl reference`` times the oracle instead (host cores, bounded samples of
the same workload, same metric).  Multi-GPU runs (torchrun) are independent
replicas: every rank runs the whole workload on its own GPU, nothing is
exchanged; ``value`` sums the ranks' bytes over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gqa_inputs as gi  # noqa: E402

METRIC = "KV-cache read GB/s (fraction of GB300 HBM peak); µs per decode step"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(gi.WORKLOADS), default="long")
    ap.add_argument("--s-kv", type=int, default=0,
                    help="contiguous workloads: override S_kv (smaller cases for profiler captures)")
    ap.add_argument("--elem", choices=["f16", "bf16"], default="f16",
                    help="element type of Q, K, V and O (the same draws, rounded to bfloat16 for bf16)")
    ap.add_argument("--block-size", type=int, default=0,
                    help="paged workload: override the KV block size")
    ap.add_argument("--head-group", type=int, default=0,
                    help="paged workload: KV heads per work item (1, 2, 4; 0 = library default)")
    ap.add_argument("--partition-size", type=int, default=-1,
                    help="paged workloads: override the partition size (0 = automatic v1 / v2)")
    ap.add_argument("--n-splits", type=int, default=0)
    ap.add_argument("--merge-mode", type=int, default=0)
    ap.add_argument("--mma-path", type=int, default=0,
                    help="contiguous workloads: 0 automatic, 1 mma.sync split kernel, 2 tcgen05 kernel")
    ap.add_argument("--shard", choices=["none", "skv"], default="none",
                    help="contiguous workloads under torchrun: 'skv' splits every sequence's keys over the "
                         "ranks (sharded_decode: a partial per rank, one all-gather, the merge); the job's "
                         "bytes are counted once (strong scaling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float) -> float:
    """Max of a per-rank float over all ranks (identity without a process group)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_step: int, steps: int, world: int, t_max_ms: float) -> float:
    """Whole-job GB/s: every rank processed steps x bytes_per_step; the slowest rank's time counts."""
    return bytes_per_step * steps * world / (t_max_ms * 1e-3) / 1e9


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# device-code files that define each timed kernel (its template instantiations, the shared
# kernel helpers and the PTX wrappers); a traffic record is valid while these are unchanged
KERNEL_SOURCES = {
    "gqa_split_kernel": ["gqa_kernels.cuh", "gqa_instances.cuh", "ptx.cuh", "gqa_contig_*.cu", "gqa_cluster_*.cu"],
    "gqa_paged_kernel": ["gqa_kernels.cuh", "gqa_instances.cuh", "ptx.cuh", "gqa_paged_*.cu"],
    "gqa_tc_kernel": ["gqa_kernels.cuh", "gqa_tc.cuh", "ptx.cuh", "gqa_tc_*.cu"],
}


def _code_only(text: str) -> str:
    """Source without comments and blank-line / trailing-space differences: a comment edit does not
    change the kernel the counters were taken on."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash(kernel: str, root: str = ROOT) -> str:
    h = hashlib.sha256()
    files = set()
    for pat in KERNEL_SOURCES[kernel]:
        files.update(glob.glob(os.path.join(root, "decode_attention_03_gb300", "csrc", pat)))
    for p in sorted(files):
        with open(p, encoding="utf-8") as f:
            h.update(os.path.basename(p).encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current source of
    the kernel that dominates the step."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("kernel") == kernel and e.get("source_hash") == kernel_source_hash(kernel):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        time.sleep(0.15)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        inside = [p for (t, p) in self.samples if t0 - 0.15 <= t <= t1 + 0.15]
        use = inside if inside else [p for (_, p) in self.samples]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(p[1]) for p in use if p[1].replace(".", "").isdigit()]
        mx = [float(p[2]) for p in use if p[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for p in use:
            for i, n in enumerate(names):
                if p[5 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(use), "in_window": bool(inside)}


# ---------------------------------------------------------------------------------------------
def load_inputs(name: str, s_kv: int = 0, block_size: int = 0, partition_size: int = -1, elem: str = "f16"):
    import dataclasses
    w = gi.WORKLOADS[name]
    if elem != w.elem:
        w = dataclasses.replace(w, name=f"{w.name}[{elem}]", elem=elem)
    if partition_size >= 0 and w.kind == "paged" and partition_size != w.partition_size:
        w = dataclasses.replace(w, name=f"{w.name}[partition={partition_size}]", partition_size=int(partition_size))
    if s_kv and w.kind == "contiguous" and s_kv != w.S_kv:
        w = dataclasses.replace(w, name=f"{w.name}[S_kv={s_kv}]", S_kv=int(s_kv))
    if block_size and w.kind == "paged" and block_size != w.block_size:
        w = dataclasses.replace(w, name=f"{w.name}[block={block_size}]", block_size=int(block_size))
    x = gi.make(w)
    return w, x


def host_tensor(a: np.ndarray) -> torch.Tensor:
    """A CPU tensor of an input array: bfloat16 bit patterns (uint16) become torch.bfloat16."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(a)


def to_device(x: dict, dev):
    keys = ("q", "k", "v") if "k" in x else ("q", "k_pool", "v_pool", "block_tables", "seq_lens")
    return {k: host_tensor(x[k]).to(dev) for k in keys}


def make_step(pkg, w, x, d, out, ws, args):
    if w.kind == "contiguous" and args.shard == "skv":
        from decode_attention_03_gb300.sharded import sharded_decode

        def step():
            sharded_decode(d["q"], d["k"], d["v"], w.h_q, w.h_kv, w.scale, out=out)
        return step
    if w.kind == "contiguous":
        def step():
            pkg.gqa_decode(d["q"], d["k"], d["v"], w.h_q, w.h_kv, w.scale, out=out, workspace_tensor=ws,
                           n_splits=args.n_splits, merge_mode=args.merge_mode, mma_path=args.mma_path)
    else:
        q2 = d["q"].reshape(w.batch, -1)
        fn = pkg.gqa_decode_paged_vllm if w.layout == "vllm" else pkg.gqa_decode_paged

        def step():
            fn(q2, d["k_pool"], d["v_pool"], d["block_tables"], d["seq_lens"], w.h_q, w.h_kv,
               w.scale, max_seq_len=x["max_seq_len"], partition_size=w.partition_size,
               out=out, workspace_tensor=ws, head_group=args.head_group)
    return step


def oracle_sample(x, w, target_s: float, threads: int = 0):
    """Time the CPU oracle on a bounded sample of the workload (all host cores, or ``threads``);
    returns (bytes/s, desc, threads)."""
    import oracle
    threads = threads or os.cpu_count() or 1
    prev = torch.get_num_threads()
    torch.set_num_threads(threads)
    try:
        return _oracle_sample(oracle, x, w, target_s, threads)
    finally:
        torch.set_num_threads(prev)


def _oracle_sample(oracle, x, w, target_s: float, threads: int):
    def vals(a):   # exact values of the inputs (bfloat16 bit patterns decoded)
        return a if w.elem == "f16" else gi.values(a, w.elem)

    if w.kind == "contiguous":
        S = x["k"].shape[1]
        s_len = min(S, 4096)
        units = [(0, 0)]

        def run(n):
            oracle.decode(vals(x["q"][:1]), vals(x["k"][:1, :n]), vals(x["v"][:1, :n]), w.h_q, w.h_kv, w.d_head,
                          w.scale, units=units)

        def nbytes(n):
            return 2 * n * w.d_head * 2 + 2 * w.T_q * w.G * w.d_head * 2
        # grow the sample until one pass takes ~target_s / 4
        t = 0.0
        while True:
            t0 = time.perf_counter()
            run(s_len)
            t = time.perf_counter() - t0
            if t > target_s / 4 or s_len >= S:
                break
            s_len = min(S, s_len * 4)
        reps, t_tot = 0, 0.0
        while t_tot < target_s or reps == 0:
            t0 = time.perf_counter()
            run(s_len)
            t_tot += time.perf_counter() - t0
            reps += 1
        desc = f"sequence 0, KV head 0 ({w.G * w.T_q} query rows) over the first {s_len} keys, {reps} passes"
        return reps * nbytes(s_len) / t_tot, desc, threads
    else:
        lens = x["seq_lens"]
        q, kp, vp = vals(x["q"]), vals(x["k_pool"]), vals(x["v_pool"])
        seqs = []
        total, t_tot, reps = 0, 0.0, 0
        row = w.h_kv * w.d_head * 2
        order = list(range(len(lens)))
        i = 0
        while t_tot < target_s or reps == 0:
            b = order[i % len(order)]
            t0 = time.perf_counter()
            oracle.decode_paged_seq(q, kp, vp, x["block_tables"], lens, b, w.h_q, w.h_kv, w.d_head, w.scale,
                                    w.block_size, w.layout)
            t_tot += time.perf_counter() - t0
            total += 2 * int(lens[b]) * row + 2 * w.h_q * w.d_head * 2
            reps += 1
            i += 1
            seqs.append(b)
        desc = f"{reps} whole sequences of the paged workload ({sorted(set(seqs))[:8]}...)"
        return total / t_tot, desc, threads


def run_reference(args, rank, world):
    """The oracle as the reference arm: host cores, bounded samples, the same metric."""
    if rank != 0:
        return 0
    w, x = load_inputs(args.workload, args.s_kv, args.block_size, args.partition_size, args.elem)
    steps = args.steps if args.steps is not None else 5
    warm = args.warmup if args.warmup is not None else 1
    per_step = max(0.2, min(10.0, 150.0 / max(1, steps + warm)))
    for _ in range(warm):
        oracle_sample(x, w, per_step * 0.25)
    vals, descs, t_total = [], [], 0.0
    for _ in range(steps):
        t0 = time.perf_counter()
        bps, desc, threads = oracle_sample(x, w, per_step)
        t_total += time.perf_counter() - t0
        vals.append(bps)
        descs.append(desc)
    gbs = statistics.median(vals) / 1e9
    bytes_step = gi.kv_bytes(x)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": warm, "ms_per_step": round(bytes_step / (gbs * 1e9) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, x, None, note="CPU float64 oracle on bounded samples of this workload"),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": descs[0]},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(w, x, n_splits, note=None, shard_world=None):
    c = {"workload": w.name, "kind": w.kind, "batch": w.batch, "T_q": w.T_q, "h_q": w.h_q, "h_kv": w.h_kv,
         "d_head": w.d_head, "scale": w.scale, "parallelism": "replicas (no exchange)"}
    if shard_world is not None:
        c["parallelism"] = f"S_kv sharded over {shard_world} rank(s): one partial each, all-gather, merge"
    if w.kind == "contiguous":
        c["S_kv"] = w.S_kv
    else:
        c.update(block_size=w.block_size, partition_size=w.partition_size,
                 tokens=int(np.asarray(x["seq_lens"], dtype=np.int64).sum()), max_seq_len=int(x["max_seq_len"]))
    if n_splits is not None:
        c["n_splits"] = n_splits
    c["bytes_per_step"] = gi.kv_bytes(x)
    if note:
        c["note"] = note
    return c


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from decode_attention_03_gb300 import build as _b
    _b.build()
    import decode_attention_03_gb300 as pkg

    w, x = load_inputs(args.workload, args.s_kv, args.block_size, args.partition_size, args.elem)
    bytes_step = gi.kv_bytes(x)
    shard = None
    if args.shard == "skv":
        if w.kind != "contiguous" or w.elem != "f16":
            raise SystemExit("--shard skv takes a contiguous float16 workload")
        from decode_attention_03_gb300.sharded import shard_range
        shard = shard_range(w.S_kv, rank, world)          # this rank's keys of every sequence
        b0, n = shard
        x = dict(x, k=np.ascontiguousarray(x["k"][:, b0:b0 + n]), v=np.ascontiguousarray(x["v"][:, b0:b0 + n]))
        args.no_e2e = True
    d = to_device(x, dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    big = bytes_step > 2 * l2
    variant = {}     # which kernel variant and fold a contiguous step runs (gqa_decode_plan_ex)
    stream = torch.cuda.Stream(dev)
    out = torch.empty(w.batch * w.T_q * w.h_q * w.d_head, dtype=torch.bfloat16 if w.elem == "bf16" else torch.float16,
                      device=dev)
    out = out.reshape(w.batch, w.T_q, -1) if w.kind == "contiguous" else out.reshape(w.batch, -1)
    if w.kind == "contiguous" and shard is not None:
        nbytes = 256
        n_splits, mma_path, contig_launches = pkg.gqa_decode_plan(
            w.batch, w.T_q, max(shard[1], 1), w.h_q, w.h_kv, w.d_head)
        contig_launches += 1                              # the merge of the ranks' partials
    elif w.kind == "contiguous":
        nbytes = pkg.gqa_decode_workspace_size(w.batch, w.T_q, w.S_kv, w.h_q, w.h_kv, w.d_head, args.n_splits)
        plan = pkg.gqa_decode_plan(w.batch, w.T_q, w.S_kv, w.h_q, w.h_kv, w.d_head, n_splits=args.n_splits,
                                   merge_mode=args.merge_mode, mma_path=args.mma_path, detail=True)
        n_splits, mma_path, contig_launches = plan["n_splits"], plan["mma_path"], plan["launches"]
        variant = {"kernel_variant": plan["kernel"], "fold": plan["fold"]}
    else:
        nbytes = pkg.gqa_paged_workspace_size(w.batch, w.h_q, w.h_kv, w.d_head, x["max_seq_len"], w.partition_size)
        n_splits, mma_path, contig_launches = None, 0, 0
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    step = make_step(pkg, w, x, d, out, ws, args)
    flush = None if big else torch.empty(int(2 * l2), dtype=torch.uint8, device=dev)

    # default step counts: about two seconds of timed work
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(5):
            step()
    torch.cuda.synchronize()
    est = (time.perf_counter() - t0) / 5
    steps = args.steps if args.steps is not None else int(min(5000, max(20, 2.0 / max(est, 1e-6))))
    warm = args.warmup if args.warmup is not None else 10

    with torch.cuda.stream(stream):
        for _ in range(warm):
            if flush is not None:
                flush.zero_()
            step()
    torch.cuda.synchronize()
    if pkg.gqa_workspace_check(ws, stream) != 0:
        raise RuntimeError("device status word set during warm-up")

    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)] \
        if flush is not None else None
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    with torch.cuda.stream(stream):
        if flush is None:
            e0.record(stream)
            for _ in range(steps):
                step()
            e1.record(stream)
        else:
            for i in range(steps):
                flush.zero_()
                ev[i][0].record(stream)
                step()
                ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    clocks.stop()
    if flush is None:
        t_ms = e0.elapsed_time(e1)
    else:
        t_ms = sum(a.elapsed_time(b) for a, b in ev)
    status = pkg.gqa_workspace_check(ws, stream)
    if status != 0:
        raise RuntimeError(f"device status word set in the timed region: {status}")
    l2_hot = None
    if flush is not None:
        # small workloads also report back-to-back steps with the inputs resident in L2,
        # replayed from a CUDA graph so that host submission does not pace the GPU
        n_graph = 50
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                for _ in range(n_graph):
                    step()
            graph.replay()
            torch.cuda.synchronize()
            h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = max(1, steps // n_graph)
            h0.record(stream)
            for _ in range(reps):
                graph.replay()
            h1.record(stream)
        torch.cuda.synchronize()
        hot_ms = h0.elapsed_time(h1) / (reps * n_graph)
        l2_hot = {"us_per_step": round(hot_ms * 1e3, 3), "GB/s": round(bytes_step / (hot_ms * 1e-3) / 1e9, 2),
                  "how": f"CUDA graph of {n_graph} back-to-back steps, inputs L2-resident"}
    t_max = max_over_ranks(t_ms)
    ms_step = t_max / steps
    # replicas: every rank moved the workload's bytes; key shards: the ranks moved them once between them
    value = job_throughput(bytes_step, steps, 1 if shard is not None else world, t_max)
    rank_bytes = bytes_step / world if shard is not None else bytes_step     # what one GPU moved per step
    per_launch_gbs = rank_bytes / (ms_step * 1e-3) / 1e9
    peak, peak_src = measured_peak()

    # ---- end to end: pinned host inputs -> device, decode, output -> host, every step
    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(pkg, w, x, d, out, ws, stream, args, steps_hint=steps)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        bps, desc, threads = oracle_sample(x, w, 10.0)
        cpu = {"value": round(bps / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": desc}
        if w.name == "tiny":   # the launch-bound case: the oracle on one core as well
            bps1, desc1, _ = oracle_sample(x, w, 3.0, threads=1)
            cpu["one_core"] = {"value": round(bps1 / 1e9, 4), "cores": 1, "sample": desc1}

    if rank == 0:
        if w.kind == "paged":   # partition pass, plus the merge pass when a sequence spans partitions
            part, hg, launches_per_step = pkg.gqa_paged_plan(w.batch, w.h_q, w.h_kv, w.d_head, int(x["max_seq_len"]),
                                                             w.partition_size, block_size=w.block_size,
                                                             vllm_layout=w.layout == "vllm",
                                                             head_group=args.head_group)
            kernel = "gqa_paged_kernel"
        else:
            launches_per_step = contig_launches
            kernel = "gqa_tc_kernel" if mma_path == 2 else "gqa_split_kernel"
        traffic = recorded_traffic(w.name, kernel)
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": steps,
            "warmup": warm, "ms_per_step": round(ms_step, 6), "us_per_step": round(ms_step * 1e3, 3),
            "higher_is_better": True, "scaling": "strong" if shard is not None else "weak", "vs_baseline": None,
            "dtype": w.elem, "data": "synthetic",
            "config": dict(config_of(w, x, n_splits, shard_world=world if shard is not None else None), **variant,
                           accum="f32",
                           l2=("inputs larger than L2, no flush" if flush is None
                               else f"L2 flushed ({2 * l2 >> 20} MiB write) before every timed step, outside events")),
            "roofline": {"bound": "hbm", "achieved": round(per_launch_gbs, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(per_launch_gbs / peak, 4), "traffic": traffic,
                         "peak_source": peak_src, "kernel": kernel,
                         "frac_of_nominal_7900": round(per_launch_gbs / NOMINAL_HBM_GBS, 4)},
            "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": steps * launches_per_step, "l2_hot": l2_hot,
            "clocks": clocks.summary(wall0, wall1),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def end_to_end(pkg, w, x, d, out, ws, stream, args, steps_hint):
    keys = list(d.keys())
    host = {k: host_tensor(x[k]).pin_memory() for k in keys}
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = host_out.numel() * host_out.element_size()
    step = make_step(pkg, w, x, d, out, ws, args)

    def one():
        for k in keys:
            d[k].copy_(host[k], non_blocking=True)
        step()
        host_out.copy_(out, non_blocking=True)

    with torch.cuda.stream(stream):
        one()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        one()
    torch.cuda.synchronize()
    est = time.perf_counter() - t0
    n = int(min(max(3, 2.0 / max(est, 1e-6)), max(3, steps_hint)))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n):
            one()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    return {"value": round(gi.kv_bytes(x) / (ms * 1e-3) / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4), "steps": n}


if __name__ == "__main__":
    sys.exit(main())
