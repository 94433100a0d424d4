"""Decode-attention benchmark over a prefix-shared KV tree (one JSON line).

Metric: decode-attention step time and effective unique-KV bandwidth (unique
K/V bytes of the tree / step time) against the measured HBM peak, on the
7B-shaped shared-prefix workload by default (32 heads, d=128, fp16, batch 32,
1024 shared + 512 private tokens per sequence, chunk 64).  Inputs are seeded
synthetic tensors drawn on the GPU; the pool and tables are resident before
the timed region; L2 is flushed (a 256 MiB write) between timed steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

N > 1 runs one independent replica per GPU (the path has no exchange step),
launched by torchrun; rank 0 prints the line with the max-over-ranks time.
--impl reference times the fp64 CPU oracle on the host cores instead.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn μs/step and unique-KV GB/s vs HBM peak, shared-prefix batch"
UNIT = "GB/s (unique KV)"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="share1k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--min-share", type=int, default=0)
    ap.add_argument("--flags", type=int, default=0)
    ap.add_argument("--loop-steps", type=int, default=128, help="decode-loop steps (0: skip)")
    ap.add_argument("--sweep", choices=["batch", "divergence", "generality"], default=None,
                    help="one line per workload of a family instead of the single default line")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank number over all ranks (identity on one process)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(unique_bytes_per_rank: int, ms_per_step: float, world: int) -> float:
    """Aggregate unique-KV GB/s of `world` replicas that each process one step
    of the workload per `ms_per_step` (the max over ranks)."""
    return world * unique_bytes_per_rank / (ms_per_step * 1e-3) / 1e9


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def step_bytes(spec):
    """Algorithmic bytes of one decode step: unique K/V + q + out."""
    es = {"f16": 2, "bf16": 2, "f32": 4}[spec.dtype]
    qo = 2 * spec.n_sequences * spec.n_q_heads * spec.head_dim * es
    return spec.unique_kv_bytes() + qo


def private_bytes(spec, min_share=2):
    """Algorithmic bytes of the sequence-first kernel: K/V of chunks covered by fewer
    than min_share sequences, plus the q rows it reads."""
    es = {"f16": 2, "bf16": 2, "f32": 4}[spec.dtype]
    tok, mult = 0, 1
    for n, fan in spec.levels:
        mult *= fan
        cover = spec.n_sequences // mult
        if cover < min_share:
            tok += mult * n
    return tok * spec.bytes_per_token() + spec.n_sequences * spec.n_q_heads * spec.head_dim * es


def shared_bytes(spec, min_share=2):
    es = {"f16": 2, "bf16": 2, "f32": 4}[spec.dtype]
    tok, mult = 0, 1
    for n, fan in spec.levels:
        mult *= fan
        cover = spec.n_sequences // mult
        if cover >= min_share:
            tok += mult * n
    return tok * spec.bytes_per_token() + spec.n_sequences * spec.n_q_heads * spec.head_dim * es


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"pst_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        peak_power = max(r[2] for r in rows)
        loaded = [r for r in rows if r[2] >= 0.5 * peak_power] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, x in enumerate(r[3]) if x.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(loaded)}


def source_digest(files) -> str:
    """sha256 (first 16 hex digits) of the listed kernel sources, concatenated."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "prefix_shared_kv_tree_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current source of that kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d[workload][kernel]
        if source_digest(ent["sources"]) != ent["sources_sha256_16"]:
            return None
        return float(ent["bytes_per_launch"])
    except Exception:
        return None


# ------------------------------------------------------------------ oracle leg
def oracle_rate(config: str, budget_s: float, max_rows=None):
    """Time the fp64 oracle (as it stands) on whole sequences of the workload,
    single-threaded BLAS, in a subprocess.  Returns (GB/s unique-KV equivalent,
    rows timed, seconds)."""
    code = f"""
import os, sys, time, json
sys.path.insert(0, {ROOT!r})
import numpy as np, torch
torch.set_num_threads(1)
from prefix_shared_kv_tree_gb300 import workloads as W
from oracle import attention as A
spec = W.SPECS[{config!r}]
wl = W.generate(spec)
q = wl.q.float().double().numpy()
rows = 0; t_total = 0.0; seqs = 0
u = 0
while t_total < {budget_s!r} and (({max_rows!r} is None) or rows < {max_rows!r}):
    k = wl.seq_k(u).float().numpy(); v = wl.seq_v(u).float().numpy()
    t0 = time.perf_counter()
    A.decode_attention([(k, v)], q[u:u+1])
    t_total += time.perf_counter() - t0
    rows += spec.n_q_heads; seqs += 1
    u = (u + 1) % spec.n_sequences
print(json.dumps({{"rows": rows, "seconds": t_total, "seqs": seqs}}))
"""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError("oracle timing failed: " + r.stderr[-2000:])
    res = json.loads(r.stdout.strip().splitlines()[-1])
    from prefix_shared_kv_tree_gb300 import workloads as W
    spec = W.SPECS[config]
    t_row = res["seconds"] / res["rows"]
    step_s = t_row * spec.n_sequences * spec.n_q_heads
    return spec.unique_kv_bytes() / step_s / 1e9, res, step_s


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from prefix_shared_kv_tree_gb300 import workloads as W
    spec = W.SPECS[args.config]
    total_budget = 150.0
    per_step = max(0.05, total_budget / max(1, args.steps + args.warmup))
    gbs, res, step_s = oracle_rate(args.config, per_step * (args.steps + args.warmup))
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 6), "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{spec.name}: {W.DESCRIPTIONS[spec.name]}"},
        "cpu_baseline": {"value": round(gbs, 6), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{res['seqs']} whole sequences x {spec.n_q_heads} heads "
                                   f"({res['seconds']:.1f} s, single-threaded numpy fp64), scaled to a "
                                   f"{spec.n_sequences}-sequence step"},
        "e2e": {"value": round(gbs, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- GPU leg
def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", init_method="env://")
    else:
        torch.cuda.set_device(0)
    dev = torch.cuda.current_device()

    import numpy as np
    from prefix_shared_kv_tree_gb300 import build as B
    B.build_library()
    from prefix_shared_kv_tree_gb300 import pst
    from prefix_shared_kv_tree_gb300 import workloads as W

    spec = W.SPECS[args.config]
    wl = W.generate(spec, device="cuda")
    chunks = 0
    mult = 1
    for n, fan in spec.levels:
        mult *= fan
        chunks += mult * math.ceil(n / spec.chunk_size)
    # spare chunks for the decode loop's appends (a new leaf chunk every c steps)
    spare = 64 + spec.n_sequences * (2 + args.loop_steps // spec.chunk_size)
    pool = pst.Pool(spec.n_q_heads, spec.n_kv_heads, spec.head_dim, spec.chunk_size, chunks + spare, spec.dtype,
                    args.min_share, 0, args.flags, device=dev)
    W.insert_all(pool, wl)
    q = wl.q.contiguous()
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream()
    # L2 flush between steps: write a 256 MiB buffer (evicts everything), then read
    # another 256 MiB so the dirty lines of the write are written back before the
    # timed step instead of during it.
    flush_w = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    flush_r = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")

    class _Flush:
        def fill_(self, x):
            flush_w.fill_(x)
            flush_r.sum()
    flush = _Flush()
    pool.decode_attention(q, out)
    torch.cuda.synchronize()
    assert pool.check_device() == 0

    for _ in range(max(3, args.warmup)):
        flush.fill_(1.0)
        pool.decode_attention(q, out)
    torch.cuda.synchronize()

    clocks = ClockSampler(dev)
    clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    launches = 0
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.fill_(1.0)
        ev[i][0].record(stream)
        pool.decode_attention(q, out)
        ev[i][1].record(stream)
        launches += pool.last_launch_count()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    times = [a.elapsed_time(b) for a, b in ev]
    ms = max_over_ranks(sum(times) / len(times), device="cuda")

    # ---- per-kernel durations (library events on the streams the kernels run on);
    # a separate pass, because events between the kernels can stop them overlapping
    pool.set_profiling(True)
    n_prof = max(3, min(args.steps, 100))
    phase = []
    for i in range(n_prof):
        flush.fill_(1.0)
        pool.decode_attention(q, out)
        phase.append(pool.phase_times())
    pool.set_profiling(False)
    assert pool.check_device() == 0

    # ---- e2e through the host-buffer entry point (H2D q, decode, D2H out, sync)
    q_host = q.cpu().pin_memory()
    out_host = torch.empty_like(q_host).pin_memory()
    e2e_times = []
    for i in range(max(3, args.warmup) + args.steps):
        flush.fill_(1.0)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        pool.decode_attention_host(q_host, out_host)
        t1 = time.perf_counter()
        if i >= max(3, args.warmup):
            e2e_times.append(t1 - t0)
    assert torch.equal(out_host, out.cpu())
    e2e_ms = 1e3 * sum(e2e_times) / len(e2e_times)

    # ---- decode loop: per step one token appended to every sequence, then the
    # decode step replayed from a CUDA graph that the library captures again
    # only after a structural change (a new leaf chunk every c steps).  Wall
    # clock over the whole loop: appends, host table rebuilds and uploads,
    # captures and replays.  Runs last: it grows every sequence.
    loop = None
    if args.loop_steps > 0:
        ids = np.asarray(pool.batch_order(), dtype=np.int64)
        gen = torch.Generator(device="cuda").manual_seed(99)
        k_app = torch.randn(len(ids), spec.n_kv_heads, spec.head_dim, generator=gen, device="cuda").to(q.dtype)
        v_app = torch.randn(len(ids), spec.n_kv_heads, spec.head_dim, generator=gen, device="cuda").to(q.dtype)
        toks = np.full(len(ids), 5, dtype=np.int32)
        out_loop = torch.empty_like(q)
        pool.decode_attention_graph(q, out_loop)  # first capture, outside the timed loop
        torch.cuda.synchronize()
        st0 = pool.stats()
        t0 = time.perf_counter()
        sh = stream.cuda_stream  # raw handle: no per-call stream lookup in the binding
        for _ in range(args.loop_steps):
            pool.append_batch(ids, toks, k_app, v_app, stream=sh)
            pool.decode_attention_graph(q, out_loop, stream=sh)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        st1 = pool.stats()
        assert pool.check_device() == 0
        loop = {"us_per_step": round(1e6 * (t1 - t0) / args.loop_steps, 3), "steps": args.loop_steps,
                "graph_captures": st1["graph_captures"] - st0["graph_captures"],
                "table_rebuilds": st1["rebuild_count"] - st0["rebuild_count"],
                "last_rebuild_us": round(st1["last_rebuild_us"], 1),
                "step": "append_batch (one token per sequence) + pst_decode_attention_graph; wall clock, "
                        "no L2 flush between steps"}

    peak, peak_kind = measured_peak()
    st = pool.stats()
    phase_ms = [sum(p[j] for p in phase) / len(phase) for j in range(3)]
    names = ["chunk_first_tc", "sequence_first_simt", "whole_call"]
    dom = max(range(2), key=lambda j: phase_ms[j])  # the dominant kernel (not the whole call)
    min_share = args.min_share or 2
    dom_bytes = [shared_bytes(spec, min_share), private_bytes(spec, min_share)][dom]
    if phase_ms[0] == 0.0:  # no chunk-first launch: the sequence-first kernel reads every chunk
        dom_bytes = spec.unique_kv_bytes()
    achieved = dom_bytes / (phase_ms[dom] * 1e-3) / 1e9

    if rank != 0:
        return
    unique = spec.unique_kv_bytes()
    value = whole_job_gbs(unique, ms, world)
    es = {"f16": 2, "bf16": 2, "f32": 4}[spec.dtype]
    qbytes = spec.n_sequences * spec.n_q_heads * spec.head_dim * es
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 6), "us_per_step": round(ms * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": spec.dtype,
        "data": "synthetic (seeded N(0,1) Q/K/V drawn on the GPU, seeded token ids)",
        "config": {"workload": f"{spec.name}: {W.DESCRIPTIONS[spec.name]}",
                   "l2": "flushed between timed steps (256 MiB write, then 256 MiB read)",
                   "unique_kv_bytes": unique, "logical_kv_bytes": spec.logical_kv_bytes(),
                   "min_share": min_share, "flags": args.flags,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "frac_of_peak": round(value / world / peak, 4),
        "phase_ms": {names[j]: round(phase_ms[j], 5) for j in range(3)},
        "roofline": {"bound": "hbm", "kernel": names[dom], "achieved": round(achieved, 2), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "algorithmic_bytes_per_launch": dom_bytes,
                     "traffic": traffic_for(names[dom], spec.name)},
        "e2e": {"value": round(unique / (e2e_ms * 1e-3) / 1e9, 3), "unit": UNIT, "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": qbytes, "d2h_bytes_per_step": qbytes},
        "gpu_launches": launches,
        "clocks": clk,
        "pool": {k: st[k] for k in ("used_chunks", "shared_chunks", "phase1_items", "phase2_items", "partial_rows")},
        "decode_loop": loop,
    }
    if not args.no_cpu_baseline:
        gbs, res, step_s = oracle_rate(args.config, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(gbs, 6), "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"{res['seqs']} whole sequences x {spec.n_q_heads} heads "
                                          f"({res['seconds']:.1f} s, single-threaded numpy fp64), scaled to a "
                                          f"{spec.n_sequences}-sequence step ({step_s * 1e3:.0f} ms/step)"}
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_sweep(args):
    """One JSON line per workload of a family (ChunkAttention Knowl 9: batch
    scaling; Knowl 8: divergence; Knowl 10: head dims and chunk sizes), each
    from its own bench run (no CPU
    baseline, no decode loop), plus decode tokens per second (B / step time),
    the unit the pages quote."""
    from prefix_shared_kv_tree_gb300 import workloads as W
    names = {"batch": W.BATCH_FAMILY, "divergence": W.DIVERGENCE_FAMILY,
             "generality": W.GENERALITY_FAMILY}[args.sweep]
    for name in names:
        cmd = [sys.executable, os.path.abspath(__file__), "--config", name, "--steps", str(args.steps),
               "--warmup", str(args.warmup), "--no-cpu-baseline", "--loop-steps", "0",
               "--min-share", str(args.min_share), "--flags", str(args.flags)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        line = next((x for x in r.stdout.splitlines() if x.startswith("{")), None)
        if r.returncode != 0 or line is None:
            print(json.dumps({"config": name, "error": (r.stderr or r.stdout)[-400:]}), flush=True)
            continue
        d = json.loads(line)
        d["sweep"] = args.sweep
        d["decode_tokens_per_s"] = round(W.SPECS[name].n_sequences / (d["ms_per_step"] * 1e-3), 1)
        print(json.dumps(d), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
