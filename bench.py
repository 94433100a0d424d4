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
FALLBACK_BF16_TFLOPS = 1900.0
NOMINAL_HBM_GBS = 8000.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="share1k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the other workloads' step times")
    ap.add_argument("--no-prefill", action="store_true", help="skip the chunked-prefill measurement")
    ap.add_argument("--prefill-only", action="store_true",
                    help="print only the chunked-prefill measurement (the GQA tree's 1137-row prompt)")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
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


def _es(spec) -> int:
    return {"f16": 2, "bf16": 2, "f32": 4}[spec.dtype]


def qo_bytes(spec) -> int:
    """Bytes of the step's query rows (the output rows are as many)."""
    return spec.n_sequences * spec.n_q_heads * spec.head_dim * _es(spec)


def step_bytes(spec):
    """Algorithmic bytes of one decode step: unique K/V + q + out."""
    return spec.unique_kv_bytes() + 2 * qo_bytes(spec)


def decode_flops(spec) -> int:
    """Method FLOPs of one decode step: per (query row, key) 2d for q.k and 2d
    for p.v (ChunkAttention, Knowl 9 counts decode attention this way)."""
    return 4 * spec.head_dim * spec.n_q_heads * spec.n_sequences * spec.seq_len


def plain_decode_intensity(spec) -> float:
    """FLOPs per byte of decode attention without sharing (every sequence
    reads its whole K/V): Knowl 9's ~0.99 FLOP/B at one query row per KV head."""
    return decode_flops(spec) / (spec.logical_kv_bytes() + 2 * qo_bytes(spec))


def prefill_flops(p0: int, w: int, n_q_heads: int, head_dim: int) -> int:
    """Method FLOPs of a causal W-row block at positions [p0, p0 + W): row t
    attends to p0 + t + 1 keys, 4d FLOPs per (query head, key)."""
    keys = w * (p0 + 1) + w * (w - 1) // 2
    return 4 * head_dim * n_q_heads * keys


def private_bytes(spec, min_share=2):
    """Algorithmic bytes of the sequence-first kernel: K/V of chunks covered by fewer
    than min_share sequences, plus the q rows it reads."""
    tok, mult = 0, 1
    for n, fan in spec.levels:
        mult *= fan
        cover = spec.n_sequences // mult
        if cover < min_share:
            tok += mult * n
    return tok * spec.bytes_per_token() + qo_bytes(spec)


def shared_bytes(spec, min_share=2):
    tok, mult = 0, 1
    for n, fan in spec.levels:
        mult *= fan
        cover = spec.n_sequences // mult
        if cover >= min_share:
            tok += mult * n
    return tok * spec.bytes_per_token() + qo_bytes(spec)


def measured_peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, kind) from MEASURED_PEAKS.json, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def distribution(times_ms):
    """mean, median, p10, p90 of per-step times, in microseconds."""
    xs = sorted(times_ms)
    n = len(xs)

    def pct(f):
        return xs[min(n - 1, max(0, int(round(f * (n - 1)))))]
    return {"mean": round(1e3 * sum(xs) / n, 3), "median": round(1e3 * statistics.median(xs), 3),
            "p10": round(1e3 * pct(0.10), 3), "p90": round(1e3 * pct(0.90), 3), "n": n}


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


def strip_comments(src: str) -> str:
    """C/C++/CUDA source without its comments and with runs of whitespace
    collapsed, so that a digest of it changes with the code only."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":  # string or character literal: copied as is
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
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_digest(files) -> str:
    """sha256 (first 16 hex digits) of the listed kernel sources, concatenated,
    comments and whitespace left out: a summary's DRAM counters stay valid for
    as long as the code they were taken on is unchanged."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "prefix_shared_kv_tree_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(strip_comments(fh.read()).encode())
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
_ORACLE_WORKER = r"""
import json, os, sys, time
sys.path.insert(0, ROOT_DIR)
import numpy as np, torch
torch.set_num_threads(1)
from prefix_shared_kv_tree_gb300 import workloads as W
from oracle import attention as A
spec = W.SPECS[CONFIG]
wl = W.generate(spec)
segs = [(s.k.float().numpy(), s.v.float().numpy()) for s in wl.segments]
q = wl.q.float().double().numpy()
sys.stdout.write("ready\n"); sys.stdout.flush()
sys.stdin.readline()   # every worker has its inputs: start together
rows = 0; seqs = 0; u = WORKER
t0 = time.perf_counter()
while time.perf_counter() - t0 < BUDGET:
    k = np.concatenate([segs[i][0] for i in wl.seq_paths[u]])
    v = np.concatenate([segs[i][1] for i in wl.seq_paths[u]])
    A.decode_attention([(k, v)], q[u:u + 1])
    rows += spec.n_q_heads; seqs += 1
    u = (u + NWORKERS) % spec.n_sequences
print(json.dumps({"rows": rows, "seqs": seqs, "seconds": time.perf_counter() - t0}))
"""


def oracle_decode_rate(config: str, budget_s: float, workers: int):
    """Time the fp64 oracle (as it stands) on whole sequences of the workload:
    `workers` processes of one thread each (single-threaded BLAS), started
    together once each has drawn its inputs, each running for budget_s on its
    own sequences.  Returns (rows per second over all workers, detail)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    procs = []
    for w in range(workers):
        code = (_ORACLE_WORKER.replace("ROOT_DIR", repr(ROOT)).replace("CONFIG", repr(config))
                .replace("BUDGET", repr(budget_s)).replace("NWORKERS", str(workers)).replace("WORKER", str(w)))
        procs.append(subprocess.Popen([sys.executable, "-c", code], stdin=subprocess.PIPE, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True, env=env))
    for pr in procs:
        line = pr.stdout.readline()
        if line.strip() != "ready":
            raise RuntimeError("oracle worker failed: " + pr.stderr.read()[-2000:])
    for pr in procs:
        pr.stdin.write("go\n")
        pr.stdin.flush()
    res = []
    for pr in procs:
        out, err = pr.communicate()
        if pr.returncode != 0:
            raise RuntimeError("oracle worker failed: " + err[-2000:])
        res.append(json.loads(out.strip().splitlines()[-1]))
    rate = sum(r["rows"] / r["seconds"] for r in res)
    return rate, {"rows": sum(r["rows"] for r in res), "seqs": sum(r["seqs"] for r in res),
                  "seconds": max(r["seconds"] for r in res), "workers": workers}


def oracle_prefill_ms(budget_s: float):
    """The fp64 oracle's chunked prefill of the GQA tree's 1137-row prompt
    (blocks 512 / 512 / 113 over the 2048-token root): a bounded sample of
    rows of each block, single-threaded, scaled to the block.  ms per block."""
    code = f"""
import json, sys, time
sys.path.insert(0, {ROOT!r})
import numpy as np, torch
torch.set_num_threads(1)
from prefix_shared_kv_tree_gb300 import workloads as W
from oracle import attention as A
from oracle.schedule import prefill_blocks
spec = W.SPECS["gqa_tree"]
g = torch.Generator().manual_seed(spec.seed)
n0 = spec.levels[0][0]; n = n0 + spec.prefill_prompt
k = torch.randn(n, spec.n_kv_heads, spec.head_dim, generator=g).to(torch.bfloat16).float().numpy()
v = torch.randn(n, spec.n_kv_heads, spec.head_dim, generator=g).to(torch.bfloat16).float().numpy()
q = torch.randn(spec.prefill_prompt, spec.n_q_heads, spec.head_dim, generator=g).to(torch.bfloat16).float().numpy()
out = []
off = 0
blocks = prefill_blocks(spec.prefill_prompt, spec.prefill_width)
for w in blocks:
    rows = 0; t = 0.0; r = 0
    p0 = n0 + off
    while t < {budget_s!r} / len(blocks) and r < w:
        t0 = time.perf_counter()
        A.prefill_attention(k[:p0 + r + 1], v[:p0 + r + 1], q[off + r:off + r + 1], p0 + r)
        t += time.perf_counter() - t0
        rows += 1
        r = (r + 37) if r + 37 < w else (r + 1)
    # rows sampled across the block; scale by mean keys per row
    out.append({{"rows_timed": rows, "seconds": t, "block": w}})
    off += w
print(json.dumps(out))
"""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError("oracle prefill timing failed: " + r.stderr[-2000:])
    res = json.loads(r.stdout.strip().splitlines()[-1])
    return [round(1e3 * b["seconds"] / b["rows_timed"] * b["block"], 1) for b in res], res


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(config: str, seconds: float):
    """The oracle on the host cores: single-threaded, and one single-threaded
    process per core.  Value = unique-KV GB/s equivalent of the all-core rate."""
    from prefix_shared_kv_tree_gb300 import workloads as W
    spec = W.SPECS[config]
    rows_per_step = spec.n_sequences * spec.n_q_heads
    cores = cpu_cores()
    r1, d1 = oracle_decode_rate(config, seconds / 2, 1)
    rn, dn = oracle_decode_rate(config, seconds / 2, cores)
    step1, stepn = rows_per_step / r1, rows_per_step / rn
    uniq = spec.unique_kv_bytes()
    return {"value": round(uniq / stepn / 1e9, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
            "ms_per_step": round(stepn * 1e3, 2),
            "single_thread": {"value": round(uniq / step1 / 1e9, 6), "ms_per_step": round(step1 * 1e3, 2),
                              "cores": 1},
            "sample": f"{dn['seqs']} whole sequences x {spec.n_q_heads} heads in {dn['seconds']:.1f} s on {cores} "
                      f"single-threaded processes (numpy fp64), and {d1['seqs']} in {d1['seconds']:.1f} s on one; "
                      f"scaled to a {spec.n_sequences}-sequence step"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from prefix_shared_kv_tree_gb300 import workloads as W
    spec = W.SPECS[args.config]
    total_budget = 120.0
    budget = min(60.0, max(5.0, total_budget / 2))
    cb = cpu_baseline(args.config, budget)
    line = {
        "impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": cb["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{spec.name}: {W.DESCRIPTIONS[spec.name]}"},
        "cpu_baseline": cb,
        "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- GPU leg
class L2Flush:
    """Evicts L2 between timed steps: writes 256 MiB, then reads another
    256 MiB so that the write-backs of the first happen outside the step."""

    def __init__(self):
        import torch
        self.w = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
        self.r = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")

    def __call__(self):
        self.w.fill_(1.0)
        self.r.sum()


def pool_chunks(spec, spare=64):
    chunks, mult = 0, 1
    for n, fan in spec.levels:
        mult *= fan
        chunks += mult * math.ceil(n / spec.chunk_size)
    return chunks + spare


def time_steps(step, steps: int, warmup: int, flush, stream):
    """Per-step device times (ms) of `step()`, CUDA events on `stream`, L2
    flushed before every step outside the events."""
    import torch
    for _ in range(max(3, warmup)):
        flush()
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def measure_config(pst, W, name, steps, warmup, flush, stream, min_share=0, flags=0):
    """µs per decode step of one more workload, measured in this run."""
    import torch
    spec = W.SPECS[name]
    wl = W.generate(spec, device="cuda")
    pool = pst.Pool(spec.n_q_heads, spec.n_kv_heads, spec.head_dim, spec.chunk_size, pool_chunks(spec), spec.dtype,
                    min_share, 0, flags, device=torch.cuda.current_device())
    W.insert_all(pool, wl)
    q = wl.q.contiguous()
    out = torch.empty_like(q)
    pool.decode_attention(q, out)
    torch.cuda.synchronize()
    assert pool.check_device() == 0
    times = time_steps(lambda: pool.decode_attention(q, out), steps, warmup, flush, stream)
    assert pool.check_device() == 0
    hbm, _, _ = measured_peaks()
    dist = distribution(times)
    ms = dist["mean"] * 1e-3
    gbs = spec.unique_kv_bytes() / (ms * 1e-3) / 1e9
    res = {"us_per_step": dist, "unique_kv_gbs": round(gbs, 1), "frac_of_measured_hbm": round(gbs / hbm, 4),
           "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4), "unique_kv_bytes": spec.unique_kv_bytes(),
           "min_share": min_share or 2}
    pool.close()
    del wl
    torch.cuda.empty_cache()
    return res


def measure_prefill(pst, W, steps, flush, stream):
    """The GQA tree's chunked prefill (Chunked Prefill, sections 1-3): a new
    sequence that matches the 2048-token root, then its 1137 new tokens as
    causal blocks of 512 / 512 / 113 rows.  Per block: the whole call (block
    K/V appended and scattered into the pool, table upload, attention) and
    the attention kernel alone (library events), method FLOPs / kernel time
    against the measured bf16 peak."""
    import torch
    from oracle.schedule import prefill_blocks  # the block split only (Chunked Prefill, section 3)
    spec = W.SPECS["gqa_tree"]
    wl = W.generate(spec, device="cuda")
    blocks = prefill_blocks(spec.prefill_prompt, spec.prefill_width)
    pool = pst.Pool(spec.n_q_heads, spec.n_kv_heads, spec.head_dim, spec.chunk_size,
                    pool_chunks(spec, 64 + 2 * math.ceil(spec.prefill_prompt / spec.chunk_size)), spec.dtype,
                    device=torch.cuda.current_device())
    W.insert_all(pool, wl)
    root = wl.segments[0].tokens.cpu()
    n0 = root.shape[0]
    outs = [torch.empty(w, spec.n_q_heads, spec.head_dim, dtype=W.DTYPES[spec.dtype], device="cuda") for w in blocks]
    offs = [sum(blocks[:i]) for i in range(len(blocks))]
    args = [(wl.prefill_tokens[o:o + w].cpu(), wl.prefill_q[o:o + w].contiguous(),
             wl.prefill_k[o:o + w].contiguous(), wl.prefill_v[o:o + w].contiguous()) for o, w in zip(offs, blocks)]
    call_ms = [[] for _ in blocks]
    kern_ms = [[] for _ in blocks]
    total_ms = []
    for it in range(3 + steps):
        sid, m = pool.insert(root)
        assert m == n0
        flush()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(blocks) + 1)]
        ev[0].record(stream)
        for b, (tok, q, k, v) in enumerate(args):
            pool.prefill_attend(sid, tok, q, k, v, outs[b])
            ev[b + 1].record(stream)
        torch.cuda.synchronize()
        # the same blocks once more with the library's kernel events (a
        # second sequence; these events sit between launches)
        sid2, _ = pool.insert(root)
        pool.set_profiling(True)
        kt = []
        for b, (tok, q, k, v) in enumerate(args):
            pool.prefill_attend(sid2, tok, q, k, v, outs[b])
            kt.append(max(pool.phase_times()[:2]))
        pool.set_profiling(False)
        pool.remove(sid)
        pool.remove(sid2)
        if it >= 3:
            for b in range(len(blocks)):
                call_ms[b].append(ev[b].elapsed_time(ev[b + 1]))
                kern_ms[b].append(kt[b])
            total_ms.append(ev[0].elapsed_time(ev[-1]))
    assert pool.check_device() == 0
    _, tf_peak, kind = measured_peaks()
    res = {"workload": f"gqa_tree prefill: {spec.prefill_prompt} new tokens after the {n0}-token root, W = "
                       f"{spec.prefill_width} ({'/'.join(map(str, blocks))}), Hq {spec.n_q_heads} / Hkv "
                       f"{spec.n_kv_heads}, d {spec.head_dim}, bf16",
           "blocks": [], "peak_tflops": tf_peak, "peak_kind": f"{kind} bf16 dense (burst)"}
    flops_total, kern_total = 0, 0.0
    for b, (o, w) in enumerate(zip(offs, blocks)):
        fl = prefill_flops(n0 + o, w, spec.n_q_heads, spec.head_dim)
        km = statistics.median(kern_ms[b])
        cm = statistics.median(call_ms[b])
        flops_total += fl
        kern_total += km
        res["blocks"].append({"rows": w, "p0": n0 + o, "gflop": round(fl / 1e9, 3), "call_us": round(1e3 * cm, 2),
                              "kernel_us": round(1e3 * km, 2), "tflops": round(fl / (km * 1e-3) / 1e12, 1),
                              "frac_of_peak": round(fl / (km * 1e-3) / 1e12 / tf_peak, 4)})
    tm = statistics.median(total_ms)
    res.update({"gflop": round(flops_total / 1e9, 3), "total_us": round(1e3 * tm, 2),
                "kernel_us": round(1e3 * kern_total, 2),
                "tflops": round(flops_total / (kern_total * 1e-3) / 1e12, 1),
                "frac_of_peak": round(flops_total / (kern_total * 1e-3) / 1e12 / tf_peak, 4),
                "timed_iterations": steps,
                "note": "median per block; call = K/V scatter + table upload + attention, L2 flushed before "
                        "each prompt; kernel = the attention kernel alone (library events)"})
    pool.close()
    return res


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
    # spare chunks for the decode loop's appends (a new leaf chunk every c steps)
    spare = 64 + spec.n_sequences * (2 + 2 * args.loop_steps // spec.chunk_size)
    pool = pst.Pool(spec.n_q_heads, spec.n_kv_heads, spec.head_dim, spec.chunk_size, pool_chunks(spec, spare),
                    spec.dtype, args.min_share, 0, args.flags, device=dev)
    W.insert_all(pool, wl)
    q = wl.q.contiguous()
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream()
    flush = L2Flush()
    pool.decode_attention(q, out)
    torch.cuda.synchronize()
    assert pool.check_device() == 0

    clocks = ClockSampler(dev)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches = [0]

    def step():
        pool.decode_attention(q, out)
        launches[0] += pool.last_launch_count()
    times = time_steps(step, args.steps, args.warmup, flush, stream)
    launches = launches[0] * args.steps // (args.steps + max(3, args.warmup))
    st = pool.stats()  # the timed workload's tables (the decode loop below grows the tree)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    dist_us = distribution(times)
    ms = max_over_ranks(sum(times) / len(times), device="cuda")

    # ---- per-kernel durations (library events on the streams the kernels run on);
    # a separate pass, because events between the kernels can stop them overlapping
    pool.set_profiling(True)
    n_prof = max(3, min(args.steps, 100))
    phase = []
    for i in range(n_prof):
        flush()
        pool.decode_attention(q, out)
        phase.append(pool.phase_times())
    pool.set_profiling(False)
    assert pool.check_device() == 0

    # ---- e2e through the host-buffer entry point (H2D q, decode, D2H out, sync)
    q_host = q.cpu().pin_memory()
    out_host = torch.empty_like(q_host).pin_memory()
    e2e_times = []
    for i in range(max(3, args.warmup) + args.steps):
        flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        pool.decode_attention_host(q_host, out_host)
        t1 = time.perf_counter()
        if i >= max(3, args.warmup):
            e2e_times.append(t1 - t0)
    assert torch.equal(out_host, out.cpu())
    e2e_ms = 1e3 * sum(e2e_times) / len(e2e_times)

    # ---- decode loop (runs after the timed step: it grows every sequence).
    # Per step one token appended to every sequence, then the decode step
    # replayed from a CUDA graph that the library captures again only after a
    # structural change (a new leaf chunk every c steps).  (a) wall clock over
    # the whole loop.  (b) the same loop with a stand-in for the layer's
    # earlier kernels enqueued before each step (a ~200 µs spin kernel): the
    # host rebuilds the tables and captures the graph while the GPU runs it
    # (ChunkAttention, Knowl 5), so steps with a structural change should not
    # take longer on the GPU; per-step GPU periods from events at each step's
    # start, split by whether the step rebuilt the tables.
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
        # (b) overlap of the host rebuild with earlier GPU work
        spin_cycles = int(200e-6 * 1.9e9)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.loop_steps + 1)]
        rebuilt = []
        for i in range(args.loop_steps):
            evs[i].record(stream)
            torch.cuda._sleep(spin_cycles)
            before = pool.stats()["rebuild_count"]
            pool.append_batch(ids, toks, k_app, v_app, stream=sh)
            pool.decode_attention_graph(q, out_loop, stream=sh)
            rebuilt.append(pool.stats()["rebuild_count"] > before)
        evs[-1].record(stream)
        torch.cuda.synchronize()
        per = [evs[i].elapsed_time(evs[i + 1]) for i in range(args.loop_steps)]
        # the first steps fill the host's lead over the GPU; skip them
        per, rebuilt = per[4:], rebuilt[4:]
        with_rb = [1e3 * x for x, r in zip(per, rebuilt) if r]
        without = [1e3 * x for x, r in zip(per, rebuilt) if not r]
        loop["overlap"] = {
            "stand_in": "torch.cuda._sleep spin kernel of ~200 us before each step (a layer's earlier kernels)",
            "steps_with_rebuild": len(with_rb), "steps_without": len(without),
            "us_per_step_with_rebuild": round(statistics.mean(with_rb), 2) if with_rb else None,
            "us_per_step_without": round(statistics.mean(without), 2) if without else None,
            "max_us_with_rebuild": round(max(with_rb), 2) if with_rb else None,
            "last_rebuild_us": round(pool.stats()["last_rebuild_us"], 1)}
        assert pool.check_device() == 0

    hbm, tf_peak, peak_kind = measured_peaks()
    phase_ms = [sum(p[j] for p in phase) / len(phase) for j in range(3)]
    names = ["chunk_first_tc", "sequence_first_simt", "whole_call"]
    dom = max(range(2), key=lambda j: phase_ms[j])  # the dominant kernel (not the whole call)
    min_share = args.min_share or 2
    dom_bytes = [shared_bytes(spec, min_share), private_bytes(spec, min_share)][dom]
    if phase_ms[0] == 0.0:  # no chunk-first launch: the sequence-first kernel reads every chunk
        dom_bytes = spec.unique_kv_bytes() + qo_bytes(spec)
    achieved = dom_bytes / (phase_ms[dom] * 1e-3) / 1e9
    pool.close()
    del wl
    torch.cuda.empty_cache()

    # ---- the other decode workloads (share4k, noshare, gqa_tree, and the
    # sequence-first-only controls), measured in this run
    configs = None
    if world == 1 and not args.no_configs:
        csteps = max(20, min(args.steps, 200))
        configs = {}
        for name in ("share4k", "noshare", "gqa_tree"):
            configs[name] = measure_config(pst, W, name, csteps, args.warmup, flush, stream)
        # sequence-first-only controls (every chunk on the sequence-first kernel)
        for name in ("noshare", args.config):
            configs[f"{name}_seq_first_only"] = measure_config(pst, W, name, csteps, args.warmup, flush, stream,
                                                               min_share=2**31 - 1)
    prefill = None
    if world == 1 and not args.no_prefill:
        prefill = measure_prefill(pst, W, max(5, min(args.steps, 50)), flush, stream)

    if rank != 0:
        return
    unique = spec.unique_kv_bytes()
    value = whole_job_gbs(unique, ms, world)
    qbytes = qo_bytes(spec)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 6), "us_per_step": round(ms * 1e3, 3),
        "step_us": dist_us,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": spec.dtype,
        "data": "synthetic (seeded N(0,1) Q/K/V drawn on the GPU, seeded token ids)",
        "config": {"workload": f"{spec.name}: {W.DESCRIPTIONS[spec.name]}",
                   "l2": "flushed between timed steps (256 MiB write, then 256 MiB read)",
                   "unique_kv_bytes": unique, "logical_kv_bytes": spec.logical_kv_bytes(),
                   "min_share": min_share, "flags": args.flags,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "frac_of_peak": round(value / world / hbm, 4),
        "frac_of_nominal_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
        "phase_ms": {names[j]: round(phase_ms[j], 5) for j in range(3)},
        "roofline": {"bound": "hbm", "kernel": names[dom], "achieved": round(achieved, 2), "peak": hbm,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "algorithmic_bytes_per_launch": dom_bytes,
                     "traffic": traffic_for(names[dom], spec.name)},
        "e2e": {"value": round(unique / (e2e_ms * 1e-3) / 1e9, 3), "unit": UNIT, "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": qbytes, "d2h_bytes_per_step": qbytes},
        "gpu_launches": launches,
        "clocks": clk,
        "pool": {k: st[k] for k in ("used_chunks", "shared_chunks", "phase1_items", "phase2_items", "partial_rows",
                                    "phase1_ctas", "phase2_ctas", "simt_first")},
        "decode_loop": loop,
        "configs": configs,
        "prefill": prefill,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(args.config, args.cpu_seconds)
        if prefill is not None:
            ms_blocks, _ = oracle_prefill_ms(6.0)
            line["cpu_baseline"]["prefill_ms_per_block"] = ms_blocks
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
               "--warmup", str(args.warmup), "--no-cpu-baseline", "--loop-steps", "0", "--no-configs",
               "--no-prefill",
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


def run_prefill_only(args):
    import torch
    torch.cuda.set_device(0)
    from prefix_shared_kv_tree_gb300 import build as B
    B.build_library()
    from prefix_shared_kv_tree_gb300 import pst
    from prefix_shared_kv_tree_gb300 import workloads as W
    res = measure_prefill(pst, W, max(1, args.steps), L2Flush(), torch.cuda.current_stream())
    print(json.dumps({"prefill": res}), flush=True)


def main():
    args = parse()
    if args.prefill_only:
        run_prefill_only(args)
        return
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
