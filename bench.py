#!/usr/bin/env python
"""Paged decode attention benchmark on GB300.

One step = the whole decode hot path for one batch: append each sequence's
newest K/V at its slot (pa_append_kv), copy-on-write copies if the step has
any (pa_copy_blocks), and paged decode attention (pa_decode).  The workload is
the Llama-3-70B-shaped decode layer (batch 256, 64 query / 8 KV heads,
head_dim 128, block 16, context U[1024, 8192], bf16, pool 1.1x, seeded random
block placement built by the host BlockManager).  Inputs are synthetic and
seeded; the KV stream of one step (~4.8 GB) is far larger than L2, so no L2
flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line on rank 0.  ``value`` is effective HBM GB/s: algorithmic
bytes of all ranks' steps / max-over-ranks device time.  ``--impl reference``
times the CPU fp64 oracle (the reference arm of this build) on a bounded
sample of the same workload.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention: effective HBM GB/s (% of GB300 peak), tokens/s"
WORKLOAD = "llama3_70b_b256"
FALLBACK_HBM_GBS = 6800.0

# DRAM traffic of the dominant kernel per launch, from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum) of a SMALL case: the first 64
# sequences of the workload (inputs above L2, a few GB on the device).  The
# line scales it to the full launch by algorithmic bytes (traffic grows in
# proportion to the KV stream).  Keyed by a hash of the kernel sources, the
# cache type and the workload; any other key (a changed source, another
# workload or kernel instantiation) reports null.
#   (hash, kv dtype, workload): (captured dram bytes, algorithmic bytes of the captured launch)
TRAFFIC = {
    ("f1214767ababa837", "bf16", "llama3_70b_b256"): (1_217_302_272 + 7_294_976, 1_216_111_324),
    ("f1214767ababa837", "fp8_e4m3", "llama3_70b_b256"): (609_424_128 + 7_066_112, 609_141_468),
    ("f1214767ababa837", "int4", "llama3_70b_b256"): (324_384_000 + 4_621_312, 324_624_348),
}

KERNEL_SOURCES = ("decode_kernel.cuh", "decode_common.cuh", "decode_tok.cuh", "ptx.cuh")


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "paged_kv_cache_254_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def scaled_traffic(khash: str, kv: str, workload: str, alg_bytes: int):
    """Captured DRAM bytes of the small case scaled to `alg_bytes`, or None."""
    rec = TRAFFIC.get((khash, kv, workload))
    if rec is None:
        return None
    dram, alg = rec
    return int(round(dram * alg_bytes / alg))


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=WORKLOAD)
    ap.add_argument("--seed", type=int, default=None)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kv-dtype", choices=["bf16", "fp8_e4m3", "fp8_e5m2", "int4"], default="bf16",
                    help="cache element type (fp8: 8-bit cache, int4: 4-bit cache with per-row scales; "
                         "quantising append, quantized decode)")
    ap.add_argument("--plain-decode", action="store_true",
                    help="decode shared-prompt batches without the prefix-aware pass")
    ap.add_argument("--q-len", type=int, default=1,
                    help="query tokens per sequence per step (> 1: each sequence appends that many tokens and "
                         "pa_decode_multi attends them causally -- a chunked-prefill / speculative-verify step)")
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="truncate the batch (small profiling captures); the JSON line says so")
    ap.add_argument("--cpu-worker", action="store_true", help=argparse.SUPPRESS)
    return ap.parse_args(argv)


# --------------------------------------------------------------------------- accounting
def decode_bytes(ctx, Hq, Hkv, d, B, elem=2, q_elem=2, q_len=1, row_extra=0) -> int:
    """Bytes the method must move for one decode call: every cached K and V
    element once (elem bytes each, plus row_extra bytes of scales per cached
    (token, head)), Q and O once (q_len rows per sequence), the block-table
    entries in use and the context lengths."""
    ctx = [int(c) for c in ctx]
    kv = int(sum(ctx) * Hkv * (d * elem * 2 + row_extra))
    qo = 2 * len(ctx) * q_len * Hq * d * q_elem
    tables = sum(-(-c // B) for c in ctx) * 4
    return kv + qo + tables + 4 * len(ctx)


def append_bytes(T, Hkv, d, elem=2, new_elem=2, row_extra=0) -> int:
    """K and V rows read (new_elem bytes each) and written to the cache (elem
    bytes each, plus row_extra bytes of scales), plus the int64 slots."""
    return int(T * Hkv * (d * (elem + new_elem) * 2 + row_extra)) + 8 * T


def copy_bytes(n, Hkv, B, d, elem=2, row_extra=0) -> int:
    return int(2 * n * Hkv * B * (d * elem * 2 + row_extra))


def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def max_over_ranks(x: float, dist, device) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- workload
def unique_decode_bytes(tables, ctx, Hq, Hkv, d, B, elem=2, q_elem=2) -> int:
    """Like decode_bytes, but each physical block's valid tokens count once
    however many sequences share it (the shared-prompt workload)."""
    filled = {}
    for row, n in zip(tables, ctx):
        n = int(n)
        for i in range(-(-n // B)):
            b = int(row[i])
            filled[b] = max(filled.get(b, 0), min(B, n - i * B))
    kv = sum(filled.values()) * Hkv * d * elem * 2
    qo = 2 * len(ctx) * Hq * d * q_elem
    return kv + qo + sum(-(-int(c) // B) for c in ctx) * 4 + 4 * len(ctx)


FP8_SCALE = 0.25


def make_workload(name, device, seed, num_seqs=None, kv_dtype="bf16", q_len=1) -> dict:
    """Device tensors of one decode step.  Block tables, lengths, slot mapping
    and copy list come from the host BlockManager (seeded random placement);
    values from the seeded workload generators."""
    import numpy as np
    import torch

    from paged_kv_cache_254_gb300 import BlockManager
    from workloads import CONFIGS, SAMPLINGS, make_decode_case, make_sampling_case

    if name in SAMPLINGS:
        cfg = SAMPLINGS[name]
        seed = cfg.seed if seed is None else seed
        case = make_sampling_case(cfg, device=device, seed=seed)
        B, S = cfg.block_size, cfg.samples
        G = case.prompt_blocks.shape[0]
        bm = BlockManager(case.num_blocks, B, seed=seed + 17)
        for g in range(G):
            if bm.add_sequence((g, 0), cfg.prompt_len) is None:
                raise RuntimeError("pool too small")
            for j in range(1, S):
                bm.fork((g, 0), (g, j))
        seqs = [(g, j) for g in range(G) for j in range(S)]
        reqs = [(sq, int(case.tails[i]) + 1) for i, sq in enumerate(seqs)]
        t0 = time.perf_counter()
        slots = bm.append_slots(reqs)                # each sample's tail and new token
        host_ms = (time.perf_counter() - t0) * 1e3
        max_blocks = cfg.max_blocks_per_seq
        desc, Hq, Hkv, d = cfg.description, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim
    else:
        cfg = CONFIGS[name]
        seed = cfg.seed if seed is None else seed
        case = make_decode_case(cfg, device=device, seed=seed, values=True, num_seqs=num_seqs)
        B = cfg.block_size
        bm = BlockManager(case.num_blocks, B, seed=seed + 17)
        seqs = list(range(len(case.context_lens)))
        for s in seqs:
            if bm.add_sequence(s, int(case.context_lens[s]) - q_len) is None:
                raise RuntimeError("pool too small")
        t0 = time.perf_counter()
        # the newest token (or the chunk of q_len new tokens) of every sequence
        slots = bm.append_slots(seqs if q_len == 1 else [(s, q_len) for s in seqs])
        host_ms = (time.perf_counter() - t0) * 1e3
        if q_len > 1:
            from workloads import make_values
            gq = torch.Generator(device=device).manual_seed((seed or 0) + 77)
            n = len(seqs)
            case.q = make_values((n * q_len, cfg.num_q_heads, cfg.head_dim), cfg.dtype, gq, device)
            case.k_new = make_values((n * q_len, cfg.num_kv_heads, cfg.head_dim), cfg.dtype, gq, device)
            case.v_new = make_values((n * q_len, cfg.num_kv_heads, cfg.head_dim), cfg.dtype, gq, device)
        max_blocks = cfg.max_blocks_per_seq
        desc, Hq, Hkv, d = cfg.description, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim
    copies = bm.take_copies()
    tables = bm.block_tables(seqs, max_blocks)
    ctx = bm.context_lens(seqs)
    gstarts, gprefix = bm.shared_prefix_groups(seqs)
    slots = slots.astype(np.int64)
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)  # noqa: E731
    if kv_dtype == "int4":
        # a 4-bit cache of random codes and scales, one piece per (block, head)
        from workloads import make_int4_pool
        g4 = torch.Generator(device=device).manual_seed((seed or 0) + 99)
        NB, Hkv_, B_, d_ = case.k_pool.shape
        case.k_pool = None
        case.v_pool = None
        torch.cuda.empty_cache()
        case.k_pool = make_int4_pool(NB, Hkv_, B_, d_, g4, device)
        case.v_pool = None
    elif kv_dtype != "bf16":
        # an 8-bit cache of random codes: per (block, head) K rows, then V dims-first
        from workloads import make_codes
        g8 = torch.Generator(device=device).manual_seed((seed or 0) + 99)
        NB, Hkv_, B_, d_ = case.k_pool.shape
        case.k_pool = None
        case.v_pool = None
        torch.cuda.empty_cache()
        case.k_pool = make_codes((NB, Hkv_, 2, B_, d_), g8, device)   # the one 8-bit pool
        case.v_pool = None
    return {
        "name": name, "description": desc, "Hq": Hq, "Hkv": Hkv, "d": d, "B": B,
        "num_blocks": case.num_blocks, "scale": case.scale,
        "q": case.q, "k_pool": case.k_pool, "v_pool": case.v_pool, "k_new": case.k_new, "v_new": case.v_new,
        "tables_h": tables, "ctx_h": ctx, "slots_h": slots, "copies_h": copies,
        "tables": to(tables), "ctx": to(ctx), "slots": to(slots), "copies": to(copies),
        "host_block_manager_ms": host_ms, "bm_stats": bm.stats(),
        "shared": name in SAMPLINGS, "kv_dtype": kv_dtype,
        "group_starts": to(gstarts), "group_prefix": to(gprefix), "n_groups": int(gprefix.size),
        "q_len": q_len, "q_start": to((np.arange(len(seqs) + 1) * q_len).astype(np.int32)),
    }


# --------------------------------------------------------------------------- CPU oracle timing
def cpu_worker(args):
    """Time the fp64 oracle on the first sequences of the workload (host
    cores, single-threaded BLAS) and print one JSON object."""
    from oracle.attention import decode_multi_ref, decode_ref
    from workloads import CONFIGS, SAMPLINGS, make_decode_case, make_sampling_case, sampling_tables
    import torch

    if args.config in SAMPLINGS:
        cfg = SAMPLINGS[args.config]
        case = make_sampling_case(cfg, device="cpu", seed=args.seed, groups=8)
        tables, ctx_all = sampling_tables(case)
        n_total, Hq, Hkv, d, B = cfg.num_seqs, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim, cfg.block_size
    else:
        cfg = CONFIGS[args.config]
        case = make_decode_case(cfg, device="cpu", seed=args.seed, num_seqs=min(cfg.num_seqs, 160))
        tables, ctx_all = case.block_tables, case.context_lens
        n_total, Hq, Hkv, d, B = cfg.num_seqs, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim, cfg.block_size
    n_gen = len(ctx_all)
    ql = args.q_len
    if ql > 1:
        gq = torch.Generator().manual_seed(77)
        qm = torch.randn((n_gen * ql, Hq, d), generator=gq).to(case.q.dtype)
    done = 0
    t0 = time.perf_counter()
    while done < n_gen and time.perf_counter() - t0 < args.cpu_seconds:
        if ql > 1:
            decode_multi_ref(qm[done * ql:(done + 1) * ql], case.k_pool, case.v_pool, tables[done:done + 1],
                             ctx_all[done:done + 1], [0, ql], case.scale)
        else:
            rows = [(done, h) for h in range(Hq)]
            decode_ref(case.q, case.k_pool, case.v_pool, tables, ctx_all, case.scale, rows=rows)
        done += 1
    dt = time.perf_counter() - t0
    ctx_done = [int(c) for c in ctx_all[:done]]
    if args.config in SAMPLINGS:
        nbytes = unique_decode_bytes(tables[:done], ctx_done, Hq, Hkv, d, B)
    else:
        nbytes = decode_bytes(ctx_done, Hq, Hkv, d, B, q_len=ql)
    nbytes += append_bytes(done * ql, Hkv, d)
    print(json.dumps({
        "value": nbytes / dt / 1e9, "unit": "GB/s", "tokens_per_s": done * ql / dt, "seconds": dt,
        "sample": f"first {done} of {n_total} sequences of {cfg.name} (all {Hq} query heads, "
                  f"{ql} query token(s) each, {sum(ctx_done)} cached tokens), fp64 oracle",
        "cores": 1, "host_cores": len(os.sched_getaffinity(0)), "blas_threads": 1,
    }))


def run_cpu_baseline(args) -> dict:
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    env.pop("RANK", None)
    env.pop("WORLD_SIZE", None)
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-worker", "--config", args.config,
           "--cpu-seconds", str(args.cpu_seconds), "--q-len", str(args.q_len)]
    if args.seed is not None:
        cmd += ["--seed", str(args.seed)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=600)
    if r.returncode != 0:
        return {"value": None, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": "failed: " + r.stderr[-300:]}
    out = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": out["value"], "unit": "GB/s", "cores": out["cores"], "kind": "oracle",
            "sample": out["sample"], "tokens_per_s": out["tokens_per_s"], "seconds": out.get("seconds"),
            "host_cores": out.get("host_cores"), "blas_threads": out.get("blas_threads")}


def reference_arm(args):
    world, rank, local = dist_env()
    if world > 1 and rank != 0:
        return
    from workloads import CONFIGS, SAMPLINGS
    cfg = SAMPLINGS[args.config] if args.config in SAMPLINGS else CONFIGS[args.config]
    vals = []
    sample = None
    tok = []
    secs = []
    per = max(2.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup + args.steps):
        a = argparse.Namespace(**vars(args))
        a.cpu_seconds = per
        res = run_cpu_baseline(a)
        if i >= args.warmup and res["value"] is not None:
            vals.append(res["value"])
            tok.append(res["tokens_per_s"])
            secs.append(res["seconds"])
            sample = res["sample"]
    value = statistics.median(vals) if vals else None
    tps = statistics.median(tok) if tok else None
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        # wall time of one timed step: the oracle over its bounded sample
        "ms_per_step": (1e3 * statistics.median(secs)) if secs else None,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "tokens_per_s": tps,
        "config": {"workload": cfg.name, "description": cfg.description,
                   "ms_per_step": "one step = the oracle over a bounded sample of the workload (see sample)",
                   "ms_per_full_batch_at_sampled_rate": (1e3 * cfg.num_seqs * args.q_len / tps) if tps else None},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"per step, about {per:.0f} s of: {sample}"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# --------------------------------------------------------------------------- GPU arm
def timed_rows(decode_ms, append_ms, copy_ms, dec_bytes, app_bytes, cp_bytes) -> dict:
    """Per-call device times of the step's three parts over the timed steps
    (CUDA events on the launching stream): median with p10 / p90, and the
    algorithmic GB/s at the median."""
    def row(ms, nbytes):
        if not ms:
            return None
        qs = statistics.quantiles(ms, n=10, method="inclusive") if len(ms) > 1 else [ms[0]] * 9
        med = statistics.median(ms)
        return {"ms_p50": round(med, 5), "ms_p10": round(qs[0], 5), "ms_p90": round(qs[8], 5),
                "bytes": nbytes, "gbs_at_p50": round(nbytes / (med * 1e-3) / 1e9, 2) if med > 0 else None}
    return {"decode": row(decode_ms, dec_bytes), "append": row(append_ms, app_bytes),
            "copy": row(copy_ms, cp_bytes) if copy_ms else None}


def gpu_arm(args):
    import numpy as np
    import torch

    import paged_kv_cache_254_gb300 as pa
    from paged_kv_cache_254_gb300 import _build
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    _build.build()

    seed = None if args.seed is None and rank == 0 else (args.seed or 0) + 1000 * rank
    if args.q_len > 1 and (args.kv_dtype != "bf16" or args.config.startswith("parallel_sampling")):
        raise SystemExit("--q-len > 1 runs the 16-bit cache on the decode workloads")
    st = make_workload(args.config, device, seed, args.num_seqs, args.kv_dtype, q_len=args.q_len)
    multi = args.q_len > 1
    Hq, Hkv, d, B = st["Hq"], st["Hkv"], st["d"], st["B"]
    N = len(st["ctx_h"])
    T = int(st["slots_h"].shape[0])
    stream = torch.cuda.current_stream(device)
    out = torch.empty_like(st["q"])
    quant = args.kv_dtype != "bf16"
    int4 = args.kv_dtype == "int4"
    fp8 = quant and not int4
    fmt = args.kv_dtype[4:] if fp8 else None
    ws = None if (quant or multi) else pa.workspace_for(st["q"], st["k_pool"], st["tables"])
    n_copies = int(st["copies"].shape[0])
    use_prefix = st["n_groups"] > 0 and not args.plain_decode and not quant

    def step(q, k_new, v_new, slots, tables, ctx, ev=None):
        # ev: four events around the copies, the append and the decode call
        launches = 0
        if ev is not None:
            ev[0].record(stream)
        if n_copies:
            if int4:
                pa.pa_copy_blocks_int4(st["copies"], st["k_pool"])
            elif fp8:
                pa.pa_copy_blocks_fp8(st["copies"], st["k_pool"], kv_format=fmt)
            else:
                pa.pa_copy_blocks(st["copies"], st["k_pool"], st["v_pool"])
            launches += 1
        if ev is not None:
            ev[1].record(stream)
        if int4:
            pa.pa_append_kv_int4(k_new, v_new, slots, st["k_pool"])
        elif fp8:
            pa.pa_append_kv_fp8(k_new, v_new, slots, st["k_pool"], FP8_SCALE, FP8_SCALE, kv_format=fmt)
        else:
            pa.pa_append_kv(k_new, v_new, slots, st["k_pool"], st["v_pool"])
        if ev is not None:
            ev[2].record(stream)
        if int4:
            pa.pa_decode_int4(q, st["k_pool"], tables, ctx, st["scale"], out=out)
        elif fp8:
            pa.pa_decode_fp8(q, st["k_pool"], tables, ctx, st["scale"], FP8_SCALE, FP8_SCALE, kv_format=fmt, out=out)
        elif multi:
            pa.pa_decode_multi(q, st["k_pool"], st["v_pool"], tables, ctx, st["q_start"], st["scale"],
                               max_q_len=args.q_len, out=out)
        elif use_prefix:
            pa.pa_decode_shared_prefix(q, st["k_pool"], st["v_pool"], tables, ctx, st["group_starts"],
                                       st["group_prefix"], st["scale"], out=out)
            launches += 1
        else:
            pa.pa_decode(q, st["k_pool"], st["v_pool"], tables, ctx, st["scale"], out=out, workspace=ws)
        if ev is not None:
            ev[3].record(stream)
        return launches + 4   # append, and the decode call's pre-pass, attention and merge kernels

    dev_args = (st["q"], st["k_new"], st["v_new"], st["slots"], st["tables"], st["ctx"])
    for _ in range(args.warmup):
        step(*dev_args)
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    if local == 0:
        clocks.start()
        time.sleep(0.05)
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches = 0
    t_start.record(stream)
    for i in range(args.steps):
        launches += step(*dev_args, ev=evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop() if local == 0 else None
    total_ms = t_start.elapsed_time(t_end)
    decode_ms = [e[2].elapsed_time(e[3]) for e in evs]
    append_ms = [e[1].elapsed_time(e[2]) for e in evs]
    copy_ms = [e[0].elapsed_time(e[1]) for e in evs] if n_copies else None
    max_ms = max_over_ranks(total_ms, dist, device)

    # ---- end to end through the public API from pinned host buffers ----
    host = {k: t.detach().cpu().pin_memory() for k, t in zip(("q", "k_new", "v_new"), dev_args[:3])}
    host["slots"] = torch.from_numpy(st["slots_h"]).pin_memory()
    host["tables"] = torch.from_numpy(st["tables_h"]).pin_memory()
    host["ctx"] = torch.from_numpy(st["ctx_h"]).pin_memory()
    if multi:
        host["q_start"] = st["q_start"].cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    dbuf = {k: torch.empty_like(v, device=device) for k, v in host.items()}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = out_h.numel() * out_h.element_size()

    def e2e_step():
        for k in host:
            dbuf[k].copy_(host[k], non_blocking=True)
        if multi:
            st["q_start"] = dbuf["q_start"]
        step(dbuf["q"], dbuf["k_new"], dbuf["v_new"], dbuf["slots"], dbuf["tables"], dbuf["ctx"])
        out_h.copy_(out, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, device)

    # ---- numbers ----
    kv_elem = 0.5 if int4 else 1 if fp8 else 2
    rx = 8 if int4 else 0                          # fp32 K and V scale per cached (token, head)
    dbytes = decode_bytes(st["ctx_h"], Hq, Hkv, d, B, elem=kv_elem, q_len=args.q_len, row_extra=rx)
    ubytes = unique_decode_bytes(st["tables_h"], st["ctx_h"], Hq, Hkv, d, B, elem=kv_elem) if st["shared"] else dbytes
    extra = (append_bytes(T, Hkv, d, elem=kv_elem, row_extra=rx) +
             copy_bytes(n_copies, Hkv, B, d, elem=kv_elem, row_extra=rx))
    step_bytes = ubytes + extra
    value = world * args.steps * step_bytes / (max_ms * 1e-3) / 1e9
    tokens = world * args.steps * N * args.q_len / (max_ms * 1e-3)
    kv_tokens = world * args.steps * float(np.sum(st["ctx_h"])) / (max_ms * 1e-3)
    e2e_value = world * args.steps * step_bytes / (e2e_ms * 1e-3) / 1e9
    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = float(peak) if peak else FALLBACK_HBM_GBS
    dec_avg_ms = statistics.mean(decode_ms)
    achieved = ubytes / (dec_avg_ms * 1e-3) / 1e9
    khash = kernel_hash()
    traffic = None if (multi or use_prefix) else scaled_traffic(khash, args.kv_dtype, args.config, ubytes)

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = run_cpu_baseline(args)
    cfg_out = {"workload": st["name"], "description": st["description"], "num_seqs": N, "num_q_heads": Hq,
               "num_kv_heads": Hkv, "head_dim": d, "block_size": B, "num_blocks": st["num_blocks"],
               "mean_context": float(np.mean(st["ctx_h"])), "appended_tokens": T, "cow_copies": n_copies,
               "bytes_per_step": step_bytes,
               "l2": "inputs larger than L2 (KV stream %.2f GB per step), no flush" % (dbytes / 1e9),
               "parallelism": f"replicas x{world}", "truncated_batch": args.num_seqs,
               "kv_cache": args.kv_dtype, "q_len": args.q_len}
    if st["shared"]:
        cfg_out["bytes_note"] = ("value counts each shared physical block once (unique bytes); "
                                 "logical_gbs counts every sequence's reads")
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(max_ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if not quant else f"bf16 q/out, {args.kv_dtype} cache",
        "data": "synthetic (seeded N(0,1) values, random block placement)",
        "config": cfg_out,
        "tokens_per_s": round(tokens, 1),
        "kv_tokens_per_s": round(kv_tokens, 1),
        "timed_rows": timed_rows(decode_ms, append_ms, copy_ms, ubytes,
                                 append_bytes(T, Hkv, d, elem=kv_elem, row_extra=rx),
                                 copy_bytes(n_copies, Hkv, B, d, elem=kv_elem, row_extra=rx)),
        "pct_of_hbm_peak": round(100 * value / (world * peak), 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     # achieved = the whole call (all its launches) timed with CUDA events
                     "timed": ("pa_decode_shared_prefix call (prefix pass, pre-pass, decode, merge)" if use_prefix
                               else "pa_decode_multi call (pre-pass, attention, merge)" if multi
                               else "pa_decode_int4 call (pre-pass, attention, merge)" if int4
                               else "pa_decode_fp8 call (pre-pass, attention, merge)" if fp8
                               else "pa_decode call (pre-pass, attention, merge)"),
                     "kernel": ("pa_prefix_kernel + pa_decode_kernel" if use_prefix else
                                "pa_decode_kernel (4-bit cache)" if int4 else
                                "pa_decode_kernel (8-bit cache)" if fp8 else
                                ("pa_multi_tc_kernel (tcgen05)" if args.q_len * Hq // Hkv > 16 else
                                 "pa_multi_kernel (mma.sync)") if multi else "pa_decode_kernel"),
                     "traffic_source": ("ncu dram bytes of the attention kernel on the first 64 sequences, "
                                        "scaled by algorithmic bytes" if traffic is not None else None),
                     "peak_source": f"{peak_src} hbm_gbs",
                     "algorithmic_bytes_per_launch": ubytes, "avg_launch_ms": round(dec_avg_ms, 5),
                     "kernel_hash": khash},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms / args.steps, 5)},
        "gpu_launches": launches,
        "clocks": clk,
        "host_block_manager_ms": round(st["host_block_manager_ms"], 3),
        "cpu_baseline": cpu,
    }
    if use_prefix:
        cfg_out["prefix_groups"] = st["n_groups"]
    if st["shared"]:
        line["logical_gbs"] = round(world * args.steps * (dbytes + extra) / (max_ms * 1e-3) / 1e9, 2)
    print(json.dumps(line))


def main():
    args = parse_args()
    if args.cpu_worker:
        cpu_worker(args)
    elif args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
