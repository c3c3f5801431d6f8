#!/usr/bin/env python
"""Benchmark: effective KV-read bandwidth of paged fp8 verify attention on GB300.

One step = one call of the whole op (split-KV main kernel + segment reduce)
over one batch.  Default workload: 16 sequences x 35000 keys, q_len 4, 16 query
heads on 1 KV head, head_dim 256, page 16 fp8 e4m3, k/v descales 0.5 / 2.0,
num_segments 16, block tables randomly permuted over a page pool that holds 8
rotating KV replicas (2.29 GB, far above the 129 MB L2), so every timed call
reads its K/V from HBM.

    effective TB/s = sum_b C_b * H_kv * 256 * 2 bytes / time per call

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU runs are independent replicas (the op shards into independent
(sequence, KV head) units with no exchange): value = all ranks' bytes / the
slowest rank's time.  `--impl reference` times the CPU oracle on the host cores
on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import re
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

METRIC = "effective KV-read TB/s and us/call (16x35k, GQA16) vs GB300 HBM peak"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="verify_16x35k_gqa16")
    ap.add_argument("--segments", type=int, default=16)
    ap.add_argument("--replicas", type=int, default=8)
    ap.add_argument("--warm-seconds", type=float, default=1.0,
                    help="keep warming up at least this long (steady clocks and power)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ceiling-gib", type=float, default=4.0)
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip timing the other configurations after the headline one")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip timing the fp8 varlen prefill workload")
    ap.add_argument("--only-prefill", action="store_true",
                    help="time only the fp8 varlen prefill workload (prints its own JSON line)")
    ap.add_argument("--prefill-shape", default=",".join(map(str, PREFILL_SHAPE)),
                    help="batch,seqlen_q,seqlen_k,heads_q,heads_kv of the prefill timing")
    return ap.parse_args()


# --------------------------------------------------------------------------------------------
# CPU oracle timing (the reference arm, and the cpu_baseline of our arm)

def _oracle_worker(job):
    """Build one sequence of the workload on the host and time the oracle on it."""
    import torch
    import oracle
    from paged_fp8_speculative_gb300 import synth
    ctx, ql, hq, hkv, kd, vd, seed = job
    b = synth.make_batch([ctx], [ql], hq, hkv, seed=seed, k_descale=kd, v_descale=vd)
    args = (b.q.view(torch.int16).numpy(), b.k_cache.numpy(), b.v_cache.numpy(),
            b.block_tables.numpy(), b.seq_lens.numpy(), b.cu_seqlens_q.numpy(), b.k_descale,
            b.v_descale, b.softmax_scale, b.num_kv_heads)
    t0 = time.perf_counter()
    oracle.verify_attention_rows(*args)
    return time.perf_counter() - t0, ctx * hkv * 256 * 2


def _oracle_jobs(workload: str, n: int):
    from paged_fp8_speculative_gb300 import synth
    ctx, ql, hq, hkv, kd, vd = synth.workload_spec(workload)
    return [(ctx[i % len(ctx)], ql[i % len(ql)], hq, hkv, kd, vd, 123 + i) for i in range(n)]


class OraclePool:
    """A spawn-started process pool (safe next to CUDA in the parent), one BLAS thread each.

    A step runs one sequence per process concurrently; its time is the slowest
    process's oracle time (input generation excluded)."""

    def __init__(self, procs: int):
        import multiprocessing as mp
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        self.procs = procs
        self.pool = mp.get_context("spawn").Pool(procs)

    def run(self, jobs):
        res = self.pool.map(_oracle_worker, jobs, chunksize=1)
        return max(r[0] for r in res), sum(r[1] for r in res)

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(workload: str) -> dict:
    procs = min(cpu_cores(), 16)
    jobs = _oracle_jobs(workload, procs)
    pool = OraclePool(procs)
    try:
        pool.run(jobs[:1])                           # worker start-up and imports
        dt, kv_bytes = pool.run(jobs)
    finally:
        pool.close()
    return {"value": kv_bytes / dt / 1e12, "unit": "TB/s", "cores": procs, "kind": "oracle",
            "sample": f"{procs} sequence(s) of the {workload} shape, one per process "
                      f"(float64 oracle, slowest process {dt:.2f} s)"}


def run_reference(a) -> None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    procs = min(cpu_cores(), 16)
    jobs = _oracle_jobs(a.workload, procs)
    pool = OraclePool(procs)
    try:
        for _ in range(a.warmup):
            pool.run(jobs)
        runs = [pool.run(jobs) for _ in range(a.steps)]
    finally:
        pool.close()
    total_t = sum(r[0] for r in runs)
    value = sum(r[1] for r in runs) / total_t / 1e12
    line = {"metric": METRIC, "value": value, "unit": "TB/s", "impl": "reference",
            "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": 1e3 * total_t / a.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(a),
            "cpu_baseline": {"value": value, "unit": "TB/s", "cores": procs, "kind": "oracle",
                             "sample": f"each step: {procs} sequence(s) of the {a.workload} "
                                       "shape, one per process"},
            "e2e": {"value": value, "unit": "TB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------------------------
# clocks, peaks, ncu traffic

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid: str | None):
        self.path = tempfile.mktemp(prefix="clk", suffix=".csv")
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if gpu_uuid:
            cmd += ["-i", gpu_uuid]
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 9:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), float(parts[3]),
                             parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [r for r in rows if r[3] >= 50] or rows
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in loaded for n, v in zip(names, r[4]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples_under_load": len(loaded), "samples": len(rows),
                "power_w_max": max(r[2] for r in loaded)}


def bf16_peak() -> tuple[float, str]:
    """Dense bf16 tensor TFLOP/s measured on this machine (burst), else the stated fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def hbm_peak() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# The prefill kernel's translation unit; the verify kernels (main, reduce) build from the rest.
PREFILL_SOURCES = ("fmha_prefill.cu",)


def source_digest(kernel: str = "verify") -> str:
    """Digest of a kernel's sources with comments and blank space removed, so that a profile
    summary stays attached to the code it measured when only comments change.  "verify" covers
    every csrc file but the prefill kernel's own; "prefill" covers that one and the headers
    it includes."""
    h = hashlib.sha256()
    for path in sorted(glob.glob(os.path.join(ROOT, "paged_fp8_speculative_gb300", "csrc", "*"))):
        name = os.path.basename(path)
        if kernel == "verify" and name in PREFILL_SOURCES:
            continue
        if kernel == "prefill" and name not in PREFILL_SOURCES + ("common.cuh", "sm100.cuh"):
            continue
        with open(path, encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)        # block comments
        text = re.sub(r"//[^\n]*", " ", text)                      # line comments
        text = " ".join(text.split())
        h.update(os.path.basename(path).encode() + text.encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str) -> float | None:
    """DRAM bytes per call from the committed ncu summary, if it matches the current sources."""
    for path in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        kv = {}
        for line in open(path):
            if ":" in line and line.lstrip().startswith("- "):
                k, v = line.lstrip()[2:].split(":", 1)
                kv[k.strip()] = v.strip().strip("`")
        if kv.get("workload") == workload and kv.get("source_digest") == source_digest() and \
                "dram_bytes_per_call" in kv:
            return float(kv["dram_bytes_per_call"])
    return None


def workload_config(a) -> dict:
    from paged_fp8_speculative_gb300 import synth
    cfg = {"workload": a.workload}
    shapes = {"verify_16x35k_gqa16": (16, 35000, 4, 16, 1), "verify_16x70k_gqa16": (16, 70000, 4, 16, 1),
              "verify_16x35k_gqa8": (16, 35000, 4, 8, 1), "verify_4x35k_gqa16": (4, 35000, 4, 16, 1)}
    if a.workload in shapes:
        b, c, ql, hq, hkv = shapes[a.workload]
        cfg.update(num_seqs=b, context=c, q_len=ql, num_q_heads=hq, num_kv_heads=hkv)
    cfg.update(head_dim=256, page_size=16, kv="fp8 e4m3", q="bf16", out="bf16",
               num_segments=a.segments if a.segments else "heuristic",
               kv_replicas=a.replicas, l2="inputs larger than L2: rotating KV replicas, "
               "randomly permuted page tables", parallelism=f"replicas x{a.gpus}")
    return cfg


# --------------------------------------------------------------------------------------------
# our arm

def slowest_rank(values, device) -> list:
    """Each rank's timings (ms) reduced to the slowest rank's: the whole job ends when the
    last replica does."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_tbs(kv_bytes_per_rank: int, world: int, steps: int, ms: float) -> float:
    """Whole-job effective KV-read rate: the KV bytes every rank read in `steps` calls,
    over the slowest rank's time."""
    return world * kv_bytes_per_rank * steps / (ms * 1e-3) / 1e12


# Every configuration of the workload list is also timed in the same run, the same way as
# the headline one (cold L2 through rotating KV replicas, CUDA events around back-to-back
# calls after warm-up): name -> (workload, num_segments (0 = the library's heuristic), KV
# replicas, entry point: "exact" mtp_verify_attn_fwd, "qp_fp8" the fp8 Q/P tier).
PER_CONFIG = {
    "verify_16x35k_gqa16": ("verify_16x35k_gqa16", 16, 8, "exact"),
    "verify_16x70k_gqa16": ("verify_16x70k_gqa16", 16, 8, "exact"),
    "verify_16x35k_gqa8": ("verify_16x35k_gqa8", 16, 8, "exact"),
    "verify_4x35k_gqa16": ("verify_4x35k_gqa16", 64, 8, "exact"),
    "draft_extend_8": ("draft_extend_8", 0, 16, "exact"),
    "decode_8": ("decode_8", 0, 16, "exact"),
    "verify_16x35k_gqa16_qp_fp8": ("verify_16x35k_gqa16", 16, 8, "qp_fp8"),
}


def alg_bytes_of(batch) -> int:
    """Algorithmic bytes of one call: K/V, Q and out, and the block-table entries read."""
    total_pages = sum((int(c) + 15) // 16 for c in batch.seq_lens.tolist())
    return batch.kv_bytes() + 2 * batch.q.numel() * 2 + 4 * total_pages * batch.num_kv_heads


def hold_stream(stream, cycles: int = 200_000) -> None:
    """Keep `stream` busy for about 0.1 ms (a spin kernel of `cycles` SM clocks) while the host
    enqueues the first calls of a timed region that starts right after it, so that the device
    timing does not include the host's launch latency of the first call (the GPU would idle
    between the start event and the first kernel otherwise)."""
    import torch
    sleep = getattr(torch.cuda, "_sleep", None)      # PyTorch's spin kernel (private API)
    if sleep is None:
        return
    with torch.cuda.stream(stream):
        sleep(cycles)


def time_calls(call, R: int, warmup: int, steps: int, warm_seconds: float, stream,
               barrier=None) -> float:
    """Milliseconds for `steps` back-to-back calls (CUDA events on the launching stream) after
    `warmup` calls and at least `warm_seconds` of calls; call(i) uses KV replica i % R.
    `barrier` (multi-rank runs) is called between the warm-up and the timed region."""
    import torch
    t_end = time.time() + warm_seconds
    i = 0
    while i < warmup or time.time() < t_end:
        call(i)
        i += 1
        if i % 64 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    if barrier is not None:
        barrier()
        torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_stream(stream)
    t0.record(stream)
    for i in range(steps):
        call(i)
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1)


def per_config_numbers(api, synth, dev, stream, peak, warmup, uuid, names=None) -> dict:
    """us/call, effective TB/s and roofline fraction of every configuration, measured in this
    process on this GPU (each with its own clock record)."""
    import torch
    res = {}
    for name, (wl, S0, R, tier) in PER_CONFIG.items():
        if names is not None and name not in names:
            continue
        fwd = api.mtp_verify_attn_fwd_qp_fp8 if tier == "qp_fp8" else api.mtp_verify_attn_fwd
        b = synth.workload(wl, seed=1, replicas=R, device="cuda")
        tables = [b.block_tables] + b.replica_tables
        # S0 = 0: the library chooses S at every call (and may share the slots out by length)
        S = S0 or api.mtp_verify_attn_num_segments(b.num_seqs, b.num_kv_heads,
                                                   b.block_tables.shape[1])
        kd = torch.tensor([b.k_descale], dtype=torch.float32, device=dev)
        vd = torch.tensor([b.v_descale], dtype=torch.float32, device=dev)
        ws = torch.zeros(api.mtp_verify_attn_workspace_size(b.total_q, b.num_q_heads, S),
                         dtype=torch.uint8, device=dev)
        out = torch.empty_like(b.q)

        def call(i):
            fwd(b.q, b.k_cache, b.v_cache, tables[i % len(tables)], b.seq_lens, b.cu_seqlens_q,
                kd, vd, b.softmax_scale, num_segments=S0, out=out, workspace=ws, stream=stream)

        # a short probe sizes the timed region to about a quarter of a second
        probe = time_calls(call, len(tables), max(3, warmup), 20, 0.0, stream) / 20
        steps = max(200, int(250.0 / max(probe, 1e-3)))
        clocks = ClockSampler(uuid)
        ms = time_calls(call, len(tables), max(3, warmup), steps, 0.3, stream)
        clk = clocks.stop()
        us = 1e3 * ms / steps
        kv = b.kv_bytes()
        res[name] = {"us_per_call": us, "tbs": kv / (us * 1e-6) / 1e12,
                     "frac_of_8tbs_nominal": kv / (us * 1e-6) / 8e12,
                     "roofline_frac": alg_bytes_of(b) / (us * 1e-6) / 1e9 / peak,
                     "num_segments": S, "kv_replicas": R, "kv_bytes": kv, "steps": steps,
                     "entry": "mtp_verify_attn_fwd_qp_fp8" if tier == "qp_fp8" else
                              "mtp_verify_attn_fwd", "clocks": clk}
        del b, tables, ws, out
        torch.cuda.empty_cache()
    return res


# fp8 varlen prefill (the second workload): the page's target shape, batch 1, 12288 queries
# over 14336 keys, 96 query and KV heads, q/k head dim 192, v 128; causal and not.
PREFILL_SHAPE = (1, 12288, 14336, 96, 96)


def prefill_numbers(api, synth, warmup: int, uuid, shape=PREFILL_SHAPE) -> dict:
    """us/call and TFLOP/s of the prefill kernel on `shape` (both products over the visible
    pairs, as the page counts them), against the fp8 tensor peak: twice the measured bf16 rate
    (the nominal fp8/bf16 ratio)."""
    import torch
    B, lq, lk, hq, hkv = shape
    b = synth.make_prefill_batch([lq] * B, [lk] * B, hq, hkv, seed=7, device="cuda")
    out = torch.empty(b.q.shape[0], hq, 128, dtype=torch.bfloat16, device="cuda")
    peak_bf16, kind = bf16_peak()
    res = {"shape": {"batch": B, "seqlen_q": lq, "seqlen_k": lk, "heads_q": hq, "heads_kv": hkv,
                     "head_dim_qk": 192, "head_dim_v": 128, "dtype": "e4m3 q/k/v, bf16 out"},
           "peak_tflops": 2 * peak_bf16, "peak_source": f"2 x {kind} bf16_tflops"}
    for causal in (False, True):
        def call():
            api.fmha_fwd_fp8_varlen(b.q, b.k, b.v, b.q_descale, b.k_descale, b.v_descale,
                                    b.cu_seqlens_q, b.cu_seqlens_k, lq, lk, is_causal=causal,
                                    out=out)
        for _ in range(max(3, warmup // 4)):
            call()
        torch.cuda.synchronize()
        clocks = ClockSampler(uuid)
        n = 10
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_stream(torch.cuda.current_stream())
        e0.record()
        for _ in range(n):
            call()
        e1.record()
        torch.cuda.synchronize()
        clk = clocks.stop()
        us = e0.elapsed_time(e1) * 1e3 / n
        flops = b.flops(causal)
        tf = flops / (us * 1e-6) / 1e12
        res["causal" if causal else "non_causal"] = {
            "us_per_call": us, "tflops": tf, "flops": flops, "frac_of_peak": tf / (2 * peak_bf16),
            "calls": n, "clocks": clk}
    del b, out
    torch.cuda.empty_cache()
    return res


def run_ours(a) -> None:
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    cpu_base = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cpu_base = cpu_baseline(a.workload)      # spawn pool, before any CUDA work

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl")

    from paged_fp8_speculative_gb300 import api, synth

    batch = synth.workload(a.workload, seed=1000 + rank, replicas=a.replicas, device="cuda")
    tables = [batch.block_tables] + batch.replica_tables
    R = len(tables)
    S = a.segments or api.mtp_verify_attn_num_segments(batch.num_seqs, batch.num_kv_heads,
                                                       batch.block_tables.shape[1])
    kd = torch.tensor([batch.k_descale], dtype=torch.float32, device=dev)
    vd = torch.tensor([batch.v_descale], dtype=torch.float32, device=dev)
    ws = torch.zeros(api.mtp_verify_attn_workspace_size(batch.total_q, batch.num_q_heads, S),
                     dtype=torch.uint8, device=dev)
    out = torch.empty_like(batch.q)
    stream = torch.cuda.current_stream()

    def call(i, q=batch.q, bt=None, sl=batch.seq_lens, cu=batch.cu_seqlens_q, o=out):
        api.mtp_verify_attn_fwd(q, batch.k_cache, batch.v_cache, tables[i % R] if bt is None else bt,
                                sl, cu, kd, vd, batch.softmax_scale, num_segments=S, out=o,
                                workspace=ws, stream=stream)

    kv_bytes = batch.kv_bytes()
    alg_bytes = alg_bytes_of(batch)

    # streaming-read ceiling, in the same session
    ceil_buf = torch.empty(int(a.ceiling_gib * (1 << 30)) // 16 * 16, dtype=torch.uint8, device=dev)
    for _ in range(3):
        api.mtpattn_stream_read(ceil_buf, stream=stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(10):
        api.mtpattn_stream_read(ceil_buf, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ceiling_gbs = 10 * ceil_buf.numel() / (e0.elapsed_time(e1) * 1e-3) / 1e9
    del ceil_buf
    torch.cuda.empty_cache()

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)

    # warm-up: W calls and at least `warm_seconds` of calls, a barrier across ranks, then the
    # timed region (every rank's events bracket its own calls)
    ms = time_calls(call, R, a.warmup, a.steps, a.warm_seconds, stream,
                    barrier=dist.barrier if world > 1 else None)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    # End to end through the public API: every step uploads its inputs from pinned host memory
    # and downloads its output.  Run the way a decode loop runs it, as CUDA graphs captured from
    # the public call: a step computes while, on a branch of its own, it uploads the next step's
    # inputs into the other of two buffer sets and downloads the previous step's output from
    # there.  The last step's output is downloaded after the loop, inside the timed region.
    pin = lambda t: t.cpu().pin_memory()
    h_q, h_sl, h_cu = pin(batch.q), pin(batch.seq_lens), pin(batch.cu_seqlens_q)
    h_bt = [pin(t) for t in tables]
    h_out = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    sets = [dict(q=torch.empty_like(batch.q), sl=torch.empty_like(batch.seq_lens),
                 cu=torch.empty_like(batch.cu_seqlens_q), bt=torch.empty_like(tables[0]),
                 o=torch.empty_like(out)) for _ in range(2)]
    h2d = h_q.numel() * 2 + h_sl.numel() * 4 + h_cu.numel() * 4 + h_bt[0].numel() * 4
    d2h = h_out[0].numel() * 2

    def upload(i, d):
        d["q"].copy_(h_q, non_blocking=True)
        d["bt"].copy_(h_bt[i % R], non_blocking=True)
        d["sl"].copy_(h_sl, non_blocking=True)
        d["cu"].copy_(h_cu, non_blocking=True)

    G = R if R % 2 == 0 else 2 * R              # steps i and i + G use the same buffers and table
    cap, side = torch.cuda.Stream(), torch.cuda.Stream()

    def capture_step(g):
        d, dn = sets[g % 2], sets[(g + 1) % 2]
        fork = torch.cuda.Event()
        fork.record(cap)
        side.wait_event(fork)
        with torch.cuda.stream(side):              # next step's inputs up, previous output down
            upload(g + 1, dn)
            h_out[(g + 1) % 2].copy_(dn["o"], non_blocking=True)
            join = torch.cuda.Event()
            join.record(side)
        api.mtp_verify_attn_fwd(d["q"], batch.k_cache, batch.v_cache, d["bt"], d["sl"], d["cu"],
                                kd, vd, batch.softmax_scale, num_segments=S, out=d["o"],
                                workspace=ws, stream=cap)
        cap.wait_event(join)

    # One graph per step (for a remainder), and one graph of G consecutive steps, inside which
    # a step's kernels can start while the previous step's finish (programmatic launch).
    singles = []
    for g in range(G):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=cap):
            capture_step(g)
        singles.append(gr)
    block = torch.cuda.CUDAGraph()
    with torch.cuda.graph(block, stream=cap):
        for g in range(G):
            capture_step(g)
    torch.cuda.synchronize()

    def run_steps(n):
        for _ in range(n // G):
            block.replay()
        for i in range(n - n % G, n):
            singles[i % G].replay()

    with torch.cuda.stream(cap):
        upload(0, sets[0])
        run_steps(max(G, a.warmup // 4))
        cap.synchronize()
        upload(0, sets[0])                         # the first step's inputs, then the timed steps
        cap.synchronize()
        if world > 1:
            dist.barrier()
        hold_stream(cap)
        t0.record(cap)
        run_steps(a.steps)
        last = (a.steps - 1) % 2
        h_out[last].copy_(sets[last]["o"], non_blocking=True)
        t1.record(cap)
    torch.cuda.synchronize()
    ms_e2e = t0.elapsed_time(t1)
    # The last step's downloaded output against the device loop's last call (same inputs):
    # equal up to the float32 re-association of balanced tile sharing.
    got, ref = h_out[(a.steps - 1) % 2].float(), out.cpu().float()
    diff, scale = (got - ref).abs().max().item(), ref.abs().max().item()
    if diff > 2 ** -7 * scale:
        raise RuntimeError(f"end-to-end output differs from the device loop's: {diff} (scale {scale})")

    # Host time of one eager call through the public API (argument checks, pointer checks of
    # the C entry, tensor-map cache, two launches), the GPU kept busy so no call waits.
    torch.cuda.synchronize()
    n_host = 200
    h0 = time.perf_counter()
    for i in range(n_host):
        call(i)
    host_us = (time.perf_counter() - h0) / n_host * 1e6
    torch.cuda.synchronize()

    if world > 1:
        ms, ms_e2e = slowest_rank([ms, ms_e2e], dev)
        dist.destroy_process_group()
    if rank != 0:
        return
    peak, peak_kind = hbm_peak()
    per_config = None
    if world == 1 and not a.no_per_config:
        del sets, h_q, h_bt, h_out
        torch.cuda.empty_cache()
        per_config = per_config_numbers(api, synth, dev, stream, peak, a.warmup, uuid)
    prefill = None
    if world == 1 and not a.no_prefill:
        prefill = prefill_numbers(api, synth, a.warmup, uuid,
                                  tuple(int(x) for x in a.prefill_shape.split(",")))

    us_call = 1e3 * ms / a.steps
    value = job_tbs(kv_bytes, world, a.steps, ms)
    achieved = alg_bytes / (us_call * 1e-6) / 1e9
    traffic = ncu_traffic(a.workload)
    line = {
        "metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": ms / a.steps, "us_per_call": us_call,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic",
        "config": workload_config(a) | {"num_segments": S},
        # how this implementation cut the work (not part of the workload, so not in config)
        "scheduling": ("planned" if api.mtp_verify_attn_get_scheduling() == api.SCHED_PLANNED
                       else "chunked"),
        "timing": "CUDA events on the launching stream around exactly `steps` calls; a 0.1 ms "
                  "spin kernel ahead of the start event keeps the host's launch latency of the "
                  "first call out of the device time",
        "frac_of_8tbs_nominal": value / world / 8.0,
        "read_ceiling": {"value_gbs": ceiling_gbs, "frac": value / world * 1e3 / ceiling_gbs,
                         "kernel": "mtpattn_stream_read, 16-B loads"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "mtp_verify_attn_fwd (main + reduce)",
                     "peak_source": f"{peak_kind} hbm_gbs", "alg_bytes_per_call": alg_bytes},
        "cpu_baseline": cpu_base,
        "e2e": {"value": job_tbs(kv_bytes, world, a.steps, ms_e2e), "unit": "TB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "us_per_step": 1e3 * ms_e2e / a.steps,
                "pipelining": "CUDA graphs of consecutive steps captured from the public call; each "
                              "step's inputs go up and its output comes down beside the neighbouring "
                              "steps' compute"},
        "gpu_launches": 2 * a.steps,
        # host cost of one eager call (python wrapper + C entry + launches; not in `value`)
        "host_us_per_eager_call": host_us,
        "clocks": clk,
        # every configuration, each timed like the headline one in this run (not part of value)
        "per_config": per_config,
        # the second workload, fp8 varlen prefill attention (tensor-bound; not part of value)
        "prefill": prefill,
    }
    print(json.dumps(line), flush=True)


def run_prefill_only(a) -> None:
    import torch
    from paged_fp8_speculative_gb300 import api, synth
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    shape = tuple(int(x) for x in a.prefill_shape.split(","))
    res = prefill_numbers(api, synth, a.warmup, None, shape)
    print(json.dumps({"workload": "fmha_fwd_fp8_varlen", "prefill": res}), flush=True)


def main():
    a = parse_args()
    if a.impl == "reference":
        run_reference(a)
    elif a.only_prefill:
        run_prefill_only(a)
    else:
        run_ours(a)


if __name__ == "__main__":
    main()
