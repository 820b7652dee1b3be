#!/usr/bin/env python
"""Benchmark of the MSA hot path on GB300; prints ONE JSON line on rank 0.

Headline: MSA decode at the agentic shape (8 requests x 60,000 cached tokens,
Hq=64, G=8, D=128, Di=64, top-16 blocks of 128 tokens): one step = index scoring
-> top-k -> page tables -> paged sparse attention for the whole batch.  The
prefill chunk (8,192 new rows on a 60,000-token prefix) is timed the same way and
reported in the "prefill" object of the same line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl msa|reference]

With N > 1 (torchrun, one rank per GPU) every rank runs its own batch: weak
scaling, no collective on the data path; the time is the max over ranks.
--impl reference times the fp64 CPU oracle on the same workload and metric.
"""
from __future__ import annotations

import argparse
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

METRIC = "MSA decode tok/s & prefill q-tok/s at 60k ctx; % of HBM / tensor-core roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PROFILES = os.path.join(ROOT, "profiles")
CSRC = os.path.join(ROOT, "block_sparse_attention_06_gb300", "csrc")
SWEEP = ("decode1m", "ragged1", "ragged8", "ragged32", "ragged64")
L2_FLUSH_BYTES = 256 << 20   # read between timed steps of the small workloads (L2 is 129 MB)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["msa", "reference"], default="msa")
    ap.add_argument("--only", choices=["all", "decode", "prefill"], default="all",
                    help="time one workload alone (profiling); the JSON line then omits the other")
    ap.add_argument("--prefill-prefix", type=int, default=60000, help="cached tokens before the prefill chunk")
    ap.add_argument("--prefill-chunk", type=int, default=8192, help="new query rows in the prefill chunk")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing (profiling runs)")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the decode1m and ragged-batch decode objects (profiling runs)")
    return ap.parse_args()


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a per-rank scalar over all ranks (the job's wall time is the slowest rank's)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return units_per_rank * world / max_seconds


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="msa_clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "-i", str(self.idx),
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def ncu_traffic(kernel: str):
    """DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of `kernel` on its bench
    workload, from the machine-readable line of its ncu summary under profiles/:

        <!-- traffic kernel=NAME source=FILE.cu sha256_16=HEX dram_bytes_per_launch=N -->

    Reported only while the kernel's source is the one that was profiled (same sha256 prefix);
    otherwise (traffic None, "stale ...") so that a changed kernel never carries old counters."""
    import hashlib
    import re
    pat = re.compile(r"<!-- traffic kernel=(\S+) source=(\S+) sha256_16=([0-9a-f]{16}) dram_bytes_per_launch=(\d+) -->")
    for name in sorted(os.listdir(PROFILES)) if os.path.isdir(PROFILES) else []:
        with open(os.path.join(PROFILES, name)) as fh:
            for m in pat.finditer(fh.read()):
                if m.group(1) != kernel:
                    continue
                with open(os.path.join(CSRC, m.group(2)), "rb") as src:
                    now = hashlib.sha256(src.read()).hexdigest()[:16]
                if now != m.group(3):
                    return None, f"stale: profiles/{name} profiled {m.group(2)} at {m.group(3)}, source is now {now}"
                return int(m.group(4)), f"profiles/{name}"
    return None, "no ncu capture of this kernel"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ GPU arm

def decode_bytes(case) -> int:
    """Algorithmic bytes of one decode step's index scan: every cached token's
    index key of every group is read once (L * G * Di * 2 per request)."""
    d = case.dims
    return int(sum(int(L) for L in case.seq_lens.tolist()) * d.G * d.Di * 2)


def prefill_scoring_flops(case) -> float:
    """Algorithmic flops of prefill index scoring: 2 * Di per (row, group, causally visible token)."""
    d = case.dims
    return float((case.q_pos.long() + 1).sum().item()) * d.G * 2 * d.Di


def prefill_attention_flops(step, case) -> float:
    """Algorithmic flops of block-major attention: 4 * D per (query head, attended token)."""
    import torch
    d = case.dims
    sel = step.sel.long()
    pos = case.q_pos.long()[:, None, None]
    vis = (pos - sel * 128 + 1).clamp(min=0, max=128)
    vis = torch.where(sel >= 0, vis, torch.zeros_like(vis))
    hpg = d.Hq // d.G
    return float(vis.sum().item()) * hpg * 4 * d.D


def run_msa(args, rank, world, local):
    import torch
    import block_sparse_attention_06_gb300 as msa
    import msa_inputs as mi

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    peaks, peak_src = load_peaks()
    K, W = args.steps, args.warmup

    line = {}
    clocks = ClockSampler(local).start()
    case = None
    if args.only in ("all", "decode"):
        dec, case = bench_decode(args, rank, world, local, dev, peaks, peak_src)
        line.update(dec)
        line["decode_multi"] = bench_decode_multi(args, world, dev, peaks, peak_src)
        if not args.no_sweep:
            line["decode_sweep"] = {name: bench_decode_sweep(name, args, world, dev, peaks, peak_src)
                                    for name in SWEEP}
    if args.only in ("all", "prefill"):
        line["prefill"] = bench_prefill(args, world, dev, peaks, peak_src, rank)
    if args.only == "all" and not args.no_sweep:
        line["mixed"] = bench_mixed(args, world, dev)
    line["clocks"] = clocks.stop()
    if case is not None:
        line["cpu_baseline"] = (cpu_baseline_decode(rank, case=case)
                                if rank == 0 and not args.no_cpu_baseline else None)
    if args.only == "prefill":
        pre = line["prefill"]
        line = {"metric": METRIC, "value": pre["value"], "unit": pre["unit"], "n_gpus": world, "steps": K,
                "warmup": W, "ms_per_step": pre["ms_per_step"], "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16)",
                "config": pre["config"], "gpu_launches": pre["gpu_launches"], "roofline": pre["roofline"],
                "clocks": line["clocks"], "cpu_baseline": pre.get("cpu_baseline")}
    if rank == 0:
        print(json.dumps(line), flush=True)


def bench_decode(args, rank, world, local, dev, peaks, peak_src):
    import torch
    import block_sparse_attention_06_gb300 as msa
    import msa_inputs as mi
    K, W = args.steps, args.warmup
    case = mi.named_case("decode60k", device=dev)
    dims = msa.dims_of(case)
    B = case.n_rows
    step = msa.DecodeStep(dims, B, case.n_req, case.n_pages, dev)
    call = lambda: step(case.q, case.q_idx, case.k_cache, case.v_cache, case.kidx_cache, case.block_table,
                        case.seq_lens, case.q_pos)
    def timed_loop(fn):
        for _ in range(W):
            fn()
        msa.msa_check(step.err)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        t0.record()
        for k in range(K):
            fn()
        t1.record()
        torch.cuda.synchronize()
        barrier(world)
        msa.msa_check(step.err)
        return max_over_ranks(t0.elapsed_time(t1), world, dev)

    # the step as a serving engine runs it, replayed from a CUDA graph; and launched kernel by kernel
    step.capture(case.q, case.q_idx, case.k_cache, case.v_cache, case.kidx_cache, case.block_table, case.seq_lens)
    dec_ms = timed_loop(step.replay)
    stream_ms = timed_loop(call)

    # ---------------- the dominant kernel alone (index scan), same stream and inputs,
    # one CUDA-event pair per launch: its duration gives the roofline line
    s1_b = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    s1_e = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    torch.cuda.synchronize()
    for k in range(K):
        s1_b[k].record()
        step.scores_only(case.q_idx, case.kidx_cache, case.block_table, case.q_pos)
        s1_e[k].record()
    torch.cuda.synchronize()
    s1_ms = statistics.mean(s1_b[k].elapsed_time(s1_e[k]) for k in range(K))
    msa.msa_check(step.err)
    value = aggregate_throughput(B * K, world, dec_ms / 1e3)
    tr, tr_src = ncu_traffic("k_score_decode")
    s1_bytes = decode_bytes(case)
    s1_gbs = s1_bytes / (s1_ms / 1e3) / 1e9

    # ---------------- e2e through the public API: pinned host inputs in, result out.
    # The step's inputs sit packed in one page-locked buffer (msa.DecodeInputs) and go up
    # by one staging kernel (msa_stage_from_host); the attention kernel writes out and lse
    # straight into a page-locked host buffer.
    inputs = msa.DecodeInputs(dims, B, dev)
    for n in ("q", "q_idx", "q_pos", "seq_lens", "block_table"):
        getattr(inputs, "h_" + n).copy_(getattr(case, n).cpu())
    host_res, _ = step.host_results()
    h2d = inputs.nbytes
    d2h = host_res.numel()

    e2e_graph = msa.DecodeStep(dims, B, case.n_req, case.n_pages, dev)
    e2e_graph.capture(inputs.q, inputs.q_idx, case.k_cache, case.v_cache, case.kidx_cache, inputs.block_table,
                      inputs.seq_lens, inputs=inputs, host_results=host_res)

    def e2e_step():   # one replay = upload of the step's inputs, the step, out and lse into host memory
        e2e_graph.replay()

    for _ in range(W):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        e2e_step()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    msa.msa_check(e2e_graph.err)
    e2e_value = aggregate_throughput(B * K, world, e2e_ms / 1e3)

    return {
        "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": dec_ms / K, "ms_per_step_stream_launched": stream_ms / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16, planted needle blocks)",
        "config": {"workload": "decode60k", "batch": B, "ctx": 60000, "Hq": dims.Hq, "G": dims.G, "D": dims.D,
                   "Di": dims.Di, "topk": dims.topk, "page": 128, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (491.5 MB k-index scan per step)",
                   "launch": "msa_decode_step replayed from a CUDA graph (ms_per_step_stream_launched: the "
                             "same step launched kernel by kernel); steps back to back, mean"},
        "gpu_launches": step.kernel_launches * K,
        "roofline": {"bound": "hbm", "kernel": "k_score_decode", "achieved": s1_gbs, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": s1_gbs / peaks["hbm_gbs"], "traffic": tr, "traffic_source": tr_src,
                     "bytes_per_launch": s1_bytes, "ms_per_launch": s1_ms,
                     "peak_source": f"{peak_src} hbm_gbs"},
        "e2e": {"value": e2e_value, "unit": "tok/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms / K},
    }, case


def bench_decode_sweep(name, args, world, dev, peaks, peak_src):
    """One decode workload besides the headline: decode1m (2 requests x 1,048,576 tokens) or a ragged
    batch (1, 8, 32 or 64 requests of 4k-128k tokens).  Each timed step is one msa_decode_step replayed
    from a CUDA graph, with its own CUDA-event pair; a 256 MB buffer is read between steps so that no
    step finds the previous step's pages in L2 (a one-request batch reads less than L2 holds) -- read,
    not written, so that no dirty lines are written back during the next step; the median is reported.
    Roofline: the step's algorithmic bytes -- every cached index key once plus the selected K and V
    (row_len tokens of D bf16 each, per (request, group) row) -- over the median step time, against
    the measured copy bandwidth."""
    import torch
    import block_sparse_attention_06_gb300 as msa
    import msa_inputs as mi
    K, W = args.steps, args.warmup
    case = mi.named_case(name, device=dev)
    dims = msa.dims_of(case)
    B = case.n_rows
    step = msa.DecodeStep(dims, B, case.n_req, case.n_pages, dev)
    step.capture(case.q, case.q_idx, case.k_cache, case.v_cache, case.kidx_cache, case.block_table,
                 case.seq_lens)
    call = step.replay
    flush = torch.ones(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(W):
        call()
    msa.msa_check(step.err)
    torch.cuda.synchronize()
    barrier(world)
    b_ev = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    e_ev = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for k in range(K):
        flush.sum(dtype=torch.int32)   # evicts the previous step's lines from L2
        b_ev[k].record()
        call()
        e_ev[k].record()
    torch.cuda.synchronize()
    barrier(world)
    msa.msa_check(step.err)
    ms = statistics.median(b_ev[k].elapsed_time(e_ev[k]) for k in range(K))
    ms = max_over_ranks(ms, world, dev)
    scan = decode_bytes(case)
    kv = int(step.row_len.long().sum().item()) * dims.D * 2 * 2
    gbs = (scan + kv) / (ms / 1e3) / 1e9
    lens = case.seq_lens.tolist()
    out = {
        "metric": "MSA decode tok/s", "value": aggregate_throughput(B, world, ms / 1e3), "unit": "tok/s",
        "ms_per_step": ms, "steps": K,
        "config": {"workload": name, "batch": B, "ctx_min": int(min(lens)), "ctx_max": int(max(lens)),
                   "ctx_total": int(sum(lens)), "Hq": dims.Hq, "G": dims.G, "D": dims.D, "Di": dims.Di,
                   "topk": dims.topk, "l2": f"{L2_FLUSH_BYTES >> 20} MB read between timed steps",
                   "timing": "median of per-step CUDA-event times, the step replayed from a CUDA graph"},
        "gpu_launches": step.kernel_launches * K,
        "roofline": {"bound": "hbm", "kernel": "msa_decode_step (index scan, select, attention)",
                     "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                     "traffic": None, "traffic_source": "no ncu capture of this workload",
                     "bytes_per_step": scan + kv, "index_bytes": scan, "kv_bytes": kv,
                     "peak_source": f"{peak_src} hbm_gbs"},
    }
    del case, step, flush
    torch.cuda.empty_cache()
    return out


def bench_mixed(args, world, dev):
    """A chunked-prefill engine step: decode60k's batch (8 decode requests x 60,000 tokens) and
    prefill68k's chunk (8,192 rows on a 60,000-token prefix) in ONE step over one page pool
    (MixedStep).  Timed serially on one stream and with the decode half on a side stream; each
    timed step has its own CUDA-event pair on the caller's stream (which joins the side stream
    before the end event).  Reported: rows per second of the whole step (decode tokens plus
    prefill rows), and both timings next to the two halves timed alone."""
    import torch
    import block_sparse_attention_06_gb300 as msa
    import msa_inputs as mi
    K, W = args.steps, args.warmup
    dec, pre = mi.named_case("mixed", device=dev)
    dims = msa.dims_of(dec)
    margs = (dec.k_cache, dec.v_cache, dec.kidx_cache, dec.q, dec.q_idx, dec.block_table, dec.seq_lens, pre.q,
             pre.q_idx, pre.block_table, pre.q_req, pre.q_pos)

    def timed(fn, errs):
        for _ in range(W):
            fn()
        for e in errs:
            msa.msa_check(e)
        torch.cuda.synchronize()
        barrier(world)
        b_ev = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        e_ev = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        for k in range(K):
            b_ev[k].record()
            fn()
            e_ev[k].record()
        torch.cuda.synchronize()
        barrier(world)
        for e in errs:
            msa.msa_check(e)
        return max_over_ranks(statistics.median(b_ev[k].elapsed_time(e_ev[k]) for k in range(K)), world, dev)

    res = {}
    for overlap in (False, True):
        ms = msa.MixedStep(dims, dec.n_rows, pre.n_rows, pre.n_req, dec.n_pages, dev, overlap=overlap)
        res[overlap] = timed(lambda: ms(*margs), ms.err_words)
    d_only = timed(lambda: ms.decode(dec.q, dec.q_idx, dec.k_cache, dec.v_cache, dec.kidx_cache, dec.block_table,
                                     dec.seq_lens), [ms.decode.err])
    p_only = timed(lambda: ms.prefill(pre.q, pre.q_idx, pre.k_cache, pre.v_cache, pre.kidx_cache, pre.block_table,
                                      pre.q_req, pre.q_pos), [ms.prefill.err])
    rows = dec.n_rows + pre.n_rows
    best = min(res.values())
    out = {
        "metric": "MSA mixed step rows/s (decode tokens + prefill rows)",
        "value": aggregate_throughput(rows, world, best / 1e3), "unit": "rows/s",
        "ms_per_step": best, "ms_per_step_serial": res[False], "ms_per_step_overlapped": res[True],
        "ms_decode_half_alone": d_only, "ms_prefill_half_alone": p_only,
        "config": {"workload": "mixed: decode60k batch + prefill68k chunk over one pool", "decode_requests": dec.n_rows,
                   "prefill_rows": pre.n_rows, "Hq": dims.Hq, "G": dims.G, "D": dims.D, "Di": dims.Di,
                   "topk": dims.topk, "timing": "median of per-step CUDA-event times on the caller's stream"},
        "gpu_launches": ms.kernel_launches * K,
    }
    del dec, pre, ms
    torch.cuda.empty_cache()
    return out


def bench_decode_multi(args, world, dev, peaks, peak_src, T=8):
    """Multi-token (speculative) decode scoring: decode60k's 8 requests with T query rows each.  The
    MSA_PHASE_DECODE_MULTI scan reads each request's k-index once for all its rows; the row-wise scan
    (MSA_PHASE_DECODE) on the same rows reads it T times.  Reported: scored rows per second of the
    multi-token scan and its HBM roofline against the k-index bytes read once per request."""
    import torch
    import block_sparse_attention_06_gb300 as msa
    import msa_inputs as mi
    K, W = args.steps, args.warmup
    case = mi.multi_token_decode_case([60000] * 8, T, Hq=64, G=8, D=128, Di=64, topk=16, pool_pages=4096,
                                      seed=1001, device=dev)
    dims = msa.dims_of(case)
    err = msa.new_err_word(dev)
    sc = torch.empty((case.n_rows, dims.G, dims.max_blocks), dtype=torch.float32, device=dev)

    def timed(phase):
        f = lambda: msa.msa_index_score(case.q_idx, case.kidx_cache, case.block_table, case.q_req, case.q_pos,
                                        dims, phase, scores=sc, err_word=err)
        for _ in range(W):
            f()
        torch.cuda.synchronize()
        barrier(world)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(K):
            f()
        b.record()
        torch.cuda.synchronize()
        barrier(world)
        msa.msa_check(err)
        return max_over_ranks(a.elapsed_time(b), world, dev) / K

    multi_ms = timed(msa.MSA_PHASE_DECODE_MULTI)
    tr, tr_src = ncu_traffic("k_score_decode_mt")
    row_ms = timed(msa.MSA_PHASE_DECODE)
    kbytes = sum(int(L) for L in case.seq_lens.tolist()) * dims.G * dims.Di * 2
    gbs = kbytes / (multi_ms / 1e3) / 1e9
    return {
        "metric": "multi-token decode scoring rows/s", "value": aggregate_throughput(case.n_rows, world, multi_ms / 1e3),
        "unit": "rows/s", "ms_per_launch": multi_ms, "rowwise_ms_per_launch": row_ms,
        "config": {"workload": f"decode60k with {T} query rows per request", "batch": 8, "rows": case.n_rows,
                   "ctx": 60000, "G": dims.G, "Di": dims.Di},
        "roofline": {"bound": "hbm", "kernel": "k_score_decode_mt", "achieved": gbs, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"], "traffic": tr, "traffic_source": tr_src,
                     "bytes_per_launch": kbytes,
                     "peak_source": f"{peak_src} hbm_gbs"},
    }


def bench_prefill(args, world, dev, peaks, peak_src, rank=0):
    import torch
    import block_sparse_attention_06_gb300 as msa
    import msa_inputs as mi
    K, W = args.steps, args.warmup
    if (args.prefill_prefix, args.prefill_chunk) == (60000, 8192):
        pc = mi.named_case("prefill68k", device=dev)
    else:
        pc = mi.prefill_case(args.prefill_prefix, args.prefill_chunk, Hq=64, G=8, D=128, Di=64, topk=16,
                             pool_pages=(args.prefill_prefix + args.prefill_chunk) // 128 + 64, seed=1002,
                             device=dev)
    pd = msa.dims_of(pc)
    ps = msa.PrefillStep(pd, pc.n_rows, pc.n_req, dev)
    pcall = lambda: ps(pc.q, pc.q_idx, pc.k_cache, pc.v_cache, pc.kidx_cache, pc.block_table, pc.q_req,
                       pc.q_pos)
    for _ in range(W):
        pcall()
    msa.msa_check(ps.err)
    torch.cuda.synchronize()
    ev = lambda: [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    sel_ev, a_b, a_e, m_e = ev(), ev(), ev(), ev()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    p0.record()
    for k in range(K):
        sel_ev[k].record()
        ps.select(pc.q_idx, pc.kidx_cache, pc.block_table, pc.q_req, pc.q_pos)
        a_b[k].record()
        msa.msa_sparse_attn_prefill(pc.q, pc.k_cache, pc.v_cache, pc.block_table, pc.q_req, pc.q_pos,
                                    ps.blk_off, ps.blk_ent, pd, ps.o_part, ps.lse_part, ps.attn_ws, err_word=ps.err)
        a_e[k].record()
        msa.msa_lse_merge(ps.o_part, ps.lse_part, ps.sel, ps.ent_pos, pd, ps.out, ps.lse, err_word=ps.err)
        m_e[k].record()
    p1.record()
    torch.cuda.synchronize()
    barrier(world)
    pre_ms = max_over_ranks(p0.elapsed_time(p1), world, dev)
    attn_ms = statistics.mean(a_b[k].elapsed_time(a_e[k]) for k in range(K))
    sel_ms = statistics.mean(sel_ev[k].elapsed_time(a_b[k]) for k in range(K))
    merge_ms = statistics.mean(a_e[k].elapsed_time(m_e[k]) for k in range(K))
    sflops = prefill_scoring_flops(pc)
    tr, tr_src = ncu_traffic("k_attn_prefill")
    msa.msa_check(ps.err)
    flops = prefill_attention_flops(ps, pc)
    tflops = flops / (attn_ms / 1e3) / 1e12
    prefill = {
        "metric": "MSA prefill q-tok/s", "value": aggregate_throughput(pc.n_rows * K, world, pre_ms / 1e3),
        "unit": "q-tok/s", "ms_per_step": pre_ms / K, "steps": K,
        "config": {"workload": "prefill68k" if pc.name == "prefill68k" else "prefill",
                   "prefix": args.prefill_prefix, "chunk": pc.n_rows, "Hq": pd.Hq, "G": pd.G,
                   "D": pd.D, "Di": pd.Di, "topk": pd.topk,
                   "l2": "working set larger than L2 (about 2.1 GB of partials written and read per step)"},
        "gpu_launches": ps.kernel_launches * K,
        "roofline": {"bound": "tensor", "kernel": "k_attn_prefill", "achieved": tflops,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": tflops / peaks["bf16_tflops"], "traffic": tr, "traffic_source": tr_src,
                     "flops_per_launch": flops, "ms_per_launch": attn_ms,
                     "peak_source": f"{peak_src} bf16_tflops (burst)"},
        "select": {"call": "msa_select_invert_prefill (tensor-core scoring with the top-k fused, list merge, "
                           "inversion)" if ps.fuse_topk else "msa_index_score + msa_topk_blocks + msa_invert_selection",
                   "ms_per_launch": sel_ms, "scoring_flops_per_launch": sflops,
                   "scoring_tflops": sflops / (sel_ms / 1e3) / 1e12,
                   "frac_of_bf16_peak": sflops / (sel_ms / 1e3) / 1e12 / peaks["bf16_tflops"]},
        "merge": {"kernel": "k_lse_merge", "ms_per_launch": merge_ms},
        "timing": "CUDA events on the stream around each call, mean over the timed steps",
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        prefill["cpu_baseline"] = cpu_baseline_prefill(pc)
    return prefill


# ------------------------------------------------------------------ oracle legs (CPU)

def _oracle_decode_one(case, b):
    """The fp64 oracle's decode of request b (scores, top-k, page table, attention),
    on host copies of just the pages it reads.  Returns the oracle's CPU seconds."""
    import torch
    import oracle
    bt = case.block_table[b:b + 1].cpu()
    pages = bt[bt >= 0].long()
    kidx = case.kidx_cache[pages.to(case.kidx_cache.device)].cpu()
    bt_c = torch.full_like(bt, -1)
    bt_c[bt >= 0] = torch.arange(len(pages), dtype=torch.int32)
    q_pos = case.q_pos[b:b + 1].cpu()
    local = torch.zeros(1, dtype=torch.int32)
    t = time.perf_counter()
    sc = oracle.block_scores(case.q_idx[b:b + 1].cpu(), kidx, bt_c, local, q_pos, case.max_blocks)
    sel = oracle.topk(sc, q_pos, case.dims.topk)
    t_sel = time.perf_counter() - t
    used = sorted({int(bt[0, j]) for j in sel.flatten().tolist() if j >= 0})
    remap = {p: i for i, p in enumerate(used)}
    kc = case.k_cache[torch.tensor(used, device=case.k_cache.device)].cpu()
    vc = case.v_cache[torch.tensor(used, device=case.v_cache.device)].cpu()
    bt_a = torch.tensor([[remap.get(int(p), 0) for p in bt[0].tolist()]], dtype=torch.int32)
    t = time.perf_counter()
    pt, rl = oracle.page_table(sel, bt_a, q_pos + 1)
    oracle.paged_attention(case.q[b:b + 1].cpu(), kc, vc, pt, rl, case.dims.sm_scale)
    return t_sel + time.perf_counter() - t


def cpu_baseline_prefill(pc, budget_s: float = 10.0, max_rows: int = 2048):
    """The fp64 oracle's prefill of single rows of the chunk -- scores against the row's
    candidate blocks, top-k, attention over the selected tokens -- on host copies of the
    chunk's pages, over rows spread through the chunk, until budget_s of CPU time."""
    import torch
    import oracle
    bt = pc.block_table.cpu()
    pages = torch.unique(bt[bt >= 0]).long()
    local = torch.full((int(pages.max()) + 1,), -1, dtype=torch.int32)
    local[pages] = torch.arange(len(pages), dtype=torch.int32)
    bt_l = torch.where(bt >= 0, local[bt.clamp(min=0).long()], torch.full_like(bt, -1))
    dev_pages = pages.to(pc.kidx_cache.device)
    kidx, kc, vc = pc.kidx_cache[dev_pages].cpu(), pc.k_cache[dev_pages].cpu(), pc.v_cache[dev_pages].cpu()
    q_idx, q, q_pos, q_req = pc.q_idx.cpu(), pc.q.cpu(), pc.q_pos.cpu(), pc.q_req.cpu()
    zero = torch.zeros(1, dtype=torch.int32)
    spent, done = 0.0, 0
    for i in range(max_rows):
        r = (i * 2654435761) % pc.n_rows      # rows spread over the chunk, every row position alike
        b = int(q_req[r])
        t = time.perf_counter()
        sc = oracle.block_scores(q_idx[r:r + 1], kidx, bt_l[b:b + 1], zero, q_pos[r:r + 1], pc.max_blocks)
        sel = oracle.topk(sc, q_pos[r:r + 1], pc.dims.topk)
        oracle.attention(q[r:r + 1], kc, vc, bt_l[b:b + 1], zero, q_pos[r:r + 1], sel, pc.dims.sm_scale)
        spent += time.perf_counter() - t
        done += 1
        if spent >= budget_s:
            break
    return {"value": done / spent, "unit": "q-tok/s", "cores": 1, "kind": "oracle", "host_cores": os.cpu_count(),
            "sample": f"{done} rows spread over the {pc.n_rows}-row chunk, each scored against its candidate "
                      f"blocks, selected and attended by the single-threaded fp64 C oracle, {spent:.1f} s of "
                      f"CPU time"}


def cpu_baseline_decode(rank: int, budget_s: float = 12.0, max_reqs: int = 1000, case=None):
    import torch
    import msa_inputs as mi
    if case is None:
        dev = "cuda:0" if torch.cuda.is_available() else "cpu"
        case = mi.named_case("decode60k", device=dev)
    spent, n = 0.0, 0
    while spent < budget_s and n < max_reqs:
        spent += _oracle_decode_one(case, n % case.n_rows)
        n += 1
    return {"value": n / spent, "unit": "tok/s", "cores": 1, "kind": "oracle",
            "host_cores": os.cpu_count(),
            "sample": f"{n} decode requests of the decode60k workload (60,000 cached tokens each), "
                      f"single-threaded fp64 C oracle, {spent:.1f} s of CPU time"}


def run_reference(args, rank, world):
    """The oracle as the reference arm: rank 0 only, a bounded sample per step."""
    if rank != 0:
        return
    import torch
    import msa_inputs as mi
    dev = "cuda:0" if torch.cuda.is_available() else "cpu"
    case = mi.named_case("decode60k", device=dev)
    for i in range(args.warmup):
        _oracle_decode_one(case, i % case.n_rows)
    spent = 0.0
    for k in range(args.steps):
        spent += _oracle_decode_one(case, k % case.n_rows)
    value = args.steps / spent
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": spent / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16, planted needle blocks)",
        "config": {"workload": "decode60k", "batch": case.n_rows, "ctx": 60000, "Hq": 64, "G": 8, "D": 128,
                   "Di": 64, "topk": 16, "page": 128, "parallelism": "single host thread"},
        "cpu_baseline": {"value": value, "unit": "tok/s", "kind": "oracle", "cores": 1,
                         "sample": "each step = the full decode of one request of decode60k "
                                   "(60,000-token index scan, top-16, attention over 2,016 tokens), "
                                   "single-threaded fp64 C oracle"},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_msa(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
