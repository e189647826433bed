"""Benchmark of the fused shared-prefix decode-attention launch on one GB300
(or N independent replicas under torchrun, one per GPU: weak scaling).

A step is one psattn_decode launch over one synthetic batch: the
Llama-3-8B-shaped workload (64 prefix groups x 32 requests, prefix 2048
tokens, suffix uniform in [64, 512], 32 query / 8 KV heads, head_dim 128,
bf16, 16-token blocks).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

--impl reference times the CPU oracle (the only reference this method has),
on a bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = ("shared-prefix decode attention queries/s and achieved HBM GB/s "
          "(% of roofline), 1 GB300")
UNIT = "queries/s"
L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0

DESCRIPTIONS = {
    "llama8b": "Llama-3-8B attention shape: 64 prefix groups x 32 requests (2048), prefix 2048, "
               "suffix U[64,512], 32 q / 8 kv heads, d 128, bf16, block 16",
    "long_prefix": "8 groups x 100 requests, prefix U[1024,10240], suffix U[16,256], 32/8 heads, "
                   "d 128, bf16, block 16",
    "skewed": "1024 requests, Zipf(1.2) over 128 groups, 10% ungrouped, prefix LN(1500,0.8) "
              "[64,8192], suffix LN(200,0.7) [1,2048], 32/8 heads, d 128, bf16",
    "two_level": "4096 requests, level-1 prefix 4096 shared by all, level-2 1024 per 64 groups of "
                 "64, suffix U[32,256], 32/8 heads, d 128, bf16; the plan folds level 1 into the "
                 "level-2 groups' tensor-core items (2 partials per request; --no-fold keeps "
                 "the 3-partial merge), level 1 counted once in the roofline bytes",
    "two_level_flat": "the two-level workload flattened to one 5120-token level per group",
    "tiny_fp32": "2 groups x 8 requests, prefix 256, suffix U[1,64], 4/4 heads, d 64, fp32",
    "chunked": "7 prefill chunks of U[256,512] queries beside 256 decode requests (8 groups x 32, "
               "prefix 2048, suffix U[64,512]), 32/8 heads, d 128, bf16; chunks expanded into "
               "decode rows: each chunk's suffix one ragged level masked per row "
               "(--chunk-form ragged, default) or levels of --level-tokens",
}


def _dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def _peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _peak_bf16():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def _visible_tokens(p):
    """Tokens each row attends to, summed over rows (prefix chain + suffix; a
    ragged leaf level counts its leaf_len tokens)."""
    leaf = getattr(p, "leaf_len", None)
    total = int(p.suffix_len.sum())
    for r in range(p.num_req):
        ch = p.chain(r)
        total += sum(int(p.prefix_len[g]) for g in ch)
        if leaf is not None and leaf[r] >= 0 and ch:
            total -= int(p.prefix_len[ch[-1]]) - int(leaf[r])
    return total


def _traffic_record(workload, default_plan=True):
    """Per-launch DRAM bytes from the committed ncu summary of this workload
    (profiles/psattn_fused_decode_<workload>.md), if that summary records a
    full-size launch (a ``dram_bytes_per_launch:`` line) taken on the current
    kernel source; else None.  Returns (bytes or None, where they come from).
    The summaries are of the default plan, so any plan or size override gives
    None.  The bytes are copied from the summary, not measured in this run."""
    if not default_plan:
        return None, "none: the committed summaries cover the default plan only"
    src = os.path.join(ROOT, "shared_prefix_kv_gb300", "csrc", "decode.cu")
    rel = os.path.join("profiles", f"psattn_fused_decode_{workload}.md")
    try:
        text = open(os.path.join(ROOT, rel)).read()
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
        m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
        m_b = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
        if m_sha and m_b and m_sha.group(1) == sha:
            return int(m_b.group(1)), (f"{rel} (ncu dram__bytes_read.sum + dram__bytes_write.sum "
                                       f"of one full-size launch, same kernel source)")
        if m_b:
            return None, f"none: {rel} was taken on another kernel source"
    except OSError:
        pass
    return None, f"none: no summary with full-launch DRAM bytes at {rel}"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 100):
        self.index = index
        self.period_ms = period_ms
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.samples = []
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:  # a sampler stuck in the driver: no samples
                out = ""
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                self.samples.append((float(parts[0]), float(parts[1]), parts[3:7]))
            except ValueError:
                pass

    def summary(self):
        if not getattr(self, "samples", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in self.samples for i, v in enumerate(r)
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(s[0] for s in self.samples),
                "sm_max_mhz": max(s[1] for s in self.samples), "reasons": reasons,
                "samples": len(self.samples)}


def _oracle_threads(world: int) -> int:
    """Threads for the CPU oracle: the OpenMP default (0) in a single process.
    Under torchrun every rank gets OMP_NUM_THREADS=1, but the oracle runs on
    rank 0 alone, so there it takes every core this process may run on."""
    if world <= 1:
        return 0
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def _oracle_rate(p, budget_s: float, max_req=None, nthreads: int = 0):
    """Queries/s of the CPU oracle over the first requests of the batch, run in
    blocks until `budget_s` of wall time is spent."""
    import oracle
    order = np.arange(p.num_req)
    done, t0 = 0, time.perf_counter()
    block = 16
    while done < p.num_req and (max_req is None or done < max_req):
        req = order[done:done + block]
        oracle.attention(p, req, nthreads=nthreads)
        done += len(req)
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return done / dt, done, dt, oracle.max_threads()


def run_reference(args, p):
    """CPU oracle as the reference arm: each step attends a bounded sample of
    requests of the same batch; value = requests / wall time."""
    rank, world, _ = _dist_env()
    if rank != 0:
        return 0
    import oracle
    nthreads = _oracle_threads(world)
    # calibrate so that warmup + steps stay within about a minute
    rate, _, _, cores = _oracle_rate(p, 2.0, max_req=64, nthreads=nthreads)
    per_step = max(1, min(p.num_req, int(60.0 * rate / max(1, args.steps + args.warmup))))
    rng = np.random.default_rng(0)
    for _ in range(args.warmup):
        oracle.attention(p, rng.choice(p.num_req, per_step, replace=False), nthreads=nthreads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attention(p, rng.choice(p.num_req, per_step, replace=False), nthreads=nthreads)
    dt = time.perf_counter() - t0
    value = per_step * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _config(args, p),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} random requests of the batch per step "
                                   f"(all Hq heads, full prefix+suffix each)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def _overrides(args):
    return {} if args.groups is None else {"n_groups": args.groups}


def _make(args, seed=None):
    return _make_named(args.workload, seed, _overrides(args), args.chunk_form, args.level_tokens)


def _make_named(workload, seed=None, overrides=None, chunk_form="ragged", level_tokens=256):
    """The workload's problem, and (algorithmic KV + q/out bytes, attention
    FLOPs) when the bytes differ from what the plan reports (None otherwise).
    A batch with prefill chunks runs as the library's expansion of it into
    decode rows; its algorithmic bytes count each token of the original batch
    once (a prefix once per group) plus q, out and lse of every query, and its
    FLOPs are 4 * Hq * d per (query, visible token)."""
    if workload != "chunked":
        return W.make(workload, seed=seed, poison=False, **(overrides or {})), None
    import dataclasses
    import shared_prefix_kv_gb300 as ps
    from shared_prefix_kv_gb300 import chunked
    from workloads.device import shape_of
    p, ql, q = W.make_chunked(seed=6 if seed is None else seed, poison=False)
    if chunk_form == "ragged":
        sh, bt, gor, gpar, plen, slen, leaf = chunked.expand_ragged(
            shape_of(p), p.block_table, p.group_of_req, p.group_parent, p.prefix_len,
            p.suffix_len, ql)
    else:
        sh, bt, gor, gpar, plen, slen = chunked.expand(shape_of(p), p.block_table,
                                                       p.group_of_req, p.group_parent,
                                                       p.prefix_len, p.suffix_len, ql,
                                                       level_tokens)
        leaf = None
    p2 = dataclasses.replace(p, q=q, block_table=bt, group_of_req=gor, group_parent=gpar,
                             prefix_len=plen, suffix_len=slen)
    p2.leaf_len = leaf
    used = sorted(set(int(g) for g in p.group_of_req) - {-1})
    tok = sum(int(p.prefix_len[g]) for g in used) + int(p.suffix_len.sum())
    tb = 2 * p.num_kv_heads * p.head_dim * p.elem_bytes
    qo = int(ql.sum()) * p.num_q_heads * (2 * p.head_dim * p.elem_bytes + 4)
    return p2, (tok * tb + qo, 4.0 * p.num_q_heads * p.head_dim * _visible_tokens(p2))


def _config(args, p):
    desc = DESCRIPTIONS.get(args.workload, args.workload)
    if args.groups is not None:
        desc += f" (groups overridden to {args.groups})"
    if getattr(args, "no_fold", False):
        desc += " (planned with no folding: every prefix level its own partial)"
    if getattr(args, "plan_flag", None):
        desc += " (plan flags: " + ", ".join(args.plan_flag) + ")"
    return {"workload": f"{args.workload}: {desc}",
            "requests_per_gpu": p.num_req, "global_batch": p.num_req * args.gpus,
            "parallelism": f"replicas x{args.gpus} (independent batches)",
            "l2": "flushed (256 MiB write) between timed launches; KV working set > L2",
            "seed": p.seed}


# Every workload of the benchmark's configurations, measured in the default
# run beside the headline: (label, workload, plan flag names, description).
PER_WORKLOAD = [
    ("tiny_fp32", "tiny_fp32", (), None),
    ("llama8b", "llama8b", (), None),
    ("long_prefix", "long_prefix", (), None),
    ("skewed", "skewed", (), None),
    ("two_level", "two_level", (), None),
    ("two_level_3partial", "two_level", ("NO_FOLD",),
     "the two-level workload as a 3-partial merge: level 1, the level-2 group and the "
     "suffix each their own partial (PSATTN_NO_FOLD)"),
    ("two_level_flat", "two_level_flat", (), None),
    ("chunked", "chunked", (), None),
]


def per_workload(torch, ps, local, flush, min_launches=50, min_seconds=0.4, reuse=None):
    """Each workload of PER_WORKLOAD on this GPU: >= min_launches timed
    launches (and at least min_seconds of them), L2 flushed before each,
    CUDA events around each launch on the launching stream, clocks sampled
    during the timed region; its own roofline against its algorithmic bytes,
    and the same kernel with de-duplication off.  reuse maps a workload name
    to an already built (problem, chunk_info) to skip drawing it again."""
    from workloads.device import DeviceProblem
    peak, peak_kind = _peak_hbm()
    stream = torch.cuda.current_stream()
    out = {}
    cache = dict(reuse or {})

    def timed(d, pl, n):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        torch.cuda.synchronize()
        for a, b in ev:
            flush.fill_(1)
            a.record(stream)
            d.decode(pl, stream)
            b.record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev]

    for label, wl, flag_names, desc in PER_WORKLOAD:
        if wl not in cache:
            if wl == "two_level_flat" and "two_level" in cache:
                # the same requests, pool and tables with every chain collapsed
                cache = {wl: (W.flatten_problem(cache["two_level"][0]), None)}
            else:
                cache = {wl: _make_named(wl)}  # one workload's inputs held at a time
        p, chunk_info = cache[wl]
        print(f"per_workload: {label}", file=sys.stderr, flush=True)
        flags = 0
        for f in flag_names:
            flags |= getattr(ps, f)
        d = DeviceProblem(p)
        t0 = time.perf_counter()
        pl = d.plan(flags)
        plan_ms = 1e3 * (time.perf_counter() - t0)
        info = pl.info()
        for _ in range(5):
            d.decode(pl, stream)
        est = float(np.mean(timed(d, pl, 5)))
        n = int(max(min_launches, min(4000, math.ceil(min_seconds * 1e3 / (est + 0.05)))))
        with ClockSampler(local, period_ms=50) as clk:
            times = timed(d, pl, n)
        rc, dflags = pl.status()
        ms = float(np.mean(times))
        rows = p.num_req
        alg = chunk_info[0] if chunk_info else info["unique_kv_bytes"] + info["qo_bytes"]
        achieved = alg / (ms * 1e-3) / 1e9
        traffic, traffic_src = _traffic_record(label)
        e = {"description": desc or DESCRIPTIONS.get(wl, wl),
             "dtype": "bf16" if p.dtype == W.BF16 else "f32",
             "launches": n, "ms_per_step": ms, "ms_per_step_median": float(np.median(times)),
             "value": rows / (ms * 1e-3),
             "unit": "query rows/s" if chunk_info else UNIT,
             "rows": rows,
             "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                          "frac": achieved / peak, "algorithmic_bytes_per_launch": alg,
                          "traffic": traffic, "traffic_source": traffic_src,
                          "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"},
             "plan_ms": plan_ms, "dense_items": info["dense_items"],
             "warp_items": info["warp_items"], "partial_slots": info["partial_slots"],
             "error_word": dflags if rc != 0 else 0,
             "clocks": clk.summary(),
             "l2": "flushed (256 MiB write) before every timed launch"}
        if chunk_info:
            tf = chunk_info[1] / (ms * 1e-3) / 1e12
            e["tensor"] = {"flops_per_launch": chunk_info[1], "achieved_tflops": tf,
                           "peak_tflops": _peak_bf16(), "frac": tf / _peak_bf16()}
        pl.close()
        if not flag_names:
            nd = d.plan(ps.NO_DEDUP)
            nd_times = timed(d, nd, 20)
            nd_ms = float(np.mean(nd_times))
            nd_info = nd.info()
            e["no_dedup"] = {
                "ms_per_step": nd_ms, "value": rows / (nd_ms * 1e-3), "launches": 20,
                "gbs_own_bytes": (nd_info["planned_kv_bytes"] + nd_info["qo_bytes"])
                / (nd_ms * 1e-3) / 1e9,
                "gbs_dedup_bytes": alg / (nd_ms * 1e-3) / 1e9,
                "speedup_of_dedup": nd_ms / ms}
            nd.close()
        out[label] = e
        del d
        torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama8b", choices=sorted(DESCRIPTIONS))
    ap.add_argument("--groups", type=int, default=None,
                    help="override the number of prefix groups (smaller captures for profiling)")
    ap.add_argument("--level-tokens", type=int, default=256,
                    help="causal level size for the chunked workload (multiple of 16)")
    ap.add_argument("--chunk-form", choices=["ragged", "levels"], default="ragged",
                    help="chunked workload: one ragged level per chunk, or fixed-size levels")
    ap.add_argument("--no-fold", action="store_true",
                    help="plan every prefix level as its own partial (no folding of parent "
                         "levels into their children's tensor-core items)")
    ap.add_argument("--no-baselines", action="store_true",
                    help="skip the CPU-oracle, no-dedup and end-to-end legs")
    ap.add_argument("--plan-flag", action="append", default=[],
                    choices=["SIMT", "NO_TENSOR_PREFIX", "FLATTEN", "NO_FOLD"],
                    help="extra plan flag for the headline launch (repeatable), e.g. SIMT for "
                         "the CUDA-core per-warp path")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the per_workload block (every configuration's own "
                         "measurement, single-GPU runs only)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    rank, world, local = _dist_env()

    if args.impl == "reference":
        if rank != 0:
            return 0
        p, _ = _make(args)
        return run_reference(args, p)

    import torch
    import shared_prefix_kv_gb300 as ps
    from workloads.device import DeviceProblem, shape_of  # device upload helper (torch memory only)

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    # each rank gets its own independent batch (weak scaling)
    p, chunk_info = _make(args, seed=None if rank == 0 else 1000 + rank)
    alg_override = chunk_info[0] if chunk_info else None
    d = DeviceProblem(p)
    t_plan = time.perf_counter()
    plan_flags = ps.NO_FOLD if args.no_fold else 0
    for f in args.plan_flag:
        plan_flags |= getattr(ps, f)
    plan = d.plan(plan_flags)
    t_plan = time.perf_counter() - t_plan
    info = plan.info()
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device="cuda")

    def timed(pl, steps, warm):
        for _ in range(warm):
            d.decode(pl, stream)
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        for a, b in ev:
            flush.fill_(1)
            a.record(stream)
            d.decode(pl, stream)
            b.record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        return [a.elapsed_time(b) for a, b in ev]

    with ClockSampler(local) as clk:
        times = timed(plan, args.steps, args.warmup)
    rc, dflags = plan.status()
    if rc != 0:
        raise RuntimeError(f"device error word {dflags}")
    ms = float(np.mean(times))
    if dist:
        t = torch.tensor([ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    value = p.num_req * world / (ms * 1e-3)
    alg_bytes = alg_override or (info["unique_kv_bytes"] + info["qo_bytes"])
    peak, peak_kind = _peak_hbm()
    achieved = alg_bytes / (ms * 1e-3) / 1e9
    traffic, traffic_src = _traffic_record(
        args.workload, args.groups is None and not args.no_fold and args.chunk_form == "ragged"
        and not args.plan_flag)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if p.dtype == W.BF16 else "f32",
        "data": "synthetic (seeded N(0,1) q/K/V, shuffled paged block tables)",
        "config": _config(args, p),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "traffic_source": traffic_src,
                     "kernel": "psattn_fused_decode",
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s"},
        "achieved_hbm_gbs": achieved,
        "pct_of_roofline": 100.0 * achieved / peak,
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
        "plan_ms": 1e3 * t_plan,
        "ms_per_step_median": float(np.median(times)),
    }
    if chunk_info:  # prefill chunks make the batch heavy on the tensor cores too
        tf = chunk_info[1] / (ms * 1e-3) / 1e12
        line["tensor"] = {"flops_per_launch": chunk_info[1], "achieved_tflops": tf,
                          "peak_tflops": _peak_bf16(), "frac": tf / _peak_bf16()}

    if not args.no_baselines:
        # same kernel, prefix de-duplication disabled
        nd = d.plan(ps.NO_DEDUP)
        nd_times = timed(nd, max(20, args.steps // 4), 3)
        nd_ms = float(np.mean(nd_times))
        nd_info = nd.info()
        line["no_dedup"] = {
            "value": p.num_req * world / (nd_ms * 1e-3), "unit": UNIT, "ms_per_step": nd_ms,
            "gbs_own_bytes": (nd_info["planned_kv_bytes"] + nd_info["qo_bytes"]) / (nd_ms * 1e-3) / 1e9,
            "gbs_dedup_bytes": alg_bytes / (nd_ms * 1e-3) / 1e9}
        nd.close()

        # end to end through the public call with host buffers: every step
        # copies its inputs (q, block table, group ids, lengths) from pinned host
        # memory, runs the launch and copies out and lse back; the KV pool is
        # device-resident cache state.  Two buffer sets, with the copies on
        # their own streams, let step k + 1's inputs and step k's results move
        # while a decode runs (the decodes themselves run one after another on
        # the compute stream: they share the plan's workspace).
        hq = d.q.cpu().pin_memory()
        host_in = [t.cpu().pin_memory() for t in (d.bt, d.gor, d.plen, d.slen)]
        h_out = [torch.empty(d.out.shape, dtype=d.out.dtype).pin_memory() for _ in range(2)]
        h_lse = [torch.empty(d.lse.shape, dtype=d.lse.dtype).pin_memory() for _ in range(2)]
        bufs = [dict(q=torch.empty_like(d.q), ins=[torch.empty_like(t) for t in (d.bt, d.gor, d.plen, d.slen)],
                     out=torch.empty_like(d.out), lse=torch.empty_like(d.lse)) for _ in range(2)]
        h2d = hq.numel() * hq.element_size() + sum(t.numel() * t.element_size() for t in host_in)
        d2h = h_out[0].numel() * h_out[0].element_size() + h_lse[0].numel() * h_lse[0].element_size()
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of set i landed
        ev_done = [torch.cuda.Event() for _ in range(2)]  # the decode on set i finished
        ev_out = [torch.cuda.Event() for _ in range(2)]   # results of set i are on the host

        def e2e_step(k):
            i = k % 2
            B = bufs[i]
            s_in.wait_event(ev_done[i])  # the decode two steps back is done with set i
            with torch.cuda.stream(s_in):
                B["q"].copy_(hq, non_blocking=True)
                for dv, hv in zip(B["ins"], host_in):
                    dv.copy_(hv, non_blocking=True)
            ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            stream.wait_event(ev_out[i])  # set i's previous results have left
            plan.decode(B["q"], d.pool, *B["ins"], B["out"], B["lse"], stream=stream.cuda_stream)
            ev_done[i].record(stream)
            s_out.wait_event(ev_done[i])
            with torch.cuda.stream(s_out):
                h_out[i].copy_(B["out"], non_blocking=True)
                h_lse[i].copy_(B["lse"], non_blocking=True)
            ev_out[i].record(s_out)

        for k in range(4):
            e2e_step(k)
        torch.cuda.synchronize()
        ne = max(20, args.steps // 4)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        a.record(stream)
        s_in.wait_event(a)
        for k in range(ne):
            e2e_step(k)
        stream.wait_event(ev_out[(ne - 1) % 2])
        stream.wait_event(ev_out[(ne - 2) % 2])
        b.record(stream)
        torch.cuda.synchronize()
        e_ms = a.elapsed_time(b) / ne
        # the host copy of the last step against the device-timed run's output
        # (merge order varies between launches: compare within the bound)
        ok = bool((h_out[(ne - 1) % 2].float() - d.out.float().cpu()).abs().max().item()
                  <= (1e-2 if d.out.dtype == torch.bfloat16 else 1e-4))
        if dist:
            t = torch.tensor([e_ms], device="cuda")
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            e_ms = float(t.item())
        line["e2e"] = {"value": p.num_req * world / (e_ms * 1e-3), "unit": UNIT,
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": e_ms, "double_buffered": True,
                       "l2": "not flushed (KV working set larger than L2)",
                       "result_matches_device_run": bool(ok)}
        line["gpu_launches"] = args.steps

        if rank == 0 and world == 1:
            rate, n, dt, cores = _oracle_rate(p, 15.0)
            line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                                    "sample": f"first {n} requests of the batch ({dt:.1f} s "
                                              f"wall, all heads, double precision)"}

    plan.close()
    if world == 1 and not args.no_per_workload:
        del d
        torch.cuda.empty_cache()
        reuse = {args.workload: (p, chunk_info)} if args.groups is None and \
            args.chunk_form == "ragged" and args.workload in dict(
                (w, 1) for _, w, _, _ in PER_WORKLOAD) else None
        line["per_workload"] = per_workload(torch, ps, local, flush, reuse=reuse)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
