#!/usr/bin/env python3
"""Benchmark: paged causal GQA attention on GB300, one JSON line on stdout.

Default workload (N=1): GQA decode -- batch 32, 32 q heads / 8 kv heads,
head_dim 128, per-sequence context uniform on [1024, 32768] (seeded), 16-token
pages in a shared shuffled pool, bf16 q/K/V, bf16 output.  A step is one call
of atlas_attn_decode: split-KV fold of every page (page-table gather, scores,
online softmax, PV, partial write) plus the log-sum-exp merge.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..5]
  python bench.py --impl reference   # the fp64 CPU oracle on host cores

Under torchrun each rank runs its own seeded batch on its own GPU (weak scaling,
no collective on the data path); rank 0 prints the line, timing is the max over
ranks.  KV bytes are algorithmic: every visible key's K and V row read once.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "decode KV GB/s (% of HBM peak); prefill TFLOP/s (% of bf16 TC peak)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129 * 1024 * 1024


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["atlas", "reference"], default="atlas")
    ap.add_argument("--config", type=int, default=None, choices=[1, 2, 3, 4, 5],
                    help="measure only this workload (default: GQA decode as the headline "
                         "line, every other workload under its 'configs' key)")
    ap.add_argument("--no-configs", action="store_true",
                    help="default run: skip the other workloads' measurements")
    ap.add_argument("--split-tokens", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch (smaller profiling captures)")
    ap.add_argument("--window", type=int, default=0, help="sliding window (keys); 0 = none")
    ap.add_argument("--softcap", type=float, default=0.0, help="logit softcap; 0 = none")
    ap.add_argument("--sinks", action="store_true", help="one sink logit per q head")
    ap.add_argument("--ragged", action="store_true",
                    help="ragged query counts: q_lens[b] ~ U{1..q_len} (suffix/prefill)")
    ap.add_argument("--dtype", choices=["bf16", "f32"], default=None,
                    help="override the config's q/K/V (and output) dtype")
    ap.add_argument("--pool", type=float, default=0.0,
                    help="serve the decode from a bounded hot-page pool holding this "
                         "fraction of the workload's pages (host tier in pinned memory)")
    ap.add_argument("--keep-recent", type=int, default=2048,
                    help="--pool: KeepRecent window in tokens (-1: every page)")
    ap.add_argument("--scratch-pages", type=int, default=0,
                    help="--pool: scratch slots (0: 4096 or two chunks, the larger)")
    ap.add_argument("--append", action="store_true",
                    help="time atlas_kv_append writing the workload's K/V into its pages")
    ap.add_argument("--settle-s", type=float, default=1.0,
                    help="untimed steps for this long before the timed region, so that the "
                         "clock sampler sees the GPU under load (0 for profiler runs)")
    return ap.parse_args()


def rank_seed(config_index: int, rank: int) -> int:
    """Each rank draws its own batch (weak scaling: per-rank work is fixed)."""
    return config_index + 1000 * rank


def max_over_ranks(value: float, device) -> float:
    """The slowest rank's time (identity when torch.distributed is not initialised)."""
    t = torch.tensor([value], dtype=torch.float64, device=device)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, ms_max: float, scale: float) -> float:
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    return world * units_per_rank / (ms_max * 1e-3) / scale


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            data = json.load(f)
        return data, "measured"
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS}, "fallback"


def work_of_ragged(prob, q_lens):
    """(KV bytes, FLOPs) with q_lens[b] query rows per sequence (no window)."""
    lens = prob.seq_lens.to(torch.int64).cpu()
    qn = q_lens.to(torch.int64).cpu()
    keys = int((qn * (lens - qn) + qn * (qn + 1) // 2).sum())
    kv = 2 * int(lens.sum()) * prob.n_kv_heads * prob.head_dim * prob.k_pages.element_size()
    return kv, 4 * prob.head_dim * prob.n_q_heads * keys


def work_of(prob, window: int = 0):
    """Algorithmic work of one call: (KV bytes, FLOPs).  KV bytes count each key
    any query row of a sequence may see once (K and V); FLOPs count 4*D per
    (query row, visible key) -- QK^T and PV, masked keys excluded."""
    lens = prob.seq_lens.to(torch.int64).cpu()
    sq = prob.q_len
    elem = prob.k_pages.element_size()
    if window > 0:
        kv_keys = int(torch.clamp(lens, max=window + sq - 1).sum())
        i = torch.arange(sq, dtype=torch.int64)
        vis = (lens[:, None] - sq + i[None, :] + 1).clamp(max=window)
        keys = int(vis.sum())
    else:
        kv_keys = int(lens.sum())
        keys = int((lens * sq).sum()) - sq * (sq - 1) // 2 * prob.batch
    kv = 2 * kv_keys * prob.n_kv_heads * prob.head_dim * elem
    flops = 4 * prob.head_dim * prob.n_q_heads * keys
    return kv, flops


TC_MIN_COLS = 17  # calls with more query rows per kv head take a tensor-core kernel
KERNEL_SOURCES = {"split_bf16_kernel": "split_kv.cu", "split_f32_kernel": "split_kv.cu",
                  "fmha_tc_kernel": "fmha_tc.cu", "fmha_tf32x3_kernel": "fmha_tc_f32.cu"}
# nominal dense tf32 / bf16 tensor rates of the part (1.1 and 2.25 PFLOP/s)
TF32_PER_BF16 = 1.1 / 2.25


def kernel_source_sha(kernel: str) -> str:
    """Hash of the kernel's translation unit and the headers it shares."""
    csrc = os.path.join(ROOT, "exact_causal_gqa_gb300", "csrc")
    h = hashlib.sha256()
    names = [KERNEL_SOURCES[kernel], "ptx.cuh", "internal.h"]
    if kernel.startswith("fmha_"):
        names.append("tc_order.cuh")
    for name in names:
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


def workload_traffic(args, kernel: str, workload: str):
    """traffic_record for the named workload as the committed capture measured it; None
    when this run changes the workload (batch, window, softcap, sinks, ragged rows or a
    fixed split size), whose per-launch DRAM bytes that record does not describe."""
    if args.batch or args.window or args.softcap or args.sinks or args.ragged or \
            args.split_tokens:
        return None
    return traffic_record(kernel, workload)


def traffic_record(kernel: str, workload: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if the
    kernel source is unchanged since it was captured; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = kernel_source_sha(kernel)
    for line in open(path):
        parts = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
        if parts.get("kernel") == kernel and parts.get("workload") == workload and \
                parts.get("source_sha") == sha:
            return float(parts["dram_bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self, t_begin: float, t_end: float):
        """Median SM clock and the throttle reasons seen in samples stamped inside
        [t_begin, t_end] (host wall-clock seconds)."""
        import datetime
        if not self.lines:
            return None
        sm, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                if not (t_begin <= ts <= t_end):
                    continue
                sm.append(float(f[2]))
                mx.append(float(f[3]))
                power.append(float(f[4]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, f[6:10]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "power_w": statistics.median(power), "reasons": sorted(reasons),
                "samples": len(sm)}


HEADLINE_CONFIG = 2
# The other workloads measured in a default run, prefill (the metric's second half) first.
OTHER_CONFIGS = (5, 4, 3, 1)


def changes_workload(args) -> bool:
    """True when a flag changes the named workloads (then only the headline runs)."""
    return bool(args.batch or args.window or args.softcap or args.sinks or args.ragged or
                args.split_tokens or args.dtype)


def run_atlas(args, world, rank, local):
    """The headline workload's line; in a default run (no --config, no flag that
    changes the workload) every other workload is measured the same way in the same
    process and reported under "configs"."""
    index = args.config or HEADLINE_CONFIG
    line = measure(args, index, world, rank, local, e2e=not args.no_e2e,
                   cpu_budget=None if args.no_cpu_baseline else 12.0)
    if args.config is None and not args.no_configs and not changes_workload(args):
        others = {}
        for other in OTHER_CONFIGS:
            torch.cuda.empty_cache()
            sub = measure(args, other, world, rank, local, e2e=False,
                          cpu_budget=None if args.no_cpu_baseline else 3.0)
            if sub is not None:
                others[str(other)] = config_summary(sub)
        if line is not None:
            line["configs"] = others
    return line


def config_summary(line):
    """The per-workload entry of a default run's "configs" object."""
    keep = ("value", "unit", "ms_per_step", "dtype", "roofline", "gpu_launches",
            "device_status", "clocks", "cpu_baseline")
    out = {k: line[k] for k in keep if k in line}
    c = line["config"]
    out["workload"] = c["workload"]
    out["kind"] = c["kind"]
    for k in ("kv_bytes_per_step", "flops_per_step", "l2", "per_step_ms", "main_kernel_ms",
              "merge_kernel_ms"):
        out[k] = c[k]
    return out


def measure(args, index, world, rank, local, e2e=True, cpu_budget=12.0):
    """Time workload `index` (inputs resident in HBM) and return its JSON line on
    rank 0 (None elsewhere).  Flags that change the workload apply to the headline
    workload only (run_atlas never passes them to the others)."""
    import exact_causal_gqa_gb300 as atlas
    from exact_causal_gqa_gb300 import inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    atlas.load_library()
    cfg = inputs.CONFIGS[index]
    seed = rank_seed(index, rank)
    overrides = {"B": args.batch} if args.batch else {}
    if args.dtype:
        overrides.update(dtype=args.dtype, out_dtype=args.dtype)
    prob = inputs.make_config(index, seed=seed, device=dev, **overrides)
    kv_bytes, flops = work_of(prob, args.window)
    variants = dict(window=args.window, softcap=args.softcap)
    if args.ragged:
        g = torch.Generator().manual_seed(seed + 7)
        q_lens = torch.randint(1, prob.q_len + 1, (prob.batch,), generator=g, dtype=torch.int32)
        if prob.kind == "prefill":  # a ragged prompt batch: each prompt is its own length
            prob.seq_lens = q_lens.to(dev)
        variants["q_lens"] = q_lens.to(dev)
        kv_bytes, flops = work_of_ragged(prob, q_lens)
    if args.sinks:
        g = torch.Generator().manual_seed(seed)
        variants["sinks"] = (torch.randn(prob.n_q_heads, generator=g) * 2.0).float().to(dev)
    out_dtype = torch.bfloat16 if prob.out_dtype == "bf16" else torch.float32
    out = torch.empty(prob.q.shape, dtype=out_dtype, device=dev)
    ws_bytes = atlas.workspace_size(prob.kind, prob.q.shape, prob.n_q_heads, prob.n_kv_heads,
                                    prob.head_dim, prob.page_tokens, prob.max_pages,
                                    prob.num_pages, dtype=prob.q.dtype, out_dtype=out_dtype,
                                    split_tokens=args.split_tokens, window=args.window)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    timers = [atlas.EventTimer() for _ in range(args.steps)]
    needs_flush = kv_bytes < 2 * L2_BYTES
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if needs_flush else None

    def step(timer=None):
        atlas.run(prob, out=out, workspace=ws, status=status, split_tokens=args.split_tokens,
                  events=None if timer is None else timer.handles, **variants)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during warm-up")

    step_start = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    step_end = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        # Untimed steps for about a second so the clock sampler sees the GPU under
        # this load even when the timed region is shorter than its period.
        settle_end = time.time() + args.settle_s
        while time.time() < settle_end:
            for _ in range(20):
                step()
            torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        t_begin = time.time()
        t0 = time.perf_counter()
        for k in range(args.steps):
            if flush is not None:
                flush.fill_(float(k))  # evict the previous step's inputs from L2
            step_start[k].record()
            step()
            step_end[k].record()
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
        t_end = time.time()
        # The same steps again with the library recording events around its main
        # kernel and its merge: the kernel split of the step (the events add a few
        # microseconds to a step, so the step time above is taken without them).
        for k in range(args.steps):
            if flush is not None:
                flush.fill_(float(k))
            step(timers[k])
        torch.cuda.synchronize(dev)
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(step_start, step_end)]
    main_ms = [t.main_ms() for t in timers]
    ms = sum(step_ms) / len(step_ms)
    ms_max = max_over_ranks(ms, dev)
    status_val = int(status.item())

    # ---- end to end: pinned host inputs -> device -> kernels -> host output
    e2e_res = None
    if e2e:
        host = [t.to("cpu").pin_memory() for t in (prob.q, prob.k_pages, prob.v_pages,
                                                    prob.page_table, prob.seq_lens)]
        dbuf = [torch.empty_like(t, device=dev) for t in host]
        host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        bi = sum(t.numel() * t.element_size() for t in host)
        bo = host_out.numel() * host_out.element_size()

        def e2e_step():
            for d, h in zip(dbuf, host):
                d.copy_(h, non_blocking=True)
            atlas._call(prob.kind, *dbuf, prob.n_q_heads, prob.n_kv_heads, prob.head_dim,
                        prob.page_tokens, prob.scale, out=out, workspace=ws, status=status,
                        split_tokens=args.split_tokens, **variants)
            host_out.copy_(out, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        e_steps = max(3, min(args.steps, 10))
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record()
        for _ in range(e_steps):
            e2e_step()
        ev1.record()
        torch.cuda.synchronize(dev)
        e2e_res = (max_over_ranks(ev0.elapsed_time(ev1) / e_steps, dev), bi, bo)
        del host, dbuf, host_out

    if rank != 0:
        return None
    pk, pk_kind = peaks()
    decode_like = prob.kind != "prefill"
    main_avg = sum(main_ms) / len(main_ms)
    if decode_like:
        value = job_rate(kv_bytes, world, ms_max, 1e9)
        unit = "GB/s"
        achieved = kv_bytes / (main_avg * 1e-3) / 1e9
        peak = float(pk.get("hbm_gbs", FALLBACK_HBM_GBS))
        bound = "hbm"
    else:
        value = job_rate(flops, world, ms_max, 1e12)
        unit = "TFLOP/s"
        achieved = flops / (main_avg * 1e-3) / 1e12
        peak = float(pk.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
        bound = "tensor"
    tc_path = prob.q_len * (prob.n_q_heads // prob.n_kv_heads) >= TC_MIN_COLS
    f32_tc = tc_path and prob.dtype == "f32"
    if tc_path:
        kernel = "fmha_tc_kernel" if prob.dtype == "bf16" else "fmha_tf32x3_kernel"
    else:
        kernel = "split_bf16_kernel" if prob.dtype == "bf16" else "split_f32_kernel"
    # launches per step: the main kernel, plus the merge unless the tensor-core
    # path wrote the output directly (timer event 2 then coincides with event 1)
    merge_ms = sum(t.merge_ms() for t in timers) / len(timers)
    # no workspace: the main kernel wrote the output itself (tensor-core direct mode,
    # a short bf16 context in one split, fp32 splits merged inside a cluster)
    launches_per_step = 1 if ws_bytes == 0 else 2
    if f32_tc:
        # fp32 on the tensor cores as three tf32 products per fp32 product: the
        # ceiling is a third of the tf32 peak (the measured bf16 peak x 1.1 / 2.25);
        # achieved counts algorithmic flops
        tf32 = float(pk.get("bf16_tflops", FALLBACK_BF16_TFLOPS)) * TF32_PER_BF16
        peak = tf32 / 3
        achieved = flops / (main_avg * 1e-3) / 1e12
        bound = "tensor"
        pk_kind = (f"{pk_kind} bf16 x 1.1/2.25 = {tf32:.1f} TFLOP/s tf32, / 3 tf32 products "
                   "per fp32 product")
    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(3, args.warmup),
        "ms_per_step": round(ms_max, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": prob.dtype,
        "data": "synthetic (seeded N(0,1) q/K/V, shuffled page pool)",
        "config": {
            "workload": cfg["name"] + (f" (batch {args.batch})" if args.batch else "") +
            (f" as {args.dtype}" if args.dtype and args.dtype != cfg["dtype"] else "") +
            (f" window {args.window}" if args.window else "") +
            (f" softcap {args.softcap}" if args.softcap else "") + (" sinks" if args.sinks else "") +
            (" ragged" if args.ragged else ""),
            "kind": prob.kind, "batch": prob.batch, "n_q_heads": prob.n_q_heads,
            "n_kv_heads": prob.n_kv_heads, "head_dim": prob.head_dim,
            "page_tokens": prob.page_tokens, "q_len": prob.q_len,
            "context": list(cfg["ctx"]), "sum_context": int(prob.seq_lens.sum()),
            "kv_bytes_per_step": kv_bytes, "flops_per_step": flops,
            "l2": ("flushed between steps (2x L2 write)" if flush is not None
                   else f"inputs larger than L2 ({kv_bytes / 1e9:.2f} GB KV vs 129 MB)"),
            "parallelism": f"replicas x{world} (independent batches per GPU)",
            "split_tokens": args.split_tokens or "auto",
            "variants": {"window": args.window, "softcap": args.softcap, "sinks": args.sinks},
            "per_step_ms": {"min": round(min(step_ms), 5),
                            "median": round(statistics.median(step_ms), 5)},
            "main_kernel_ms": round(main_avg, 5),
            "merge_kernel_ms": round(merge_ms, 5),
            "wall_s": round(wall, 4),
        },
        "roofline": {
            "kernel": kernel,
            "bound": bound,
            "achieved": round(achieved, 3),
            "peak": peak,
            "peak_source": pk_kind,
            "unit": "TFLOP/s" if f32_tc else unit,
            "frac": round(achieved / peak, 4),
            "traffic": workload_traffic(args, kernel, cfg["name"]),
        },
        "gpu_launches": launches_per_step * args.steps,
        "device_status": status_val,
    }
    # Samples of the timed region; if it was shorter than the 200 ms period, the
    # last half second of the identical untimed loop just before it.
    clk = clocks.summary(t_begin, t_end + 0.05) or clocks.summary(t_begin - 0.5, t_end + 0.05)
    if clk is not None:
        clk["window"] = "timed region" if clocks.summary(t_begin, t_end + 0.05) else \
            "last 0.5 s of the identical untimed loop + timed region"
    line["clocks"] = clk
    if e2e_res is not None:
        e_ms, bi, bo = e2e_res
        e_val = job_rate(kv_bytes, world, e_ms, 1e9) if decode_like else \
            job_rate(flops, world, e_ms, 1e12)
        line["e2e"] = {"value": round(e_val, 3), "unit": unit, "ms_per_step": round(e_ms, 4),
                       "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo}
    if cpu_budget is not None and world == 1:
        line["cpu_baseline"] = cpu_baseline(index, prob, decode_like, budget_s=cpu_budget)
    return line


def run_append(args, world, rank, local):
    """Time atlas_kv_append writing every token of the workload's K/V into its pages
    (as a prefill would): bytes = read + write of K and V rows."""
    import exact_causal_gqa_gb300 as atlas
    from exact_causal_gqa_gb300 import inputs
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = inputs.CONFIGS[args.config]
    overrides = {"B": args.batch} if args.batch else {}
    prob = inputs.make_config(args.config, seed=rank_seed(args.config, rank), device=dev,
                              **overrides)
    lens = prob.seq_lens.to(torch.int64)
    max_new = int(lens.max())
    g = torch.Generator(device=dev).manual_seed(5)
    k_new = torch.randn((prob.batch, prob.n_kv_heads, max_new, prob.head_dim), generator=g,
                        device=dev).to(prob.k_pages.dtype)
    v_new = torch.randn_like(k_new)
    zeros = torch.zeros(prob.batch, dtype=torch.int32, device=dev)
    moved = 2 * 2 * int(lens.sum()) * prob.n_kv_heads * prob.head_dim * prob.k_pages.element_size()
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        atlas.kv_append(k_new, v_new, prob.k_pages, prob.v_pages, prob.page_table, zeros,
                        prob.seq_lens, status=status)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dev)
    if rank != 0:
        return None
    pk, pk_kind = peaks()
    gbs = job_rate(moved, world, ms, 1e9)
    peak = float(pk.get("hbm_gbs", FALLBACK_HBM_GBS))
    return {"metric": "KV append GB/s (read + write)", "value": round(gbs, 3), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup),
            "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": prob.dtype, "data": "synthetic",
            "config": {"workload": cfg["name"] + " (append all tokens)", "bytes_moved": moved},
            "roofline": {"kernel": "kv_append_kernel", "bound": "hbm", "achieved": round(gbs, 3),
                         "peak": peak, "peak_source": pk_kind, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "traffic": None},
            "gpu_launches": args.steps, "device_status": int(status.item())}


def run_pool(args, world, rank, local):
    """A decode workload served from a bounded hot-page pool: the whole K/V in a
    pinned host tier, a fraction of its pages hot on the device, the rest streamed
    through scratch slots pass by pass.  value = KV bytes attended per step / step
    time (plan + fills + chunk passes + merge); the roofline is the fill kernel
    against a plain pinned host-to-device copy measured in the same run."""
    import exact_causal_gqa_gb300 as atlas
    from exact_causal_gqa_gb300 import inputs
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = inputs.CONFIGS[args.config]
    if cfg["kind"] != "decode":
        raise SystemExit("--pool serves decode workloads (configs 1-3)")
    overrides = {"B": args.batch} if args.batch else {}
    host = inputs.make_config(args.config, seed=rank_seed(args.config, rank), device="cpu",
                              **overrides)
    P, Hq, Hkv, D = host.page_tokens, host.n_q_heads, host.n_kv_heads, host.head_dim
    host_k, host_v = host.k_pages.pin_memory(), host.v_pages.pin_memory()
    table, lens = host.page_table.contiguous(), host.seq_lens.contiguous()
    q = host.q.to(dev)
    kv_bytes, _ = work_of(host)
    total_pages = int(((lens.to(torch.int64) + P - 1) // P).sum())
    out_dtype = torch.bfloat16 if host.out_dtype == "bf16" else torch.float32
    chunk = atlas.split_tokens_of("decode", q.shape, Hq, Hkv, D, P, host.max_pages,
                                  host.num_pages, q.dtype, out_dtype, phase=atlas.PHASE_CHUNKS)
    hot = int(args.pool * total_pages)
    scratch = args.scratch_pages or max(4096, 2 * (chunk // P + 1))
    pool = atlas.HotPagePool(host_k, host_v, hot, scratch, device=dev)
    out = torch.empty(q.shape, dtype=out_dtype, device=dev)
    ws_bytes = atlas.workspace_size("decode", q.shape, Hq, Hkv, D, P, host.max_pages,
                                    host.num_pages, q.dtype, out_dtype, phase=atlas.PHASE_CHUNKS)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        return pool.decode(q, table, lens, Hq, host.scale, keep_recent_tokens=args.keep_recent,
                           out=out, status=status, workspace=ws)

    for _ in range(max(3, args.warmup)):
        _, st = step()
    torch.cuda.synchronize(dev)
    # the pooled result equals the decode over a fully resident pool with the same
    # split size, bit for bit
    resident = inputs.Problem(**{k: (v.to(dev) if torch.is_tensor(v) else v)
                                 for k, v in vars(host).items()})
    ref = atlas.run(resident, out_dtype=out_dtype, split_tokens=chunk)
    torch.cuda.synchronize(dev)
    bitwise = bool(torch.equal(out, ref))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        atlas.run(resident, out=ref)
    e0.record()
    for _ in range(10):
        atlas.run(resident, out=ref)
    e1.record()
    torch.cuda.synchronize(dev)
    resident_ms = e0.elapsed_time(e1) / 10
    del resident, ref

    with ClockSampler(local) as clocks:
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        t_begin = time.time()
        e0.record()
        for _ in range(args.steps):
            _, st = step()
        e1.record()
        torch.cuda.synchronize(dev)
        t_end = time.time()
        time.sleep(0.3)
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dev)

    # The fill kernel alone on a full scratch load of cold pages, and the plain copy
    # of the same bytes from pinned memory (the host link's practical rate).
    n = min(scratch, host.num_pages)
    pairs = torch.stack([torch.randperm(host.num_pages)[:n].to(torch.int32),
                         torch.arange(hot, hot + n, dtype=torch.int32)], 1).to(dev)
    moved = 2 * n * pool.page_bytes
    for _ in range(2):
        pool.fill(pairs, status)
    e0.record()
    for _ in range(5):
        pool.fill(pairs, status)
    e1.record()
    torch.cuda.synchronize(dev)
    fill_gbs = moved / (e0.elapsed_time(e1) / 5 * 1e-3) / 1e9
    src = host_k.view(-1)[: moved // 2 // host_k.element_size()]
    dst = torch.empty(2 * src.numel(), dtype=src.dtype, device=dev)
    for _ in range(2):
        dst[:src.numel()].copy_(src, non_blocking=True)
        dst[src.numel():].copy_(src, non_blocking=True)
    e0.record()
    for _ in range(5):
        dst[:src.numel()].copy_(src, non_blocking=True)
        dst[src.numel():].copy_(src, non_blocking=True)
    e1.record()
    torch.cuda.synchronize(dev)
    copy_gbs = moved / (e0.elapsed_time(e1) / 5 * 1e-3) / 1e9
    if rank != 0:
        return None
    fills = st.passes  # one fill launch per pass (each pass copies something when cold)
    line = {"metric": "pooled decode KV GB/s (bounded hot-page pool)",
            "value": round(job_rate(kv_bytes, world, ms, 1e9), 3), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup),
            "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": host.dtype,
            "data": "synthetic (seeded N(0,1) q/K/V, shuffled page pool)",
            "config": {"workload": cfg["name"] + f" via hot-page pool ({args.pool:.0%} hot)",
                       "kv_bytes_per_step": kv_bytes, "pages": total_pages,
                       "hot_slots": hot, "scratch_slots": scratch,
                       "keep_recent_tokens": args.keep_recent, "chunk_tokens": chunk,
                       "pool_stats_per_step": st.as_dict(),
                       "bytes_copied_per_step": 2 * st.copies * pool.page_bytes,
                       "bitwise_equal_to_resident_decode": bitwise,
                       "resident_decode_ms": round(resident_ms, 4),
                       "l2": f"inputs larger than L2 ({kv_bytes / 1e9:.2f} GB KV vs 129 MB)"},
            "roofline": {"kernel": "pool_fill_kernel", "bound": "host_link",
                         "achieved": round(fill_gbs, 2), "peak": round(copy_gbs, 2),
                         "peak_source": "pinned host-to-device cudaMemcpy of the same bytes, "
                                        "measured in this run",
                         "unit": "GB/s", "frac": round(fill_gbs / copy_gbs, 4), "traffic": None},
            "gpu_launches": args.steps * (fills + st.passes + 1),
            "device_status": int(status.item())}
    clk = clocks.summary(t_begin, t_end + 0.05)
    line["clocks"] = clk
    return line


def oracle_sample(index, prob_host, decode_like, budget_s):
    """Time the fp64 oracle on whole (sequence, kv head) groups of the workload
    until about budget_s of CPU work; returns (value, unit, cores, sample)."""
    import numpy as np
    import oracle
    q = prob_host.q.float().numpy()
    k = prob_host.k_pages.float().numpy()
    v = prob_host.v_pages.float().numpy()
    table = prob_host.page_table.numpy()
    lens = prob_host.seq_lens.numpy()
    G = prob_host.n_q_heads // prob_host.n_kv_heads
    rng = np.random.default_rng(12345)
    groups = [(b, g) for b in range(prob_host.batch) for g in range(prob_host.n_kv_heads)]
    order = rng.permutation(len(groups))
    done_bytes, done_flops, elapsed, n_groups = 0, 0, 0.0, 0
    for gi in order:
        b, g = groups[gi]
        rows = [((b * prob_host.n_q_heads + g * G + j) * prob_host.q_len + i)
                for j in range(G) for i in range(prob_host.q_len)]
        # bound the rows of very long query blocks (prefill): take a spread of them
        if len(rows) > 512:
            rows = rows[:: max(1, len(rows) // 512)]
        t0 = time.perf_counter()
        oracle.attn(q, k, v, table, lens, prob_host.n_q_heads, prob_host.n_kv_heads,
                    prob_host.scale, rows=np.asarray(rows))
        elapsed += time.perf_counter() - t0
        L = int(lens[b])
        done_bytes += 2 * L * prob_host.head_dim * prob_host.k_pages.element_size()
        for r in rows:
            i = r % prob_host.q_len
            done_flops += 4 * prob_host.head_dim * (L - prob_host.q_len + i + 1)
        n_groups += 1
        if elapsed >= budget_s:
            break
    if decode_like:
        value, unit = done_bytes / elapsed / 1e9, "GB/s"
    else:
        value, unit = done_flops / elapsed / 1e12, "TFLOP/s"
    sample = (f"{n_groups} of {len(groups)} (sequence, kv head) groups, all their query rows "
              f"(prefill: up to 512 rows per group), {elapsed:.1f} s of oracle time")
    return value, unit, oracle.num_threads(), sample


def cpu_baseline(index, prob, decode_like, budget_s=12.0):
    try:
        host = prob.to("cpu")
        value, unit, cores, sample = oracle_sample(index, host, decode_like, budget_s)
        return {"value": round(value, 4), "unit": unit, "cores": cores, "kind": "oracle",
                "sample": sample}
    except Exception as exc:  # the baseline is reported, never fatal
        return {"value": None, "unit": None, "cores": os.cpu_count(), "kind": "oracle",
                "sample": f"failed: {exc}"}


def run_reference(args, world, rank):
    from exact_causal_gqa_gb300 import inputs
    if rank != 0:
        return None
    cfg = inputs.CONFIGS[args.config]
    prob = inputs.make_config(args.config, device="cpu")
    decode_like = prob.kind != "prefill"
    warm = max(3, args.warmup)
    per_step = max(0.5, 120.0 / (args.steps + warm))
    vals = []
    t_all = time.perf_counter()
    for k in range(warm + args.steps):
        value, unit, cores, sample = oracle_sample(args.config, prob, decode_like, per_step)
        if k >= warm:
            vals.append(value)
    wall = time.perf_counter() - t_all
    value = statistics.median(vals)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": warm,
        "ms_per_step": round(wall * 1e3 / (warm + args.steps), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded N(0,1) q/K/V, shuffled page pool)",
        "config": {"workload": cfg["name"], "kind": prob.kind},
        "cpu_baseline": {"value": round(value, 4), "unit": unit, "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    args = parse_args()
    world, rank, local = dist_env()
    if args.impl == "reference" or args.append or args.pool > 0:
        args.config = args.config or HEADLINE_CONFIG
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    else:
        if world > 1:
            torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
        fn = run_append if args.append else run_pool if args.pool > 0 else run_atlas
        line = fn(args, world, rank, local)
        if world > 1:
            torch.distributed.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
