#!/usr/bin/env python
"""Benchmark of the paged multi-token attention step on GB300.

One step = the whole hot path over one unified batch: paged KV append of the
batch's new tokens, host planning, the split-KV and tensor-core attention
kernels, the log-sum-exp merge, and a swap-out of one conversation's blocks to
pinned host memory on a side stream (the CPU cache tier), joined at the end.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--workloads all|none|a,b,...] [--impl ours|reference] [--kv-dtype bf16|fp8_e4m3]

Prints one JSON line on rank 0.  The headline (`value`, `e2e`, `roofline`) is
the Llama-2-70B grouped-query workload (`llama70b_gqa`, the largest amount of
attention work of the five workloads); `per_workload` repeats the measurement
for every workload.  For each workload:
  value     query tokens per second with inputs resident in HBM (device-timed
            with CUDA events, L2 flushed between steps);
  e2e       the same metric through the library's C ABI in a serving loop: every
            step's inputs are copied in from pinned host memory and its O/LSE
            copied out (pkv_copy_to_device / pkv_copy_to_host) inside the timed
            region, while the next step's inputs cross the link;
  e2e_replan  the same loop with the batch metadata changing every step (each
            decode's position moves), so the host plans every step inside the
            timed region;
  roofline  per attention kernel, from a pass that runs the two kernels one
            after the other so that each kernel's CUDA events bracket its own
            execution: algorithmic bytes and FLOPs per launch (planner
            statistics) over the launch's average duration, against
            MEASURED_PEAKS.json.
`cpu_baseline` times the CPU oracle on a bounded sample of the headline
workload.  With --gpus N under torchrun every rank runs its own replica of
the workload (weak scaling; no collective on the data path).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged multi-token attn: query tok/s, KV GB/s & TC util vs GB300 roofline"
UNIT = "query tok/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
HEADLINE = "llama70b_gqa"
ALL_WORKLOADS = ("tiny_mixed", "llama13b_mixed", "decode_lognormal", "llama70b_gqa", "long_skewed_evict")
REPLAN_VARIANTS = 8


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=HEADLINE, help="the headline workload")
    p.add_argument("--workloads", default="all",
                   help="workloads measured in per_workload: all, none, or a comma-separated list")
    p.add_argument("--e2e-steps", type=int, default=None)
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-oracle sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--swap-layers", type=int, default=4,
                   help="layers (one pool each) of the layer-pipelined swap-in measurement; 0 skips it")
    p.add_argument("--swap-steps", type=int, default=20)
    p.add_argument("--kv-dtype", choices=["bf16", "fp8_e4m3"], default="bf16", help="KV cache element type")
    return p.parse_args(argv)


# ----------------------------------------------------------------------------- multi-rank plumbing

def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate_ranks(tokens: float, seconds: float):
    """Whole-job totals: tokens summed over ranks, time = max over ranks (no-op on one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return tokens, seconds
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([tokens], dtype=torch.float64, device=dev)
    s = torch.tensor([seconds], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    dist.all_reduce(s, op=dist.ReduceOp.MAX)
    return float(t.item()), float(s.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ----------------------------------------------------------------------------- peaks, clocks, profiles

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


KERNEL_SOURCES = {"split_kv": "decode.cu", "tensor_core": "attn_tc.cu"}


def recorded_traffic(kernel: str, workload: str):
    """DRAM traffic per launch from the committed ncu summary, if it was taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    src = KERNEL_SOURCES.get(kernel)
    if not src or not os.path.exists(path):
        return None
    with open(os.path.join(ROOT, "paged_kv_attention_25_gb300", "csrc", src), "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()[:16]
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("source_sha256_16") != digest:
        return None
    try:
        return float(vals["dram_bytes_per_launch_full_size"])
    except (KeyError, ValueError):
        return None


def kernel_work(stats: dict, kernel: str):
    """Algorithmic bytes and FLOPs of one launch of an attention kernel (planner statistics)."""
    if kernel == "split_kv":
        return stats["decode_kv_bytes"] + stats["decode_io_bytes"], stats["decode_flops"]
    return stats["tc_kv_bytes"] + stats["tc_io_bytes"], stats["tc_flops"]


def kernel_roofline(stats: dict, kernel: str, avg_s: float, peaks: dict, peak_src: str, workload: str):
    """Roofline of one attention kernel: the binding roof is the larger of its HBM and tensor times."""
    nbytes, flops = kernel_work(stats, kernel)
    hbm = nbytes / avg_s / 1e9
    tfl = flops / avg_s / 1e12
    hbm_frac = hbm / peaks["hbm_gbs"]
    tc_frac = tfl / peaks["bf16_tflops"]
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    tensor = kernel == "tensor_core" and t_tc > t_hbm
    return {"kernel": kernel, "bound": "tensor" if tensor else "hbm",
            "achieved": tfl if tensor else hbm, "peak": peaks["bf16_tflops"] if tensor else peaks["hbm_gbs"],
            "unit": "TFLOP/s" if tensor else "GB/s", "frac": tc_frac if tensor else hbm_frac,
            "hbm_gbs": hbm, "hbm_frac": hbm_frac, "tflops": tfl, "tensor_frac": tc_frac,
            "roofline_frac": max(t_hbm, t_tc) / avg_s,
            "peak_source": f"{peak_src} (burst)", "avg_launch_us": avg_s * 1e6,
            "algorithmic_bytes": nbytes, "algorithmic_flops": flops,
            "traffic": recorded_traffic(kernel, workload)}


# ----------------------------------------------------------------------------- workload variants

def replan_variants(batch, n: int):
    """n variants of a batch's (ctx_lens, q_positions) that differ in every decode request.

    Variant v moves each one-token request's query position (and context end)
    back by v tokens, so the variants have distinct plans; multi-token requests
    are unchanged.  Every variant only reads keys the pool already holds."""
    q_lens = np.diff(batch.cu_q_lens)
    out = []
    for v in range(n):
        ctx = batch.ctx_lens.copy()
        pos = batch.q_positions.copy()
        for r in np.flatnonzero(q_lens == 1):
            s = min(v, int(ctx[r]) - 1)
            ctx[r] -= s
            pos[batch.cu_q_lens[r]] -= s
        out.append((ctx.astype(np.int32), pos.astype(np.int32)))
    return out


def config_of(batch, args):
    """The `config` object of the JSON line (the same for both arms)."""
    return {**batch.describe(), "kv_dtype": args.kv_dtype,
            "l2": "flushed between device-timed steps (258 MB write, then 258 MB read)",
            "parallelism": f"replicas x{args.gpus}"}


# ----------------------------------------------------------------------------- CPU oracle timing

FP8_SCALE = 2.0 ** -6   # k_scale = v_scale of the synthetic FP8 pools (codes span magnitudes 2 .. 240)


def oracle_pools(batch, kv_dtype: str):
    """The oracle's pools after the step's append (bf16 bits, or FP8 codes)."""
    import oracle
    from paged_kv_attention_25_gb300 import workloads as wl
    if kv_dtype == "fp8_e4m3":
        kp, vp = wl.fp8_pool_arrays(batch)
        oracle.append_fp8(kp, vp, FP8_SCALE, FP8_SCALE, batch.block_tables, batch.cu_q_lens, batch.q_positions,
                          batch.k_new, batch.v_new)
    else:
        kp, vp = batch.pool_arrays()
        oracle.append(kp, vp, batch.block_tables, batch.cu_q_lens, batch.q_positions, batch.k_new, batch.v_new)
    return kp, vp


def oracle_sample(batch, budget_s: float, kp=None, vp=None, kv_dtype: str = "bf16"):
    """Time the CPU oracle on a stratified sample of the batch's query tokens (all heads each).

    Returns (tokens_per_s, seconds, n_tokens, threads, description)."""
    import oracle
    oracle.build()
    if kp is None:
        kp, vp = oracle_pools(batch, kv_dtype)
    T, Hq = batch.num_tokens, batch.num_q_heads

    def run(tokens):
        t = np.repeat(tokens, Hq).astype(np.int32)
        h = np.tile(np.arange(Hq, dtype=np.int32), len(tokens))
        t0 = time.perf_counter()
        if kv_dtype == "fp8_e4m3":
            oracle.paged_attn_rows_fp8(batch.q, kp, vp, FP8_SCALE, FP8_SCALE, batch.block_tables, batch.ctx_lens,
                                       batch.cu_q_lens, batch.q_positions, batch.scale, t, h)
        else:
            oracle.paged_attn_rows(batch.q, kp, vp, batch.block_tables, batch.ctx_lens, batch.cu_q_lens,
                                   batch.q_positions, batch.scale, t, h)
        return time.perf_counter() - t0

    pilot_stride = max(1, T // 16)
    pilot = np.arange(0, T, pilot_stride)[:16]
    dt = run(pilot)
    per_tok = dt / len(pilot)
    n = int(max(1, min(T, budget_s / max(per_tok, 1e-9))))
    tokens = np.unique(np.linspace(0, T - 1, n).round().astype(np.int64))   # spread over the whole batch
    dt = run(tokens)
    desc = (f"{len(tokens)} of {T} query tokens (evenly spaced, all {Hq} heads) of {batch.name}; "
            f"fp64 C oracle")
    return len(tokens) / dt, dt, len(tokens), oracle.num_threads(), desc


def run_reference(args):
    world, rank, _ = dist_info()
    if rank != 0:
        return
    from paged_kv_attention_25_gb300 import workloads as wl
    batch = wl.WORKLOADS[args.workload]()
    kp, vp = oracle_pools(batch, args.kv_dtype)
    per_step = max(0.05, min(5.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(batch, per_step, kp, vp, args.kv_dtype)
    toks = secs = 0.0
    info = None
    for _ in range(args.steps):
        rate, dt, n, thr, desc = oracle_sample(batch, per_step, kp, vp, args.kv_dtype)
        toks += n
        secs += dt
        info = (thr, desc)
    value = toks / secs
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(batch, args),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": info[0], "kind": "oracle", "sample": info[1]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm

class Bench:
    """Device state shared by the workloads: streams, L2 flush buffers."""

    def __init__(self, args, dev):
        import torch
        self.args, self.dev = args, dev
        self.main = torch.cuda.current_stream()
        # The swap-out frees HBM for the next step, so a serving loop gives it
        # priority: its few CTAs are dispatched ahead of the attention CTAs
        # still waiting for an SM, and the copy runs beside the attention
        # instead of after it.
        self.side = torch.cuda.Stream(device=dev, priority=-1)
        self.flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        self.flush_r = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        self.flush_sum = torch.empty((), dtype=torch.float32, device=dev)

    def l2_flush(self):
        # Write a buffer twice the size of L2, then read another one, so that
        # each step starts with a cold L2 that holds no dirty lines of the flush
        # (whose write-back would otherwise land in the step).
        self.flush.zero_()
        self.flush_sum.copy_(self.flush_r.sum())


def measure_workload(B: Bench, name: str, headline: bool, rank: int, world: int):
    """Every measurement of one workload; returns (line fields, objects kept for the headline extras)."""
    import torch
    from paged_kv_attention_25_gb300 import pkv
    from paged_kv_attention_25_gb300 import workloads as wl

    args, dev, main, side = B.args, B.dev, B.main, B.side
    maker = wl.WORKLOADS[name]
    batch = maker() if world == 1 else maker(seed=maker.__defaults__[0] + 1000 * rank)
    fp8 = args.kv_dtype == "fp8_e4m3"
    kv_t = torch.uint8 if fp8 else torch.bfloat16
    pool_kw = {"dtype": args.kv_dtype, "k_scale": FP8_SCALE, "v_scale": FP8_SCALE} if fp8 else {}
    pool = pkv.Pool(batch.num_blocks, batch.num_kv_heads, batch.head_dim, device=dev, **pool_kw)
    (wl.fill_pool_fp8 if fp8 else wl.fill_pool)(batch, pool.k, pool.v)
    d = wl.upload(batch, dev)
    meta = pkv.HostMeta(batch.cu_q_lens, batch.ctx_lens, batch.q_positions)
    T, Hq, D = batch.num_tokens, batch.num_q_heads, batch.head_dim
    out = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, Hq), dtype=torch.float32, device=dev)
    ws = pool.workspace(pkv.pkv_paged_attn_workspace_size(pool, Hq, meta))

    # Swap-out target: the cached-history blocks (read-only in this step) of the
    # conversation with the median context, i.e. one conversation moved to the
    # CPU tier per step.
    q_lens = np.diff(batch.cu_q_lens)
    cand = np.flatnonzero(q_lens > 0)
    r_swap = int(cand[np.argsort(batch.ctx_lens[cand])[len(cand) // 2]])
    first_q = int(batch.q_positions[batch.cu_q_lens[r_swap]:batch.cu_q_lens[r_swap + 1]].min())
    swap_ids = batch.block_tables[r_swap, :max(1, first_q // 16)].astype(np.int32)
    swap_host = torch.empty((len(swap_ids), 2, batch.num_kv_heads, 16, D), dtype=kv_t).pin_memory()
    swap_bytes = swap_host.numel() * swap_host.element_size()
    begun = torch.cuda.Event()
    swapped = torch.cuda.Event()

    # The swap-out moves cached history that this step's append does not
    # write, so it starts with the step, beside the append.  fused: one
    # pkv_append_paged_attn call instead of pkv_append + pkv_paged_attn.
    def step(di=d, meta_=meta, o=out, l_=lse, fused=False):
        begun.record(main)
        side.wait_event(begun)
        pkv.pkv_swap_out(pool, swap_ids, swap_host, stream=side)
        swapped.record(side)
        if fused:
            pkv.pkv_append_paged_attn(pool, di["q"], di["q_positions"], di["block_tables"], di["ctx_lens"],
                                      di["cu_q_lens"], meta_, di["k_new"], di["v_new"], batch.scale, out=o, lse=l_,
                                      workspace=ws)
        else:
            pkv.pkv_append(pool, di["block_tables"], di["cu_q_lens"], di["q_positions"], di["k_new"], di["v_new"])
            pkv.pkv_paged_attn(pool, di["q"], di["q_positions"], di["block_tables"], di["ctx_lens"],
                               di["cu_q_lens"], meta_, batch.scale, out=o, lse=l_, workspace=ws)
        main.wait_event(swapped)

    for _ in range(max(3, args.warmup)):
        step()
        step(fused=True)
    torch.cuda.synchronize()
    if pkv.pkv_check_device_errors(pool) != 0:
        raise RuntimeError(f"{name}: device error word set during warm-up")

    def timed_steps(n, mode, fused=False):
        """n device-timed steps, L2 flushed between them; returns (per-step ms, kernel profile)."""
        pkv.pkv_profile_read(pool, reset=True)
        pkv.pkv_profile_enable(pool, mode)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        barrier()
        torch.cuda.synchronize()
        for i in range(n):
            B.l2_flush()
            starts[i].record(main)
            step(fused=fused)
            ends[i].record(main)
        torch.cuda.synchronize()
        barrier()
        pkv.pkv_profile_enable(pool, 0)
        prof = pkv.pkv_profile_read(pool, reset=True)
        if pkv.pkv_check_device_errors(pool) != 0:
            raise RuntimeError(f"{name}: device error word set during a timed region")
        return [s.elapsed_time(e) for s, e in zip(starts, ends)], prof

    # ---- value: K steps as a serving step runs them (the two attention kernels side by side)
    visible = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    gpu_index = int(visible[dev.index]) if dev.index < len(visible) and visible[dev.index].isdigit() else dev.index
    with ClockSampler(gpu_index) as clk:
        wall0 = time.perf_counter()
        step_ms, prof = timed_steps(args.steps, 1)
        wall1 = time.perf_counter()
    dev_s = sum(step_ms) / 1e3
    tokens_all, secs_all = aggregate_ranks(float(T * args.steps), dev_s)
    st = pkv.pkv_last_plan_stats(pool)
    # ---- per-kernel durations: the same steps with the two attention kernels one after the other
    ser_ms, ser_prof = timed_steps(max(10, args.steps // 2), 2)
    # ---- the fused step: pkv_append_paged_attn in place of the two calls
    fused_ms, fused_prof = timed_steps(args.steps, 1, fused=True)
    f_tok, f_sec = aggregate_ranks(float(T * args.steps), sum(fused_ms) / 1e3)
    fser_ms, fser_prof = timed_steps(max(10, args.steps // 2), 2, fused=True)

    # Host planning time for this batch, uncached (the step reuses its cached
    # plan while the batch metadata is unchanged): median of 5 plans.
    lib = pkv.load_library()
    n_items, plan_st, sms = ctypes.c_int(), pkv.pkv_plan_stats(), pkv.pkv_device_sm_count()
    plan_s = []
    for _ in range(5):   # one planner run each (the work items are counted, not copied out)
        p0 = time.perf_counter()
        rc = lib.pkv_plan_inspect(Hq, batch.num_kv_heads, D, sms, batch.num_reqs, T, ctypes.byref(meta.c), None, 0,
                                  ctypes.byref(n_items), ctypes.byref(plan_st))
        plan_s.append(time.perf_counter() - p0)
        if rc:
            raise RuntimeError(pkv.pkv_last_error())
    plan_host_us = 1e6 * float(np.median(plan_s))

    # ---- end to end through the C ABI: host inputs in, O/LSE out.
    # A serving loop: step i+1's inputs cross the link (copy stream `cin`)
    # while step i computes, and step i's O/LSE go back on `cout` (the link is
    # full duplex); inputs and outputs are double-buffered and events order the
    # reuse of each buffer.  Every step copies all of its inputs in and its
    # result out with pkv_copy_to_device / pkv_copy_to_host and runs the same
    # swap-out as the device-timed step; the timed region is the whole loop.
    # No L2 flush here: each step reads every visible KV block (hundreds of MB
    # for the bench workloads) and moves its inputs and outputs, several times
    # the 129 MB of L2, so no step finds the previous one's data in L2.
    e2e_steps = args.e2e_steps or max(10, args.steps // 4)
    host_in = {k: (v.cpu().pin_memory()) for k, v in d.items()}
    variants = replan_variants(batch, REPLAN_VARIANTS)
    host_var = [{"ctx_lens": torch.from_numpy(c).pin_memory(), "q_positions": torch.from_numpy(p).pin_memory()}
                for c, p in variants]
    meta_var = [pkv.HostMeta(batch.cu_q_lens, c, p) for c, p in variants]
    host_out = torch.empty_like(out, device="cpu").pin_memory()
    host_lse = torch.empty_like(lse, device="cpu").pin_memory()
    dev_in = [{k: torch.empty_like(v) for k, v in d.items()} for _ in range(2)]
    outs = [(torch.empty_like(out), torch.empty_like(lse)) for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = host_out.numel() * 2 + host_lse.numel() * 4
    cin, cout = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]     # step on slot s finished reading its inputs / writing O
    out_read = [torch.cuda.Event() for _ in range(2)]  # O/LSE of slot s copied to the host
    meta_e = pkv.HostMeta(host_in["cu_q_lens"].numpy(), host_in["ctx_lens"].numpy(), host_in["q_positions"].numpy())

    def copy_in(i, replan):
        s = i % 2
        cin.wait_event(done[s])
        for k in dev_in[s]:
            src = host_var[i % len(host_var)][k] if replan and k in ("ctx_lens", "q_positions") else host_in[k]
            pkv.pkv_copy_to_device(dev_in[s][k], src, stream=cin)
        in_ready[s].record(cin)

    def e2e_step(i, replan):
        s = i % 2
        di, (o_s, l_s) = dev_in[s], outs[s]
        main.wait_event(in_ready[s])
        main.wait_event(out_read[s])
        step(di, meta_var[i % len(meta_var)] if replan else meta_e, o_s, l_s)
        done[s].record(main)
        cout.wait_event(done[s])
        pkv.pkv_copy_to_host(host_out, o_s, stream=cout)
        pkv.pkv_copy_to_host(host_lse, l_s, stream=cout)
        out_read[s].record(cout)

    def e2e_loop(n, replan):
        # Step i is queued before step i+1's input copy: the copy engines take
        # transfers in order, so step i's small work-list upload must not sit
        # behind the next step's inputs (the big copy still runs during step i).
        copy_in(0, replan)
        for i in range(n):
            e2e_step(i, replan)
            if i + 1 < n:
                copy_in(i + 1, replan)
        main.wait_stream(cout)

    def e2e_timed(replan):
        for ev in done + out_read:
            ev.record(main)
        e2e_loop(3, replan)
        torch.cuda.synchronize()
        built0 = pkv.pkv_last_plan_stats(pool)["plans_built"]
        e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        e_start.record(main)
        e2e_loop(e2e_steps, replan)
        e_end.record(main)
        torch.cuda.synchronize()
        barrier()
        plans = pkv.pkv_last_plan_stats(pool)["plans_built"] - built0
        e_tok, e_sec = aggregate_ranks(float(T * e2e_steps), e_start.elapsed_time(e_end) / 1e3)
        if pkv.pkv_check_device_errors(pool) != 0:
            raise RuntimeError(f"{name}: device error word set in the end-to-end loop")
        return e_tok / e_sec, plans

    e2e_value, _ = e2e_timed(False)
    replan_value, replans = e2e_timed(True)

    peaks, peak_src = load_peaks()
    ser = {k: v for k, v in ser_prof.items() if k in KERNEL_SOURCES and v["launches"]}
    kname = name + ("_fp8" if fp8 else "")
    roofs = {k: kernel_roofline(st, k, v["total_ms"] / v["launches"] / 1e3, peaks, peak_src, kname)
             for k, v in ser.items()}
    # The kernel that dominates the step: the most device time in the pass
    # where each kernel runs alone.
    dom = max(ser, key=lambda k: ser[k]["total_ms"]) if ser else None
    step_ms_avg = 1e3 * secs_all / args.steps
    kv_bytes = st["decode_kv_bytes"] + st["tc_kv_bytes"]
    res = {
        "value": tokens_all / secs_all, "unit": UNIT, "ms_per_step": step_ms_avg,
        "config": config_of(batch, args),
        "kv_gbs": kv_bytes / (step_ms_avg / 1e3) / 1e9,
        "tflops": (st["decode_flops"] + st["tc_flops"]) / (step_ms_avg / 1e3) / 1e12,
        "kernels": {k: {"launches": v["launches"], "avg_us": 1e3 * v["total_ms"] / max(1, v["launches"])}
                    for k, v in prof.items()},
        "kernels_one_at_a_time": {k: {"launches": v["launches"], "avg_us": 1e3 * v["total_ms"] / max(1, v["launches"])}
                                  for k, v in ser_prof.items()},
        "ms_per_step_one_at_a_time": float(np.mean(ser_ms)),
        "roofline": roofs.get(dom),
        "roofline_per_kernel": roofs,
        "plan": {**{k: st[k] for k in ("num_decode_items", "num_tc_items", "num_merge_items")},
                 "host_plan_us_uncached": plan_host_us},
        "gpu_launches": int(sum(v["launches"] for v in prof.values())),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "path": "pkv_copy_to_device / pkv_copy_to_host from pinned host memory, copy engines"},
        "e2e_replan": {"value": replan_value, "unit": UNIT, "plans_built": int(replans), "steps": e2e_steps,
                       "variants": REPLAN_VARIANTS},
        "fused": {"value": f_tok / f_sec, "unit": UNIT, "ms_per_step": 1e3 * f_sec / args.steps,
                  "kernels": {k: {"launches": v["launches"], "avg_us": 1e3 * v["total_ms"] / max(1, v["launches"])}
                              for k, v in fused_prof.items()},
                  "kernels_one_at_a_time": {k: {"launches": v["launches"],
                                                "avg_us": 1e3 * v["total_ms"] / max(1, v["launches"])}
                                            for k, v in fser_prof.items()},
                  "ms_per_step_one_at_a_time": float(np.mean(fser_ms))},
        "clocks": clk.summary(),
        "wall_s_timed": wall1 - wall0,
        "swap_out_bytes_per_step": swap_bytes,
    }
    keep = {"batch": batch, "pool": pool, "ws": ws, "d": d, "meta": meta, "out": out, "lse": lse,
            "swap_ids": swap_ids, "swap_host": swap_host, "kv_t": kv_t, "pool_kw": pool_kw} if headline else None
    return res, keep


def headline_extras(B: Bench, k: dict):
    """Swap bandwidth and the layer-pipelined swap-in, on the headline workload."""
    import torch
    from paged_kv_attention_25_gb300 import pkv
    args, dev, main = B.args, B.dev, B.main
    batch, pool, d, meta = k["batch"], k["pool"], k["d"], k["meta"]
    D, Hq = batch.head_dim, batch.num_q_heads
    swap_ids, swap_host = k["swap_ids"], k["swap_host"]

    # ---- swap bandwidth alone (both directions, pinned host)
    ids = batch.used_blocks[:min(len(batch.used_blocks), 4096)].astype(np.int32)
    sh = torch.empty((len(ids), 2, batch.num_kv_heads, 16, D), dtype=k["kv_t"]).pin_memory()
    pkv.pkv_swap_out(pool, ids, sh)
    torch.cuda.synchronize()
    e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    e0.record(main)
    pkv.pkv_swap_out(pool, ids, sh)
    e1.record(main)
    pkv.pkv_swap_in(pool, ids, sh)
    e2.record(main)
    torch.cuda.synchronize()
    swap_bw_bytes = sh.numel() * sh.element_size()
    swap = {"out_gbs": swap_bw_bytes / (e0.elapsed_time(e1) / 1e3) / 1e9,
            "in_gbs": swap_bw_bytes / (e1.elapsed_time(e2) / 1e3) / 1e9, "bytes": swap_bw_bytes}
    del sh

    # ---- layer-pipelined swap-in.  L layers, each its own pool holding the
    # same KV, each getting back the step's swapped-out conversation history
    # (swap_ids, swapped in from a pinned host copy of the same blocks, so the
    # attention inputs do not change).  Three ways of running a step:
    #   compute: every layer's append + attention, no swap-in;
    #   serial:  per layer, the swap kernel brings the blocks in, then append +
    #            attention (the swap-in sits on the critical path);
    #   ahead:   every layer's pkv_swap_in_ahead on one copy stream at the
    #            start of the step, then the layers in order, each waiting only
    #            for its own blocks.
    pipe = None
    if args.swap_layers > 0:
        layers = [(pool, k["ws"])]
        for _ in range(args.swap_layers - 1):
            p = pkv.Pool(batch.num_blocks, batch.num_kv_heads, D, device=dev, **k["pool_kw"])
            p.k.copy_(pool.k)
            p.v.copy_(pool.v)
            layers.append((p, p.workspace(pkv.pkv_paged_attn_workspace_size(p, Hq, meta))))
        hosts = [torch.empty_like(swap_host).pin_memory() for _ in layers]
        for (p, _), h in zip(layers, hosts):
            pkv.pkv_swap_out(p, swap_ids, h)
        cstream = torch.cuda.Stream(device=dev)
        torch.cuda.synchronize()

        def layer_step(p, w):
            pkv.pkv_append(p, d["block_tables"], d["cu_q_lens"], d["q_positions"], d["k_new"], d["v_new"])
            pkv.pkv_paged_attn(p, d["q"], d["q_positions"], d["block_tables"], d["ctx_lens"], d["cu_q_lens"],
                               meta, batch.scale, out=k["out"], lse=k["lse"], workspace=w)

        def run_mode(mode):
            if mode == "ahead":
                for (p, _), h in zip(layers, hosts):
                    pkv.pkv_swap_in_ahead(p, swap_ids, h, cstream, stream=main)
            for (p, w), h in zip(layers, hosts):
                if mode == "serial":
                    pkv.pkv_swap_in(p, swap_ids, h)
                layer_step(p, w)

        modes = ("compute", "serial", "ahead")
        for m in modes:
            for _ in range(3):
                run_mode(m)
        torch.cuda.synchronize()
        times = {m: [] for m in modes}
        for i in range(args.swap_steps):
            for m in modes:   # interleaved, so that clock drift hits every mode alike
                B.l2_flush()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(main)
                run_mode(m)
                b.record(main)
                times[m].append((a, b))
        torch.cuda.synchronize()
        ms = {m: float(np.median([a.elapsed_time(b) for a, b in times[m]])) for m in modes}
        for p, _ in layers:
            if pkv.pkv_check_device_errors(p) != 0:
                raise RuntimeError("device error word set in the swap-in pipeline")
        exposed = ms["serial"] - ms["compute"]
        pipe = {"layers": len(layers), "swap_in_bytes_per_layer": swap_host.numel() * swap_host.element_size(),
                "steps": args.swap_steps, "ms_per_step_median": ms,
                "swap_in_hidden_frac": (ms["serial"] - ms["ahead"]) / exposed if exposed > 0 else None}
        for p, _ in layers[1:]:
            p.close()
        del layers, hosts
    return swap, pipe


def run_ours(args):
    import torch
    import torch.distributed as dist
    from paged_kv_attention_25_gb300 import build as pkv_build

    world, rank, local = dist_info()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    if rank == 0:
        pkv_build.build()
    barrier()
    pkv_build.build()   # no-op when fresh; other ranks wait for rank 0 above
    args.gpus = world
    B = Bench(args, dev)

    head, keep = measure_workload(B, args.workload, True, rank, world)
    swap, pipe = headline_extras(B, keep)
    batch = keep["batch"]
    keep["pool"].close()
    del keep
    torch.cuda.empty_cache()

    if args.workloads == "all":
        names = list(ALL_WORKLOADS)
    elif args.workloads == "none":
        names = []
    else:
        names = [n for n in args.workloads.split(",") if n]
    keys = ("value", "ms_per_step", "e2e", "e2e_replan", "fused", "roofline_per_kernel", "kernels_one_at_a_time",
            "plan", "kv_gbs", "tflops")
    per = {args.workload: {k: head[k] for k in keys}}
    from paged_kv_attention_25_gb300 import pkv
    for n in names:
        if n == args.workload:
            continue
        try:
            r, _ = measure_workload(B, n, False, rank, world)
        except pkv.PkvError as e:
            if e.code != pkv.PKV_EUNSUPPORTED:
                raise
            per[n] = {"unsupported": str(e)}
            torch.cuda.empty_cache()
            continue
        per[n] = {k: r[k] for k in keys}
        per[n]["config"] = r["config"]
        torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    fp8 = args.kv_dtype == "fp8_e4m3"
    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8_e4m3 KV, bf16 Q/O, fp32 softmax" if fp8 else "bf16",
        "data": "synthetic", "config": head["config"],
        "kv_gbs": head["kv_gbs"], "tflops": head["tflops"], "kernels": head["kernels"],
        "kernels_one_at_a_time": head["kernels_one_at_a_time"],
        "ms_per_step_one_at_a_time": head["ms_per_step_one_at_a_time"],
        "plan": head["plan"], "gpu_launches": head["gpu_launches"],
        "roofline": head["roofline"], "roofline_per_kernel": head["roofline_per_kernel"],
        "e2e": head["e2e"], "e2e_replan": head["e2e_replan"], "fused": head["fused"],
        "swap": swap, "swap_in_pipeline": pipe, "swap_out_bytes_per_step": head["swap_out_bytes_per_step"],
        "clocks": head["clocks"], "wall_s_timed": head["wall_s_timed"],
        "per_workload": per,
    }
    if world == 1 and not args.no_cpu_baseline:
        rate, dt, n, thr, desc = oracle_sample(batch, args.cpu_seconds, kv_dtype=args.kv_dtype)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": desc,
                                "seconds": dt}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
