#!/usr/bin/env python3
"""Benchmark of the paged KV-cache attention hot path on GB300.

Headline (one JSON line on stdout, rank 0): the Qwen3-8B-shaped single-layer
decode step -- batch 64, 32 Q heads, 8 KV heads, head_dim 128, block 16,
bf16, context lengths uniform on [128, 2048], pool 1.5x the blocks needed --
where one step is the store of the 64 new tokens (pd_reshape_and_cache) and
split-context decode attention, pieces merged in-kernel (pd_paged_attention_decode).
``value`` is the step's algorithmic bytes (K/V read once, q, out, tables and
the stored tokens) per second of device time, inputs resident in HBM, L2
flushed (256 MiB read) before every timed step.

The same line carries: the roofline of the dominant kernel (decode) against
the measured HBM copy bandwidth, the end-to-end figure through the public API
with host buffers, the float64 oracle timed on the host cores, launch count,
clocks sampled during the run, and (N=1) the other workloads: the 32-layer
long-context stack, the chunked-prefill mix (prefill TFLOP/s on the tensor
cores) and the copy-on-write fork stress.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
N > 1 runs under torch.distributed.run, one process per GPU, each on its own
replica of the batch (weak scaling, no collective on the data path).
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("Paged decode-attn achieved HBM GB/s (% of GB300 peak); KV tokens/s; "
          "prefill TFLOP/s")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# GB300's nominal figures (context beside the measured denominators)
NOMINAL_HBM_GBS = 7900.0
NOMINAL_BF16_TFLOPS = 2250.0
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true", help="headline workload only")
    ap.add_argument("--extras", default="chunked_prefill_mix,long_context_32_layers,cow_fork_stress,fp8_decode,"
                    "spec_verify,kv_handover,prefix_cache",
                    help="comma-separated extra workloads to run after the headline")
    ap.add_argument("--extra-steps", type=int, default=10)
    ap.add_argument("--long-context-layers", type=int, default=32,
                    help="layers of the long-context extra (32 = the workload; fewer only "
                         "to profile a layer's launch on a smaller device footprint)")
    ap.add_argument("--only-extras", action="store_true",
                    help="run only the --extras workloads and print their results (for "
                         "profiling one kernel); not a benchmark line")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return (float(p["hbm_gbs"]), float(p["bf16_tflops"]),
                float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured")
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS, "fallback"


def code_text(src: str) -> str:
    """C++/CUDA source without its comments, whitespace runs folded to one
    space: two sources with the same code_text compile to the same kernels."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == "/" and src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif c == "/" and src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_sha(*names) -> str:
    """First 16 hex digits of sha256 over the code (comments and whitespace
    aside) of the named files under csrc/, in order."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "paged_kv_attention_26_gb300", "csrc", n)) as f:
            h.update(code_text(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, sha: str):
    """DRAM bytes per launch recorded from an ncu capture in profiles/*.md
    (line 'traffic: kernel=<k> source_sha=<sha> bytes_per_launch=<n>'); None
    when absent or when the kernel source changed since the capture."""
    pat = re.compile(r"traffic: kernel=(\S+) source_sha=(\S+) bytes_per_launch=(\d+)")
    d = os.path.join(ROOT, "profiles")
    if not os.path.isdir(d):
        return None
    for n in sorted(os.listdir(d)):
        if not n.endswith((".md", ".txt")):
            continue
        with open(os.path.join(d, n)) as f:
            for line in f:
                m = pat.search(line)
                if m and m.group(1) == kernel and m.group(2) == sha:
                    return int(m.group(3))
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        sm.sort()
        loaded = [s for s in sm if s > 0.5 * mx] or sm
        return {"sm_mhz": loaded[len(loaded) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------------
# ranks: one replica of the workload per GPU (independent batches, no exchange)

def rank_max(seconds: float, world: int, device) -> float:
    """The slowest rank's timed seconds, on every rank (the job ends when the
    last replica does)."""
    if world <= 1:
        return seconds
    import torch
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(bytes_per_step: int, steps: int, seconds: float, world: int) -> float:
    """GB/s of the whole job: every rank moved bytes_per_step per step of its
    own batch, and the job took the slowest rank's time."""
    return world * bytes_per_step * steps / seconds / 1e9


# ---------------------------------------------------------------------------------
# workload accounting

def decode_alg_bytes(ctx, B, H, Hk, D, S, elem=2):
    """K/V read once + q read + out written + block-table entries read."""
    kv = int(sum(ctx)) * Hk * D * elem * 2
    qo = 2 * B * H * D * elem
    tables = sum((c + S - 1) // S for c in ctx) * 4
    return kv, kv + qo + tables


def store_alg_bytes(T, Hk, D, elem=2):
    return 2 * (2 * T * Hk * D * elem) + T * 8     # K,V read + written, slots read


# ---------------------------------------------------------------------------------

def run_ours(args, rank, world, local_rank):
    import torch
    import paged_kv_attention_26_gb300 as pd
    import pd_inputs

    pd.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    hbm_peak, bf16_peak, bf16_sust, peak_src = peaks()
    sampler = ClockSampler(local_rank) if rank == 0 else None
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush():
        # Evict L2 by reading a buffer twice its size.  Reading leaves clean
        # lines; writing would leave dirty ones that the next kernel pays to
        # write back.
        flush_buf.sum()

    stream = torch.cuda.current_stream()

    # ---- headline: Qwen3-8B-shaped decode step --------------------------------------
    c = pd_inputs.qwen3_8b_decode(seed=rank)
    B, H, Hk, D, S = c.B, c.H, c.Hk, c.D, c.pool.S
    ctx = c.pool.context_lens.tolist()
    mcl = c.max_context_len
    kc, vc = c.pool.key_cache.to(dev), c.pool.value_cache.to(dev)
    q = c.q.to(dev)
    bt = c.pool.block_tables.to(dev)
    cl = c.pool.context_lens.to(dev)
    nk, nv = c.new_key.to(dev), c.new_value.to(dev)
    slots = c.slot_mapping.to(dev)
    out = torch.empty_like(q)
    ws = pd.decode_workspace(B, H, D, mcl, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kv_bytes, dec_bytes = decode_alg_bytes(ctx, B, H, Hk, D, S)
    st_bytes = store_alg_bytes(B, Hk, D)
    step_bytes = dec_bytes + st_bytes

    def step():
        # one kernel: each sequence's new row is stored by the decode CTA that
        # copies its block, right before the copy
        pd.pd_decode_step_fused(out, q, kc, vc, bt, cl, mcl, c.scale, nk, nv, slots,
                                workspace=ws, dev_err=err)

    def two_kernel_step():
        pd.pd_decode_step(out, q, kc, vc, bt, cl, mcl, c.scale, nk, nv, slots, workspace=ws,
                          dev_err=err)

    def decode_only():
        pd.pd_paged_attention_decode(out, q, kc, vc, bt, cl, mcl, c.scale, ws, dev_err=err)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()

    def timed(fn):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        n0 = pd.launch_count()
        t0 = time.perf_counter()
        for i in range(args.steps):
            flush()
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        n = pd.launch_count() - n0
        if world > 1:
            torch.distributed.barrier()
        return sum(a.elapsed_time(b) for a, b in ev) * 1e-3, wall, n

    # the headline: whole decode steps (the store inside the decode)
    with nvtx_range("decode_step"):
        step_s, t_wall, launches = timed(step)
    # the same step as two grids (store, then decode as a programmatic dependent)
    with nvtx_range("decode_step_two_kernels"):
        for _ in range(args.warmup):
            flush()
            two_kernel_step()
        two_s, _, _ = timed(two_kernel_step)
    # the roofline's kernel alone: the same decode launched by itself
    with nvtx_range("decode_alone"):
        for _ in range(args.warmup):
            flush()
            decode_only()
        dec_s, _, _ = timed(decode_only)
    step_s = rank_max(step_s, world, dev)
    assert err.item() == 0, f"device error word {err.item()}"
    value = whole_job_value(step_bytes, args.steps, step_s, world)
    ms_per_step = step_s / args.steps * 1e3
    dec_avg = dec_s / args.steps
    achieved = dec_bytes / dec_avg / 1e9
    sha = source_sha("decode.cu", "pd_device.cuh")
    traffic = profiled_traffic("paged_decode", sha)

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "qwen3_8b_decode_step", "batch": B, "q_heads": H, "kv_heads": Hk,
                   "head_dim": D, "block_size": S, "context_lens": "uniform [128, 2048], seed 0",
                   "kv_tokens": int(sum(ctx)), "pool_blocks": c.pool.NB,
                   "step": "pd_decode_step_fused: one launch; the decode CTA that copies a "
                           "sequence's last block first stores the sequence's new K/V row at "
                           "its slot (the slot is checked against the table), then the "
                           "split-context decode with its in-kernel merge",
                   "l2": "inputs larger than L2 (KV 321 MB vs 129 MB L2), and L2 flushed "
                         "before every timed step by reading a 256 MiB buffer",
                   "parallelism": f"replicas x{world}"},
        "pct_of_hbm_peak": round(100 * value / world / hbm_peak, 2),
        "pct_of_nominal_hbm_peak": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "kv_tokens_per_s": round(world * sum(ctx) * args.steps / step_s, 1),
        "roofline": {"kernel": "paged_decode_split_kernel", "bound": "hbm",
                     "achieved": round(achieved, 2), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "peak_source": peak_src,
                     "nominal_peak": NOMINAL_HBM_GBS,
                     "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "alg_bytes_per_launch": dec_bytes,
                     "timing": "the decode launched alone, steps x (L2 flush, launch), CUDA "
                               "events on the launching stream",
                     "traffic": traffic, "traffic_source_sha": sha},
        "gpu_launches": launches,
        "wall_s_timed_loop": round(t_wall, 4),
        "two_kernel_step_ms": round(rank_max(two_s, world, dev) / args.steps * 1e3, 5),
        "two_kernel_step": "pd_decode_step: the store grid, then the decode as its "
                           "programmatic dependent (same result, same bytes)",
    }

    # every rank runs its replica host to host; the job takes the slowest
    with nvtx_range("e2e"):
        e2e = e2e_decode(pd, c, dev, args, step_bytes, world)
    if rank == 0:
        result["e2e"] = e2e
    if rank == 0 and world == 1:
        step()                                   # the output of one whole step, for parity
        torch.cuda.synchronize()
        result["cpu_baseline"] = cpu_baseline_decode(c, step_bytes, gpu_out=out)
        result["parity"] = result["cpu_baseline"].pop("parity")
    wanted = [] if args.no_extras else [x for x in args.extras.split(",") if x]
    if world == 1 and wanted:
        del kc, vc
        torch.cuda.empty_cache()
        extras = run_extras(pd, pd_inputs, dev, args, flush, wanted, hbm_peak, bf16_peak,
                            peak_src)
        if "chunked_prefill_mix" in extras:
            pm = extras["chunked_prefill_mix"]
            result["prefill_tflops"] = pm["prefill_tflops"]
            result["prefill_pct_of_bf16_peak"] = round(100 * pm["prefill_frac"], 2)
        result["extras"] = extras
    if sampler is not None:
        result["clocks"] = sampler.stop()
    return result


class nvtx_range:
    """An NVTX range around one bench phase (seen by nsys/ncu timelines)."""

    def __init__(self, name):
        self.name = name

    def __enter__(self):
        import torch
        torch.cuda.nvtx.range_push(self.name)

    def __exit__(self, *exc):
        import torch
        torch.cuda.nvtx.range_pop()
        return False


def run_extras(pd, pd_inputs, dev, args, flush, wanted, hbm_peak, bf16_peak, peak_src):
    extras = {}
    with nvtx_range("extras"):
        _run_extras(extras, pd, pd_inputs, dev, args, flush, wanted, hbm_peak, bf16_peak,
                    peak_src)
    return extras


def _run_extras(extras, pd, pd_inputs, dev, args, flush, wanted, hbm_peak, bf16_peak, peak_src):
    if "chunked_prefill_mix" in wanted:
        extras["chunked_prefill_mix"] = bench_prefill_mix(pd, pd_inputs, dev, args, flush,
                                                          bf16_peak, hbm_peak, peak_src)
    if "long_context_32_layers" in wanted:
        extras["long_context_32_layers"] = bench_long_context(pd, pd_inputs, dev, args,
                                                               flush, hbm_peak)
    if "cow_fork_stress" in wanted:
        extras["cow_fork_stress"] = bench_cow(pd, pd_inputs, dev, args, flush, hbm_peak)
    if "fp8_decode" in wanted:
        extras["fp8_decode"] = bench_fp8_decode(pd, pd_inputs, dev, args, flush, hbm_peak)
    if "spec_verify" in wanted:
        extras["spec_verify"] = bench_spec_verify(pd, pd_inputs, dev, args, flush, hbm_peak,
                                                  bf16_peak)
    if "kv_handover" in wanted:
        extras["kv_handover"] = bench_kv_handover(pd, pd_inputs, dev, args, flush, hbm_peak)
    if "prefix_cache" in wanted:
        extras["prefix_cache"] = bench_prefix_cache(pd, args)


def run_only_extras(args):
    """The --extras workloads alone, on cuda:0 (a profiling aid)."""
    import torch
    import paged_kv_attention_26_gb300 as pd
    import pd_inputs
    pd.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    hbm_peak, bf16_peak, _, peak_src = peaks()
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    wanted = [x for x in args.extras.split(",") if x]
    return {"only_extras": run_extras(pd, pd_inputs, dev, args, lambda: flush_buf.sum(), wanted,
                                      hbm_peak, bf16_peak, peak_src)}


def e2e_decode(pd, c, dev, args, step_bytes, world=1):
    """The same step through the public API from pinned host memory:
    ``DecodeStep(fused=True)`` (one pinned buffer holding q, the new K/V,
    slots, block tables and context lengths, all read by the kernel over the
    host link, and ``out`` written back the same way, synchronize), replayed
    from a CUDA graph; the same object run eagerly is reported beside it."""
    import torch
    kc, vc = c.pool.key_cache.to(dev), c.pool.value_cache.to(dev)
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    res = {}
    for graph in (True, False):
        st = pd.DecodeStep(kc, vc, c.B, c.H, c.B, c.pool.block_tables.shape[1],
                           c.max_context_len, c.scale, c.dtype, graph=graph, fused=True)
        h = st.host
        h["q"].copy_(c.q)
        h["key"].copy_(c.new_key)
        h["value"].copy_(c.new_value)
        h["slot_mapping"].copy_(c.slot_mapping)
        h["block_tables"].copy_(c.pool.block_tables)
        h["context_lens"].copy_(c.pool.context_lens)
        for _ in range(args.warmup):
            st()
        total = 0.0
        for _ in range(args.steps):
            flush_buf.sum()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            st()
            total += time.perf_counter() - t0
        assert st.dev_err.item() == 0
        res[graph] = (total, st.h2d_bytes, st.d2h_bytes)
        del st
    total, h2d, d2h = res[True]
    eager = res[False][0]
    if world > 1:
        torch.distributed.barrier()
    total = rank_max(total, world, dev)
    eager = rank_max(eager, world, dev)
    return {"value": round(whole_job_value(step_bytes, args.steps, total, world), 2), "unit": "GB/s",
            "ms_per_step": round(total / args.steps * 1e3, 4),
            "h2d_bytes_per_step": h2d * world, "d2h_bytes_per_step": d2h * world,
            "path": "DecodeStep replayed from a CUDA graph: pd_decode_step_fused reading q, the "
                    "new K/V, the slots, the block tables and the context lengths from one "
                    "pinned host buffer and writing out into pinned host memory over the "
                    "host link, synchronize; host wall clock per step, L2 flushed before "
                    "each; the byte counts are every input and output byte of the step",
            "eager_value": round(whole_job_value(step_bytes, args.steps, eager, world), 2),
            "eager_ms_per_step": round(eager / args.steps * 1e3, 4)}


def cpu_baseline_decode(c, step_bytes, gpu_out=None, budget_s=8.0):
    """The float64 oracle (as it stands) on this host's cores, on the same step:
    store + decode of all 64 sequences, repeated until ``budget_s`` elapsed, on
    all cores and then on one core.  When ``gpu_out`` (the GPU step's output)
    is given, the oracle's result of the same step also gives the headline's
    parity record: max-abs and max-rel error and the count of elements outside
    |gpu - oracle| <= 2e-3 + 1e-2 |oracle|."""
    import numpy as np
    import torch
    import oracle
    threads = oracle.default_threads()
    kc0 = c.pool.key_cache.view(torch.int16).numpy().view(np.uint16)
    vc0 = c.pool.value_cache.view(torch.int16).numpy().view(np.uint16)

    def run(nthreads, max_reps):
        reps, total, ref = 0, 0.0, None
        while (total < budget_s or reps == 0) and reps < max_reps:
            kc, vc = kc0.copy(), vc0.copy()
            t0 = time.perf_counter()
            oracle.reshape_and_cache(c.new_key, c.new_value, kc, vc, c.slot_mapping, c.pool.S)
            ref = oracle.decode(c.q, kc, vc, c.pool.block_tables, c.pool.context_lens, c.scale,
                                oracle.BF16, threads=nthreads)
            total += time.perf_counter() - t0
            reps += 1
        return reps, total, ref

    reps, total, ref = run(threads, 50)
    reps1, total1, _ = run(1, 10)
    res = {"value": round(step_bytes * reps / total / 1e9, 4), "unit": "GB/s",
           "cores": threads, "kind": "oracle",
           "sample": f"{reps} full steps (store + decode of all 64 sequences), "
                     f"{total:.1f} s on {threads} threads",
           "one_core": {"value": round(step_bytes * reps1 / total1 / 1e9, 4), "unit": "GB/s",
                        "cores": 1,
                        "sample": f"{reps1} full steps, {total1:.1f} s on 1 thread"}}
    if gpu_out is not None:
        g = gpu_out.detach().cpu().double().numpy().reshape(ref.shape)
        err = np.abs(g - ref)
        big = np.abs(ref) >= 1e-3                 # relative error where it means something
        res["parity"] = {
            "elements": int(err.size),
            "max_abs": float(err.max()),
            "max_rel": float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0,
            "failing": int((~(err <= 2e-3 + 1e-2 * np.abs(ref))).sum()),
            "tolerance": "|gpu - oracle| <= 2e-3 + 1e-2 |oracle|; max_rel over |oracle| >= 1e-3"}
    return res


def _time_calls(fn, n, flush, warm=3):
    import torch
    for _ in range(warm):
        flush()
        fn()
    torch.cuda.synchronize()
    # every call is enqueued behind its L2 flush before any is waited for, so
    # the host's launch overhead hides behind the flush and the events time the
    # device work alone
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    for a, b in ev:
        flush()
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    ts = [a.elapsed_time(b) * 1e-3 for a, b in ev]
    # mean without the slowest tenth of the calls (at least one when n >= 5): a
    # single call held up by something else on the machine should not move the
    # figure of a workload that runs in tens of microseconds
    ts.sort()
    keep = ts[:len(ts) - (max(1, len(ts) // 10) if len(ts) >= 5 else 0)]
    return sum(keep) / len(keep)


def bench_prefill_mix(pd, pd_inputs, dev, args, flush, bf16_peak, hbm_peak, peak_src):
    import torch
    m = pd_inputs.chunked_prefill_mixed()
    kc, vc = m.pool.key_cache.to(dev), m.pool.value_cache.to(dev)
    nk, nv, sl = m.new_key.to(dev), m.new_value.to(dev), m.slot_mapping.to(dev)
    q = m.q_prefill.to(dev)
    out = torch.empty_like(q)
    cu = m.cu_q_lens.to(dev)
    btp, clp = m.pool.block_tables[:m.Bp].to(dev), m.pool.context_lens[:m.Bp].to(dev)
    btd, cld = m.pool.block_tables[m.Bp:].to(dev), m.pool.context_lens[m.Bp:].to(dev)
    qd = m.q_decode.to(dev)
    od = torch.empty_like(qd)
    mcl = int(cld.max())
    ws = pd.decode_workspace(m.Bd, m.H, m.D, mcl, device=dev)
    P = m.prior_lens.double()
    C = (m.cu_q_lens[1:] - m.cu_q_lens[:-1]).double()
    flops = float(4 * m.D * m.H * (C * P + C * (C + 1) / 2).sum())
    dctx = m.pool.context_lens[m.Bp:].tolist()
    _, dbytes = decode_alg_bytes(dctx, m.Bd, m.H, m.Hk, m.D, m.pool.S)
    sbytes = store_alg_bytes(sl.numel(), m.Hk, m.D)
    n = args.extra_steps
    t_store = _time_calls(lambda: pd.pd_reshape_and_cache(nk, nv, kc, vc, sl), n, flush)
    t_pre = _time_calls(lambda: pd.pd_paged_prefill_chunk(out, q, cu, m.max_q_len, kc, vc, btp,
                                                          clp, m.scale), n, flush)
    t_dec = _time_calls(lambda: pd.pd_paged_attention_decode(od, qd, kc, vc, btd, cld, mcl,
                                                             m.scale, ws), n, flush)

    def whole():
        pd.pd_reshape_and_cache(nk, nv, kc, vc, sl)
        pd.pd_paged_prefill_chunk(out, q, cu, m.max_q_len, kc, vc, btp, clp, m.scale)
        pd.pd_paged_attention_decode(od, qd, kc, vc, btd, cld, mcl, m.scale, ws)

    t_step = _time_calls(whole, n, flush)
    return {"workload": "16 prefill chunks of 512 (prior U[0,8192]) + 48 decode (ctx U[256,4096])",
            "step_ms": round(t_step * 1e3, 4),
            "prefill_ms": round(t_pre * 1e3, 4), "prefill_gflop": round(flops / 1e9, 2),
            "prefill_tflops": round(flops / t_pre / 1e12, 2),
            "prefill_frac": round(flops / t_pre / 1e12 / bf16_peak, 4),
            "prefill_frac_of_nominal": round(flops / t_pre / 1e12 / NOMINAL_BF16_TFLOPS, 4),
            "prefill_peak_tflops": bf16_peak, "peak_source": peak_src,
            "store_tokens": sl.numel(), "store_gbs": round(sbytes / t_store / 1e9, 1),
            "decode_ms": round(t_dec * 1e3, 4), "decode_gbs": round(dbytes / t_dec / 1e9, 1),
            "decode_frac": round(dbytes / t_dec / 1e9 / hbm_peak, 4)}


def bench_long_context(pd, pd_inputs, dev, args, flush, hbm_peak):
    import torch
    res = {}
    nl = args.long_context_layers
    for point, (B, ctx) in enumerate(pd_inputs.LONG_CONTEXT_POINTS):
        layers = []
        for layer in range(nl):
            lc = pd_inputs.long_context_layer(point, layer, device=dev)
            layers.append((lc.pool.key_cache, lc.pool.value_cache, lc.q))
        bt = lc.pool.block_tables.to(dev)
        cl = lc.pool.context_lens.to(dev)
        outs = [torch.empty_like(x[2]) for x in layers]
        ws = pd.decode_workspace(B, lc.H, lc.D, ctx, device=dev)

        def step():
            for (k, v, q), o in zip(layers, outs):
                pd.pd_paged_attention_decode(o, q, k, v, bt, cl, ctx, lc.scale, ws)

        t = _time_calls(step, max(3, args.extra_steps // 2), flush, warm=2)
        kv, alg = decode_alg_bytes([ctx] * B, B, lc.H, lc.Hk, lc.D, lc.pool.S)
        res[f"{B}x{ctx}"] = {"layers": nl, "step_ms": round(t * 1e3, 3),
                             "gbs": round(nl * alg / t / 1e9, 1),
                             "frac": round(nl * alg / t / 1e9 / hbm_peak, 4),
                             "kv_tokens_per_s": round(nl * B * ctx / t, 1),
                             "partitions": -(-ctx // pd.pd_decode_partition_tokens(ctx))}
        del layers, outs
        torch.cuda.empty_cache()
    return res


def bench_fp8_decode(pd, pd_inputs, dev, args, flush, hbm_peak):
    """The headline Qwen3-8B batch with E4M3 pools (one byte per K/V value, per-head
    scales): algorithmic bytes = FP8 K/V + q + out + block tables."""
    import torch
    c = pd_inputs.qwen3_8b_decode(seed=0)
    kc8, vc8, ks, vs = pd_inputs.fp8_pools(c.pool.key_cache, c.pool.value_cache)
    kc8, vc8, ks, vs = kc8.to(dev), vc8.to(dev), ks.to(dev), vs.to(dev)
    q = c.q.to(dev)
    out = torch.empty_like(q)
    bt, cl = c.pool.block_tables.to(dev), c.pool.context_lens.to(dev)
    mcl = c.max_context_len
    ws = pd.decode_workspace(c.B, c.H, c.D, mcl, device=dev)
    pd.pd_reshape_and_cache_fp8(c.new_key.to(dev), c.new_value.to(dev), kc8, vc8,
                                c.slot_mapping.to(dev), ks, vs)
    t = _time_calls(lambda: pd.pd_paged_attention_decode_fp8(out, q, kc8, vc8, ks, vs, bt, cl, mcl,
                                                             c.scale, ws), args.extra_steps, flush)
    nk, nv, sl = c.new_key.to(dev), c.new_value.to(dev), c.slot_mapping.to(dev)
    ts = _time_calls(lambda: pd.pd_decode_step(out, q, kc8, vc8, bt, cl, mcl, c.scale, nk, nv, sl,
                                               workspace=ws, k_scale=ks, v_scale=vs),
                     args.extra_steps, flush)
    ctx = c.pool.context_lens.tolist()
    kv = sum(ctx) * c.Hk * c.D * 2                 # one byte per K and per V value
    other = 2 * c.B * c.H * c.D * 2 + sum(4 * -(-x // c.pool.S) for x in ctx)
    res = {"workload": "qwen3_8b_decode_step, E4M3 K/V with per-head scales",
           "ms": round(t * 1e3, 4), "gbs": round((kv + other) / t / 1e9, 1),
           "frac": round((kv + other) / t / 1e9 / hbm_peak, 4),
           "kv_tokens_per_s": round(sum(ctx) / t, 1),
           "step_ms": round(ts * 1e3, 4),
           "step_kv_tokens_per_s": round(sum(ctx) / ts, 1),
           "step": "pd_decode_step_fp8 (quantising store of 64 tokens, then the decode)"}
    del kc8, vc8
    torch.cuda.empty_cache()
    return res


def bench_spec_verify(pd, pd_inputs, dev, args, flush, hbm_peak, bf16_peak):
    """Speculative verification of 4 tokens per sequence (64 sequences, prior
    context U[128, 2048], Qwen3-8B shape) through the chunked-prefill kernel:
    K/V bytes read per second (the bound) and causal TFLOP/s."""
    import torch
    m = pd_inputs.spec_verify()
    kc, vc = m.pool.key_cache.to(dev), m.pool.value_cache.to(dev)
    pd.pd_reshape_and_cache(m.new_key.to(dev), m.new_value.to(dev), kc, vc,
                            m.slot_mapping.to(dev))
    q = m.q_prefill.to(dev)
    out = torch.empty_like(q)
    cu = m.cu_q_lens.to(dev)
    bt = m.pool.block_tables[:m.Bp].to(dev)
    cl = m.pool.context_lens[:m.Bp].to(dev)
    tp = _time_calls(lambda: pd.pd_paged_prefill_chunk(out, q, cu, m.max_q_len, kc, vc, bt, cl,
                                                       m.scale), args.extra_steps, flush)
    nq = m.max_q_len
    mcl = int(m.pool.context_lens[:m.Bp].max())
    q4, o4 = q.view(m.Bp, nq, m.H, m.D), out.view(m.Bp, nq, m.H, m.D)
    ws = pd.verify_workspace(m.Bp, nq, m.H, m.D, mcl, device=dev)
    t = _time_calls(lambda: pd.pd_paged_attention_verify(o4, q4, kc, vc, bt, cl, mcl, m.scale, ws),
                    args.extra_steps, flush)
    nk, nv, sl = m.new_key.to(dev), m.new_value.to(dev), m.slot_mapping.to(dev)
    tstep = _time_calls(lambda: pd.pd_verify_step(o4, q4, kc, vc, bt, cl, mcl, m.scale, nk, nv, sl,
                                                  workspace=ws), args.extra_steps, flush)
    ctx = m.pool.context_lens[:m.Bp].double()
    kv = float(ctx.sum()) * m.Hk * m.D * 2 * 2
    P = m.prior_lens.double()
    flops = float(4 * m.D * m.H * (nq * P + nq * (nq + 1) / 2).sum())
    res = {"workload": f"{m.Bp} sequences x {nq} query tokens, prior U[128, 2048], bf16",
           "path": "pd_paged_attention_verify (decode kernel, (head, query) columns)",
           "ms": round(t * 1e3, 4), "kv_gbs": round(kv / t / 1e9, 1),
           "kv_frac": round(kv / t / 1e9 / hbm_peak, 4), "tflops": round(flops / t / 1e12, 2),
           "query_tokens_per_s": round(m.Bp * nq / t, 1),
           "step_ms": round(tstep * 1e3, 4),
           "step": "pd_verify_step: store the drafted tokens, then verify as a dependent grid",
           "via_prefill_chunk": {"ms": round(tp * 1e3, 4), "kv_gbs": round(kv / tp / 1e9, 1),
                                 "kv_frac": round(kv / tp / 1e9 / hbm_peak, 4)}}
    del kc, vc
    torch.cuda.empty_cache()
    return res


def bench_prefix_cache(pd, args):
    """Host prefix cache (pd_pc_*): 64 requests of 2048 tokens (S 16, 128 full
    blocks each) that share a 1024-token prefix; every request looks its
    prompt up (hash chain over its blocks) and inserts what missed.  Reports
    blocks hashed per second and the hit rate."""
    import numpy as np
    S, n_req, n_tok, shared = 16, 64, 2048, 1024
    rng = np.random.default_rng(0)
    prefix = rng.integers(0, 150000, shared)
    prompts = [np.concatenate([prefix, rng.integers(0, 150000, n_tok - shared)]).tolist()
               for _ in range(n_req)]
    pc = pd.PrefixCache(capacity_blocks=n_req * n_tok // S, block_size=S)
    next_block, hit_tokens = 0, 0
    t0 = time.perf_counter()
    for toks in prompts:
        hit, keys, _ = pc.lookup(toks)
        hit_tokens += hit
        fresh = list(range(next_block, next_block + len(keys)))
        next_block += len(keys)
        pc.insert(keys, fresh)
    dt = time.perf_counter() - t0
    blocks = n_req * (n_tok // S)
    return {"workload": f"{n_req} requests x {n_tok} tokens, {shared}-token shared prefix, S {S}",
            "blocks_per_s": round(blocks / dt, 1), "us_per_request": round(dt / n_req * 1e6, 1),
            "hit_rate": round(pc.hit_rate, 4),
            "token_hit_fraction": round(hit_tokens / (n_req * n_tok), 4),
            "note": "host C++ (SHA-256 chain, LRU) through the binding; no GPU work"}


def bench_kv_handover(pd, pd_inputs, dev, args, flush, hbm_peak):
    """KV hand-over of 4 sequences x 2048 tokens, 32 layers, Qwen3-8B kv shape:
    pack on the sending side, unpack into the receiving pool (1 GiB of KV each
    way; bytes = read + written)."""
    import torch
    c = pd_inputs.kv_transfer(seed=0, device=dev)
    send = c.block_ids(c.send_tables).to(dev)
    recv = c.block_ids(c.recv_tables).to(dev)
    st = pd.kv_staging(c.L, send.numel(), c.key_caches[0])
    rk = [torch.empty(c.NB_recv, c.Hk, c.S, c.D, dtype=c.dtype, device=dev) for _ in range(c.L)]
    rv = [torch.empty_like(t) for t in rk]
    n = args.extra_steps
    t_pack = _time_calls(lambda: pd.pd_kv_pack(st, c.key_caches, c.value_caches, send), n, flush)
    t_unpack = _time_calls(lambda: pd.pd_kv_unpack(st, rk, rv, recv), n, flush)
    kv = st.numel() * st.element_size()
    res = {"workload": "32 layers, 4 x 2048 tokens, 8 kv heads x 128, S 16, bf16",
           "kv_bytes": kv,
           "pack_ms": round(t_pack * 1e3, 4), "pack_gbs": round(2 * kv / t_pack / 1e9, 1),
           "pack_frac": round(2 * kv / t_pack / 1e9 / hbm_peak, 4),
           "unpack_ms": round(t_unpack * 1e3, 4), "unpack_gbs": round(2 * kv / t_unpack / 1e9, 1),
           "unpack_frac": round(2 * kv / t_unpack / 1e9 / hbm_peak, 4)}
    del c, st, rk, rv
    torch.cuda.empty_cache()
    return res


def bench_cow(pd, pd_inputs, dev, args, flush, hbm_peak):
    import torch
    res = {}
    for S in (8, 16, 32, 64):
        fc = pd_inputs.cow_fork_stress(S)
        bm = pd.BlockManager(fc.NB, S)
        tables, ctxs, slots, pairs = [], [], [], []
        nid = 0
        for L in fc.prompt_lens.tolist():
            parent = nid
            nid += 1
            bm.add_seq(parent)
            for _ in range(L):
                bm.append_slot(parent)
            kids = list(range(nid, nid + fc.n_fork))
            nid += fc.n_fork
            for k in kids:
                bm.fork(parent, k)
            bm.release(parent)
            for k in kids:
                s, cp = bm.append_slot(k)
                slots.append(s)
                if cp:
                    pairs.append(cp)
                tables.append(bm.block_table(k))
                ctxs.append(L + 1)
        kc, vc = fc.key_cache.to(dev), fc.value_cache.to(dev)
        mb = max(len(t) for t in tables)
        bt = torch.zeros(len(tables), mb, dtype=torch.int32)
        for i, t in enumerate(tables):
            bt[i, :len(t)] = torch.tensor(t, dtype=torch.int32)
        bt, cl = bt.to(dev), torch.tensor(ctxs, dtype=torch.int32, device=dev)
        pr = torch.tensor(pairs, dtype=torch.int64, device=dev).view(-1, 2)
        sl = torch.tensor(slots, dtype=torch.int64, device=dev)
        nk, nv, q = fc.new_key.to(dev), fc.new_value.to(dev), fc.q.to(dev)
        out = torch.empty_like(q)
        mcl = max(ctxs)
        ws = pd.decode_workspace(len(tables), fc.H, fc.D, mcl, device=dev)
        n = args.extra_steps
        t_copy = _time_calls(lambda: pd.pd_copy_blocks([kc], [vc], pr), n, flush)
        t_dec = _time_calls(lambda: pd.pd_paged_attention_decode(out, q, kc, vc, bt, cl, mcl,
                                                                 fc.scale, ws), n, flush)

        def whole():
            pd.pd_copy_blocks([kc], [vc], pr)
            pd.pd_reshape_and_cache(nk, nv, kc, vc, sl)
            pd.pd_paged_attention_decode(out, q, kc, vc, bt, cl, mcl, fc.scale, ws)

        t_step = _time_calls(whole, n, flush)
        # the same decode with each prompt's shared blocks read once for its
        # forks: groups from the host helper (outside the timing)
        grp_starts, grp_shared = pd.find_shared_prefixes(bt.cpu(), cl.cpu(), S,
                                                         max_group=fc.n_fork)
        gs_d, sl_d = grp_starts.to(dev), grp_shared.to(dev)
        ws_sh = pd.decode_shared_workspace(grp_shared.numel(), fc.n_fork, fc.H, fc.Hk, fc.D,
                                           device=dev)

        def shared_decode():
            pd.pd_paged_attention_decode_shared(out, q, kc, vc, bt, cl, mcl, fc.scale, gs_d, sl_d,
                                                fc.n_fork, ws_sh)

        t_sh = _time_calls(shared_decode, n, flush)

        def whole_shared():
            # copies -> store -> shared-prefix decode as one chain of dependent grids
            pd.pd_decode_step_shared(out, q, kc, vc, bt, cl, mcl, fc.scale, gs_d, sl_d, fc.n_fork,
                                     key=nk, value=nv, slot_mapping=sl, block_mapping=pr,
                                     workspace=ws_sh)

        t_step_sh = _time_calls(whole_shared, n, flush)
        sha = source_sha("decode.cu", "pd_device.cuh")
        dram_sh = profiled_traffic(f"paged_decode_shared_cow_S{S}", sha)
        _, logical = decode_alg_bytes(ctxs, len(tables), fc.H, fc.Hk, fc.D, S)
        unique_blocks = len({b for t in tables for b in t})
        unique = unique_blocks * S * fc.Hk * fc.D * 2 * 2
        copy_bytes = 2 * len(pairs) * 2 * fc.Hk * S * fc.D * 2
        # DRAM bytes of one decode launch from the committed ncu capture of this
        # source (None once the kernel changed since)
        dram = profiled_traffic(f"paged_decode_cow_S{S}", source_sha("decode.cu", "pd_device.cuh"))
        res[f"S{S}"] = {"pairs": len(pairs), "groups": grp_shared.numel(),
                        "step_ms": round(t_step * 1e3, 4),
                        "copy_ms": round(t_copy * 1e3, 4),
                        "copy_gbs": round(copy_bytes / t_copy / 1e9, 1),
                        "decode_ms": round(t_dec * 1e3, 4),
                        "decode_logical_gbs": round(logical / t_dec / 1e9, 1),
                        "decode_unique_gbs": round(unique / t_dec / 1e9, 1),
                        "decode_unique_frac": round(unique / t_dec / 1e9 / hbm_peak, 4),
                        "decode_dram_bytes": dram,
                        "decode_dram_over_unique": round(dram / unique, 3) if dram else None,
                        "decode_dram_frac": (round(dram / t_dec / 1e9 / hbm_peak, 4)
                                             if dram else None),
                        "shared": {
                            "path": "pd_paged_attention_decode_shared (each prompt's shared "
                                    "blocks read once for its 8 forks)",
                            "decode_ms": round(t_sh * 1e3, 4),
                            "step_ms": round(t_step_sh * 1e3, 4),
                            "step": "pd_decode_step_shared: copy_blocks -> store -> shared-prefix "
                                    "decode, each grid a programmatic dependent of the last",
                            "decode_unique_gbs": round(unique / t_sh / 1e9, 1),
                            "decode_unique_frac": round(unique / t_sh / 1e9 / hbm_peak, 4),
                            "decode_logical_gbs": round(logical / t_sh / 1e9, 1),
                            "decode_dram_bytes": dram_sh,
                            "decode_dram_over_unique": (round(dram_sh / unique, 3)
                                                        if dram_sh else None),
                            "decode_dram_frac": (round(dram_sh / t_sh / 1e9 / hbm_peak, 4)
                                                 if dram_sh else None)}}
    return res


def run_reference(args, rank, world):
    """The oracle (as it stands) on the host cores, on the headline workload; a
    step = store + decode of a bounded sample of the batch's sequences."""
    import numpy as np
    import torch
    import oracle
    import pd_inputs
    if rank != 0:
        return None
    c = pd_inputs.qwen3_8b_decode()
    threads = oracle.default_threads()
    n_seq = 16                                     # sample: the first 16 of 64 sequences
    ctx = c.pool.context_lens[:n_seq].tolist()
    _, dbytes = decode_alg_bytes(ctx, n_seq, c.H, c.Hk, c.D, c.pool.S)
    sbytes = store_alg_bytes(n_seq, c.Hk, c.D)
    kc0 = c.pool.key_cache.view(torch.int16).numpy().view(np.uint16)
    vc0 = c.pool.value_cache.view(torch.int16).numpy().view(np.uint16)

    def step():
        kc, vc = kc0.copy(), vc0.copy()
        t0 = time.perf_counter()
        oracle.reshape_and_cache(c.new_key[:n_seq], c.new_value[:n_seq], kc, vc,
                                 c.slot_mapping[:n_seq], c.pool.S)
        oracle.decode(c.q, kc, vc, c.pool.block_tables, c.pool.context_lens, c.scale,
                      oracle.BF16, threads=threads, rows=(0, n_seq * c.H))
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        step()
    total = sum(step() for _ in range(args.steps))
    value = (dbytes + sbytes) * args.steps / total / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "qwen3_8b_decode_step", "batch": 64, "q_heads": 32,
                       "kv_heads": 8, "head_dim": 128, "block_size": 16,
                       "context_lens": "uniform [128, 2048], seed 0",
                       "step": f"store + decode of the first {n_seq} of 64 sequences"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                             "kind": "oracle",
                             "sample": f"first {n_seq} of 64 sequences per step"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    return line


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.only_extras:
        print(json.dumps(run_only_extras(args)), flush=True)
        return
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local_rank))
    try:
        result = run_ours(args, rank, world, local_rank)
        if rank == 0:
            print(json.dumps(result), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
