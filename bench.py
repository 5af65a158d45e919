#!/usr/bin/env python
"""Benchmark of the RocketKV hot path on GB300: decode steps/s of one full pass per step.

One step = one pass of the whole hot path over one batch of synthetic input:
  SnapKV++ compression of every (layer, KV head) of the prompt  (score passes, select, gather;
    the gather also builds the page summaries of the compact cache)
  + `decode_steps` hybrid sparse decode steps (each one launch over all layers and KV heads).
Default workload: Llama-3.1-8B attention shapes (32 layers, 32 query / 8 KV heads, d 128, bf16),
batch 1, 32K prompt, window 32, pooling 15, budget 256 (page 4, 32 of 128 channels, keep 4096),
128 decode steps. value = decode steps per second over the whole pass (prompt compression
included); the per-phase breakdown and the decode-only rate are reported beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica on its own GPU (the path has no
exchange step); rank 0 prints the JSON line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import atexit
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode attention steps/s and HBM GB/s (% of peak) at 32K–128K ctx, budget 256"
UNIT = "decode steps/s"
FALLBACK_HBM = 6800.0
FALLBACK_BF16 = 1900.0
L2_BYTES = 129 * 1000 * 1000


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama8b_32k")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline leg")
    ap.add_argument("--no-dense", action="store_true", help="skip the dense-decode comparison")
    ap.add_argument("--seed", type=int, default=2000)
    ap.add_argument("--layers", type=int, default=0,
                    help="run the workload with this many layers (smaller profiling cases)")
    ap.add_argument("--decode-sets", type=int, default=0,
                    help="copies of the compact cache the decode steps rotate through (0: as "
                         "many as keep each step's rows out of L2, see decode_sets; 1: none)")
    ap.add_argument("--ctx", type=int, default=0,
                    help="prompt length of every sequence (e.g. 131072: the 128K end of the "
                         "metric at the default workload's budget)")
    return ap.parse_args()


def select_workload(args):
    from dataclasses import replace
    from sparse_kv_cache_snapkv_gb300 import synthetic as S
    wl = S.WORKLOADS[args.workload]
    if args.layers:
        wl = wl.with_layers(args.layers)
    if args.ctx:
        wl = replace(wl, name=f"{wl.name}@ctx{args.ctx}", lens=(args.ctx,) * wl.n_seq)
    return wl


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(
            p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM, FALLBACK_BF16, 1700.0, "fallback"


# --------------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    MAX_S = 900  # the sampler ends by itself after this long, whatever happens to this process

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["timeout", str(self.MAX_S), "nvidia-smi", f"--id={self.gpu}",
                 f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            # a bench that fails inside the timed region must not leave the sampler running
            atexit.register(self._kill)
        except Exception:
            self.proc = None

    def _kill(self):
        if self.proc is not None and self.proc.poll() is None:
            self.proc.kill()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------------- oracle CPU
def _oracle_worker_init():
    os.environ["OMP_NUM_THREADS"] = "1"
    os.environ["OPENBLAS_NUM_THREADS"] = "1"


_UNIT_CACHE = {}


def _unit_data(wl, unit, seed):
    """One (layer, KV head) unit of the workload, drawn on the CPU in the worker (float64)."""
    key = (wl.name, unit, seed)
    if key not in _UNIT_CACHE:
        from dataclasses import replace
        from sparse_kv_cache_snapkv_gb300 import synthetic as S
        one = replace(wl, n_seq=1, n_layers=1, n_kv=1, lens=(wl.lens[0],))
        x = S.prefill_inputs(one, seed=seed + 7919 * unit, device="cpu")
        if len(_UNIT_CACHE) >= 2:
            _UNIT_CACHE.clear()
        _UNIT_CACHE[key] = (x["k"][0, 0].double().numpy(), x["v"][0, 0].double().numpy(),
                            x["q_win"][0].double().numpy(), int(x["seq_lens"][0]))
    return _UNIT_CACHE[key]


def _oracle_unit(args):
    """Oracle work for one (layer, KV head) unit: compress + summaries + `steps` decode steps.
    Returns (compress seconds, seconds per decode step); input drawing is not timed."""
    import numpy as np
    from oracle import rocketkv as O
    wl, unit, seed, keep, kernel, budget, page, channels, steps = args
    k, v, q_win, L = _unit_data(wl, unit, seed)
    scale = 1.0 / math.sqrt(128)
    t0 = time.perf_counter()
    kept, kc, vc, _, _ = O.snapkv_compress(k[:L], v[:L], q_win, keep, kernel, scale)
    n1 = kc.shape[0]
    kmin, kmax = O.page_summaries(kc, n1, page)
    t1 = time.perf_counter()
    rng = np.random.default_rng(seed + unit)
    for _ in range(steps):
        q = rng.standard_normal((q_win.shape[0], 128))
        O.hybrid_decode(q, kc, vc, n1, kmin, kmax, budget, page, channels, scale)
    t2 = time.perf_counter()
    return t1 - t0, (t2 - t1) / max(1, steps)


def oracle_sample(wl, keep, kernel, units, cores, seed, pool, first_unit=0):
    """One sample of the oracle on the workload: `cores` (layer, KV head) units in parallel, one
    per core, each compression + summaries + all of the workload's decode steps. Returns the
    sample's measured seconds (the slowest unit's oracle time; drawing the inputs is not timed)
    and the per-unit mean compress seconds and seconds per decode step. Both the cpu_baseline
    leg and the reference arm time the oracle through this one rule."""
    kernel = kernel or (7 if wl.max_len <= 8192 else 15 if wl.max_len <= 32768 else 31)
    n_units = min(units, cores)
    args = [(wl, (first_unit + i) % units, seed, keep, kernel, wl.budget, wl.page,
             wl.channels, wl.decode_steps) for i in range(n_units)]
    res = pool.map(_oracle_unit, args, chunksize=1)
    measured = max(r[0] + wl.decode_steps * r[1] for r in res)
    return measured, statistics.mean(r[0] for r in res), statistics.mean(r[1] for r in res)


def oracle_full_step_s(wl, units, cores, tc, td):
    """Seconds for the whole step on `cores` cores, from per-unit times: every core takes
    ceil(units / cores) units, each compression + summaries + decode_steps decode steps."""
    return math.ceil(units / cores) * (tc + wl.decode_steps * td)


def oracle_sample_text(wl, units, cores, n_samples):
    return (f"{n_samples} sample(s) of {min(units, cores)} (layer, KV head) units, one per core, "
            f"each: compression + summaries + {wl.decode_steps} decode steps; rate extrapolated "
            f"to {units} units x {wl.decode_steps} decode steps from the per-unit mean times")


# --------------------------------------------------------------------------------- helpers
def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_config(wl, keep):
    kernel = wl.kernel or (7 if wl.max_len <= 8192 else 15 if wl.max_len <= 32768 else 31)
    return {"workload": wl.name, "layers": wl.n_layers, "batch": wl.n_seq, "q_heads": wl.n_q,
            "kv_heads": wl.n_kv, "head_dim": 128, "ctx": wl.max_len, "window": wl.window,
            "pool_kernel": kernel, "budget": wl.budget, "page": wl.page,
            "channels": wl.channels, "keep": keep, "decode_steps_per_step": wl.decode_steps,
            "append": wl.append, "needles": wl.needles,
            "l2": "inputs larger than L2: prompt K/V %.2f GB per step, compact cache + summaries "
                  "%.2f GB; without appends the decode steps rotate through copies of the "
                  "compact cache so that each step reads from HBM (see decode_sets)"
                  % (2 * wl.n * wl.n_kv * wl.max_len * 256 / 1e9,
                     (wl.n * wl.n_kv * (keep or 0) * 512 * 1.25) / 1e9),
            "parallelism": "replicas"}


# --------------------------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    from sparse_kv_cache_snapkv_gb300 import rkv, synthetic as S
    from sparse_kv_cache_snapkv_gb300.pipeline import HotPath

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    rkv.load()
    dev = torch.device("cuda", local)
    wl = select_workload(args)
    hbm_peak, bf16_peak, bf16_sus, peak_src = peaks()

    # cpu-baseline pool first (spawn, before heavy GPU work)
    pool = None
    cores = min(16, len(os.sched_getaffinity(0)))
    if rank == 0 and not args.no_cpu:
        _oracle_worker_init_env()
        pool = mp.get_context("spawn").Pool(cores, initializer=_oracle_worker_init)

    x = S.prefill_inputs(wl, seed=args.seed + rank, device=dev)
    dq = S.decode_queries(wl, wl.decode_steps, seed=args.seed + 500 + rank, device=dev)
    nk = nv = None
    if wl.append:
        nk, nv = S.append_tokens(wl, wl.decode_steps, x["sigma"], seed=args.seed + 900, device=dev)
    hp = HotPath(wl, x["k"], x["v"], x["q_win"], x["seq_lens"], dq, nk, nv)
    # the e2e leg's pinned host copies of the inputs, made before the other legs run
    host_in = None if args.no_e2e else _pinned_inputs(x, dq, nk, nv)

    # eager pass: sets kernel attributes, checks device status
    hp.step()
    torch.cuda.synchronize()
    hp.check_status()
    # Cold-L2 decode: every layer is batched into one launch, so consecutive steps would find
    # the rows they re-read in L2; rotating copies of the compact cache (enough that one step's
    # rows are evicted before they come round again) makes each step read from HBM, as it would
    # in a model, where the other layers' work runs between two steps of a layer.
    sets = args.decode_sets or decode_sets(wl, hp)
    if sets > 1 and not wl.append:
        hp.rotate_decode_sets(sets)

    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graphs = []
    # the summaries phase is empty when the compression builds them and nothing is appended
    sum_empty = hp.fuse_summaries and not wl.append
    with torch.cuda.stream(stream):
        for fn in (hp.compress, None if sum_empty else hp.summaries,
                   lambda: [hp.decode(t) for t in range(wl.decode_steps)]):
            if fn is None:
                graphs.append(None)
                continue
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            graphs.append(g)
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            for g in graphs:
                if g is not None:
                    g.replay()
        torch.cuda.synchronize()
        hp.check_status()
        barrier(world)
        sampler = ClockSampler(local)
        sampler.start()
        time.sleep(0.3)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
        torch.cuda.synchronize()
        barrier(world)
        for i in range(args.steps):
            ev[i][0].record(stream)
            graphs[0].replay()
            ev[i][1].record(stream)
            if graphs[1] is not None:
                graphs[1].replay()
            ev[i][2].record(stream)
            graphs[2].replay()
            ev[i][3].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        clocks = sampler.stop()
    total_ms = ev[0][0].elapsed_time(ev[-1][3])
    total_ms = max_over_ranks(total_ms, world)
    comp_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    sum_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    dec_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in ev)
    hp.check_status()

    steps_total = args.steps * wl.decode_steps * world
    value = steps_total / (total_ms / 1e3)
    ms_per_step = total_ms / args.steps
    dec_launch_us = dec_ms * 1e3 / wl.decode_steps
    dec_bytes = hp.decode_bytes_per_launch()
    dec_gbs = dec_bytes / (dec_launch_us * 1e-6) / 1e9
    comp_bytes = hp.compress_bytes()
    comp_gbs = comp_bytes / (comp_ms * 1e-3) / 1e9
    comp_tflops = hp.compress_flops() / (comp_ms * 1e-3) / 1e12

    # dominant phase -> roofline object
    if dec_ms >= comp_ms:
        roof = {"kernel": "hybrid_decode_kernel", "bound": "hbm", "achieved": round(dec_gbs, 1),
                "peak": hbm_peak, "unit": "GB/s", "frac": round(dec_gbs / hbm_peak, 4),
                "traffic": None, "peak_source": peak_src,
                "bytes_per_launch": dec_bytes, "launch_us": round(dec_launch_us, 3)}
    else:
        roof = {"kernel": "snapkv compression (score passes + select + gather)", "bound": "hbm",
                "achieved": round(comp_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(comp_gbs / hbm_peak, 4), "traffic": None,
                "peak_source": peak_src, "bytes_per_launch": comp_bytes,
                "launch_us": round(comp_ms * 1e3, 1)}
    # the committed capture is of the default workload at 32 layers: other shapes get null
    traffic = None
    if args.workload == "llama8b_32k" and wl.n_layers == 32 and not args.ctx:
        traffic = _profiled_traffic(roof["kernel"])
    if traffic is not None:
        roof["traffic"] = traffic

    breakdown = {
        "compress_ms": round(comp_ms, 4), "summaries_ms": round(sum_ms, 4),
        "decode_ms": round(dec_ms, 4),
        "decode_only_steps_per_s": round(wl.decode_steps / (dec_ms / 1e3) * world, 1),
        "decode_launch_us": round(dec_launch_us, 3),
        "decode_hbm_gbs": round(dec_gbs, 1), "decode_frac_of_peak": round(dec_gbs / hbm_peak, 4),
        "compress_gbs": round(comp_gbs, 1), "compress_tflops": round(comp_tflops, 2),
        "compress_frac_of_peak_hbm": round(comp_gbs / hbm_peak, 4),
        "decode_cache_sets": len(getattr(hp, "sets", [None])),
    }

    # dense decode over the full prompt (the full-KV baseline), one launch over all units
    if not args.no_dense:
        breakdown["dense_decode"] = _dense_compare(hp, x, dq, wl, hbm_peak, stream, world)

    # end-to-end: host buffers -> device -> the API calls -> result back to the host
    e2e = None
    if not args.no_e2e:
        e2e = _e2e(hp, host_in, wl, stream, world, min(args.steps, 10))

    # oracle on the host cores (rank 0 only)
    cpu = None
    if pool is not None:
        units = wl.n * wl.n_kv
        oracle_sample(wl, hp.keep, wl.kernel, units, cores, args.seed, pool)  # untimed warm-up
        n_samples = 6
        res = [oracle_sample(wl, hp.keep, wl.kernel, units, cores, args.seed, pool,
                             first_unit=i * cores) for i in range(n_samples)]
        pool.close()
        tc = statistics.mean(r[1] for r in res)
        td = statistics.mean(r[2] for r in res)
        full_s = oracle_full_step_s(wl, units, cores, tc, td)
        cpu = {"value": round(wl.decode_steps / full_s, 4), "unit": UNIT, "cores": cores,
               "kind": "oracle",
               "sample": oracle_sample_text(wl, units, cores, n_samples) +
                         f"; per-unit mean {tc:.3f} s compress, {td * 1e3:.2f} ms per decode step",
               "sample_s": round(sum(r[0] for r in res), 2),
               # the same per-unit times with every unit on one core, one after another
               "value_1core": round(wl.decode_steps / oracle_full_step_s(wl, units, 1, tc, td),
                                    4)}

    launches = hp.launches_per_step() * args.steps
    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic (seeded; Llama-3.1-8B attention shapes, "
                "random K/V with lognormal channel scales and planted needles)",
                "config": workload_config(wl, hp.keep), "roofline": roof, "cpu_baseline": cpu,
                "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
                "breakdown": breakdown, "impl": "ours"}
        print(json.dumps(line), flush=True)


def decode_sets(wl, hp, l2_bytes=L2_BYTES):
    """Copies of the compact cache the decode steps rotate through: enough that 4 x L2 of other
    decode traffic passes between two reads of a copy, at most 8; 1 with appends."""
    if wl.append:
        return 1
    per_step = hp.decode_bytes_per_launch()
    return int(max(1, min(8, math.ceil(4 * l2_bytes / max(per_step, 1)))))


def _oracle_worker_init_env():
    os.environ.setdefault("OMP_NUM_THREADS", "1")


def _profiled_traffic(kernel_name):
    """DRAM bytes per launch from the committed ncu summary (profiles/traffic.md), only while the
    kernel's source file is unchanged since the capture (its hash matches); else None."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.md")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    for line in lines:
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) == 5 and cells[0] == kernel_name:
            # the hash covers every file named ("a.cu+common.cuh"), read in that order
            h = hashlib.sha256()
            try:
                for name in cells[3].split("+"):
                    src = os.path.join(ROOT, "sparse_kv_cache_snapkv_gb300", "csrc", name.strip())
                    h.update(open(src, "rb").read())
            except OSError:
                return None
            return int(cells[1]) if h.hexdigest()[:16] == cells[4] else None
    return None


def _dense_compare(hp, x, dq, wl, hbm_peak, stream, world):
    import torch
    from sparse_kv_cache_snapkv_gb300 import rkv
    n, n_kv = wl.n, wl.n_kv
    out = torch.empty(n, wl.n_q, 128, dtype=torch.bfloat16, device=x["k"].device)
    ws = rkv.workspace(rkv.rkv_dense_decode_workspace_bytes(n, n_kv, wl.gqa, wl.max_len),
                       x["k"].device)
    reps = 10
    with torch.cuda.stream(stream):
        for t in range(3):
            rkv.rkv_dense_decode(dq[t], x["k"], x["v"], x["seq_lens"], hp.scale, out, ws=ws)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for t in range(reps):
            rkv.rkv_dense_decode(dq[t % dq.shape[0]], x["k"], x["v"], x["seq_lens"], hp.scale,
                                 out, ws=ws)
        b.record(stream)
        torch.cuda.synchronize()
    rkv.rkv_check_status(ws)
    ms = a.elapsed_time(b) / reps
    byts = int(x["seq_lens"].sum().item()) * n_kv * 128 * 2 * 2 + n * wl.n_q * 128 * 4
    gbs = byts / (ms * 1e-3) / 1e9
    return {"steps_per_s": round(1e3 / ms * world, 2), "ms": round(ms, 4),
            "hbm_gbs": round(gbs, 1), "frac_of_peak": round(gbs / hbm_peak, 4),
            "bytes_per_launch": byts}


E2E_WARMUP = 3  # untimed end-to-end passes before the timed ones


def _pinned_inputs(x, dq, nk, nv):
    """Pinned host copies of a pass's inputs (the e2e leg copies them in every pass)."""
    dev_in = [x["k"], x["v"], x["q_win"], x["seq_lens"], dq]
    if nk is not None:
        dev_in += [nk, nv]
    return [t.cpu().pin_memory() for t in dev_in]


def _e2e(hp, host_in, wl, stream, world, steps):
    import torch
    dev_in = [hp.k, hp.v, hp.q_win, hp.seq_lens, hp.dec_q]
    if hp.new_k is not None:
        dev_in += [hp.new_k, hp.new_v]
    host_out = torch.empty(hp.out.shape, dtype=hp.out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out.numel() * host_out.element_size()
    def one_pass():
        for d, h in zip(dev_in, host_in):
            d.copy_(h, non_blocking=True)
        hp.step()
        host_out.copy_(hp.out, non_blocking=True)

    # every pass decodes from the cache its own compression wrote (no rotated copies here: the
    # host copies dominate this leg anyway)
    sets, hp.sets = getattr(hp, "sets", None), None

    with torch.cuda.stream(stream):
        # untimed warm-up passes: the first transfers from freshly pinned memory run slower
        for _ in range(E2E_WARMUP):
            one_pass()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            one_pass()
        b.record(stream)
        torch.cuda.synchronize()
    hp.check_status()
    hp.sets = sets
    ms = a.elapsed_time(b)
    ms = max_over_ranks(ms, world)
    return {"value": round(steps * wl.decode_steps * world / (ms / 1e3), 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms / steps, 3)}


# --------------------------------------------------------------------------------- prefill sweep
SWEEP_KERNELS = (1, 3, 7, 15, 31)
SWEEP_BUDGETS = (256, 1024, 4096)


def _time_ms(fn, stream, reps, warmup=3):
    """Mean milliseconds of fn() over `reps` back-to-back calls (CUDA events on `stream`), after
    `warmup` untimed calls."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def run_prefill_sweep(args):
    """SnapKV++ prefill sweep on one 128K prompt (32 query / 8 KV heads, window 64, so the score
    GEMM has G*W = 256 rows): the two tensor-core score passes, then the pooling + top-k select
    for every pooling kernel in {1, 3, 7, 15, 31} and budget in {256, 1024, 4096} (keep = 16 x
    budget), and the gather of each budget's kept rows. Phases are timed by difference of
    C-ABI calls that stop after them: rkv_snapkv_scores (score passes), rkv_snapkv_select
    (+ pooling and top-k), rkv_snapkv_compress (+ gather)."""
    import torch
    from sparse_kv_cache_snapkv_gb300 import rkv
    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    rkv.load()
    dev = torch.device("cuda", local)
    wl = select_workload(args)
    hbm_peak, bf16_peak, _, peak_src = peaks()
    from sparse_kv_cache_snapkv_gb300 import synthetic as S
    x = S.prefill_inputs(wl, seed=args.seed + rank, device=dev)
    n, n_kv, L = wl.n, wl.n_kv, wl.max_len
    W, G = wl.window, wl.gqa
    scale = 1.0 / math.sqrt(128)
    ws = rkv.workspace(rkv.rkv_snapkv_workspace_bytes(n, n_kv, G, L, W), dev)
    scores = torch.empty(n, n_kv, L - W, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream()
    reps = max(3, args.steps)
    warm = max(3, args.warmup)
    units = n * n_kv
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    t_scores = _time_ms(lambda: rkv.rkv_snapkv_scores(x["k"], x["seq_lens"], x["q_win"], scale,
                                                      scores, ws=ws, stream=stream),
                        stream, reps, warm)
    flops = 2 * 2 * units * G * W * L * 128
    score_tflops = flops / (t_scores * 1e-3) / 1e12
    cells = []
    for budget in SWEEP_BUDGETS:
        keep = rkv.rkv_plan(L, budget)[0]
        kept = torch.empty(n, n_kv, keep, dtype=torch.int32, device=dev)
        out_len = torch.empty(n, dtype=torch.int32, device=dev)
        k_out = torch.empty(n, n_kv, keep, 128, dtype=torch.bfloat16, device=dev)
        v_out = torch.empty_like(k_out)
        for kernel in SWEEP_KERNELS:
            t_sel = _time_ms(lambda: rkv.rkv_snapkv_select(
                x["k"], x["seq_lens"], x["q_win"], kernel, keep, scale, kept, out_len, ws=ws,
                stream=stream), stream, reps, warm)
            t_all = _time_ms(lambda: rkv.rkv_snapkv_compress(
                x["k"], x["v"], x["seq_lens"], x["q_win"], kernel, keep, scale, k_out, v_out,
                kept, out_len, ws=ws, stream=stream), stream, reps, warm)
            rkv.rkv_check_status(ws)
            select_ms = max(t_sel - t_scores, 1e-6)
            gather_ms = max(t_all - t_sel, 1e-6)
            sel_bytes = units * ((L - W) * 4 + keep * 4)       # scores read, kept list written
            gat_bytes = units * keep * 128 * 2 * 4              # K, V rows read and written
            cells.append({
                "kernel": kernel, "budget": budget, "keep": keep,
                "compress_ms": round(t_all, 4), "select_ms": round(select_ms, 4),
                "select_gbs": round(sel_bytes / (select_ms * 1e-3) / 1e9, 1),
                "gather_ms": round(gather_ms, 4),
                "gather_gbs": round(gat_bytes / (gather_ms * 1e-3) / 1e9, 1),
                "gather_frac_of_peak_hbm": round(gat_bytes / (gather_ms * 1e-3) / 1e9 / hbm_peak, 4)})
        del k_out, v_out
    clocks = sampler.stop()
    if rank == 0:
        line = {"metric": "SnapKV++ prefill sweep: score-GEMM TFLOP/s (tensor pipe) and "
                          "select / gather GB/s, 128K prompt, window 64",
                "value": round(score_tflops, 2), "unit": "TFLOP/s", "n_gpus": world,
                "steps": reps, "warmup": warm, "ms_per_step": round(t_scores, 4),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic (seeded; K/V with lognormal channel scales "
                "and planted needles)",
                "config": {"workload": wl.name, "layers": wl.n_layers, "batch": wl.n_seq,
                           "q_heads": wl.n_q, "kv_heads": n_kv, "head_dim": 128, "ctx": L,
                           "window": W, "score_rows": G * W, "kernels": list(SWEEP_KERNELS),
                           "budgets": list(SWEEP_BUDGETS),
                           "l2": "prompt K %.2f GB per score pass (larger than L2)"
                                 % (units * L * 256 / 1e9),
                           "parallelism": "replicas"},
                "roofline": {"kernel": "score_kernel (two passes)", "bound": "tensor",
                             "achieved": round(score_tflops, 1), "peak": bf16_peak,
                             "unit": "TFLOP/s", "frac": round(score_tflops / bf16_peak, 4),
                             "traffic": None, "peak_source": peak_src + " (burst)",
                             "flops_per_launch": flops // 2,
                             "launch_us": round(t_scores * 1e3 / 2, 2),
                             "hbm_gbs_of_k": round(2 * units * L * 256 / (t_scores * 1e-3) / 1e9,
                                                   1)},
                "cpu_baseline": None, "e2e": None, "clocks": clocks,
                "gpu_launches": None, "sweep": cells, "impl": "ours"}
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------------- reference
def run_reference(args):
    """The oracle (plain fp64 CPU implementation) timed on the host cores, same metric/config."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = select_workload(args)
    keep = wl.keep or min(wl.max_len, wl.budget * wl.page * 128 // wl.channels)
    cores = min(16, len(os.sched_getaffinity(0)))
    _oracle_worker_init_env()
    pool = mp.get_context("spawn").Pool(cores, initializer=_oracle_worker_init)
    units = wl.n * wl.n_kv
    res = []
    for i in range(args.warmup + args.steps):
        r = oracle_sample(wl, keep, wl.kernel, units, cores, args.seed, pool,
                          first_unit=i * cores)
        if i >= args.warmup:
            res.append(r)
    pool.close()
    tc = statistics.mean(r[1] for r in res)
    td = statistics.mean(r[2] for r in res)
    full_s = oracle_full_step_s(wl, units, cores, tc, td)
    value = wl.decode_steps / full_s
    sample_ms = statistics.mean(r[0] for r in res) * 1e3
    line = {"metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            # the measured oracle time of one sample; the whole step's time on these cores,
            # extrapolated from the sample's per-unit times, is reported beside it
            "ms_per_step": round(sample_ms, 2),
            "extrapolated_full_step_ms": round(full_s * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "config": workload_config(wl, keep),
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores,
                             "kind": "oracle",
                             "sample": oracle_sample_text(wl, units, cores, args.steps)},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "prefill128k":
        run_prefill_sweep(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
