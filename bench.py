#!/usr/bin/env python3
"""Muon-step benchmark: ms per step and achieved TFLOP/s on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c1|c2|c3|c4|c5]
                    [--impl ours|reference]

One step = momentum -> Newton-Schulz (5 steps) -> decoupled-decay update over
the whole workload, through the C ABI (libmuon).  With no --config the run
times all five workloads and prints ONE JSON line: its headline is the large
compute-bound sweep (c5: 8 x [8192,28672], 10 x [8192,8192], 4 x
[16384,16384], the largest single-GPU workload), timed over exactly K steps
after W warm-up steps; the other four sit under ``per_config`` with the same
fields (the Llama-3-8B-shaped c4 over min(K, 10) steps after 3 warm-ups, the
others over K after W).  ``--config`` times one workload alone.

Per workload:
* ``value`` -- nominal TFLOP/s: sum over matrices of 5 (4 m^2 n + 2 m^3)
  (m <= n) over the device time of a step, inputs resident in HBM;
* ``alg`` -- the same time against the algorithmic flops of the products the
  library runs (symmetric products formed once): 5 (m (m+1) n + m^2 (m+1) +
  2 m^2 n) per matrix in X space, m (m+1) n + 18 m^2 (m+1) + 2 m^2 n in Gram
  space (n >= 2 m), and that rate as a fraction of the measured dense bf16
  peak (sustained when the timed region lasts more than a second, else
  burst);
* ``roofline`` -- the dominant kernel's achieved rate (algorithmic bytes or
  flops per launch over its CUDA-event time) against the measured peak;
* ``e2e`` -- the same metric through the host-memory entry point
  (muon_step_grouped_host): W, G and Mom start in pinned host memory and W',
  Mom' end there, the library's chunked copy-in / step / copy-out pipeline
  inside the timed region;
* ``cpu_baseline`` -- the float64 oracle on the host cores on a bounded
  sample of the workload's own matrices, extrapolated to the whole workload
  (per core shape, by nominal flops) where the sample is not all of it.
Between timed steps a 512 MiB buffer is written to flush the 129 MB L2
(outside the timed events).

``--impl reference`` times the float64 CPU oracle (the deliberately slow
reference) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Muon step ms & achieved TFLOP/s vs GB300 bf16 peak (per config, 1 GPU)"
HP = dict(mu=0.95, nesterov=True, lr=0.02, wd=0.01, scale_rule=0)
STEPS_NS = 5
HEADLINE = "c5"
OTHERS = ("c1", "c2", "c3", "c4")


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from
# one ncu capture of the dominant kernel, keyed by (kernel kind, workload),
# valid only while the kernel's sources hash to the recorded value; otherwise
# the roofline reports traffic = null.
TRAFFIC = {
    ("fused_small", "c2"): {"bytes": 202.21312e6 + 126.546944e6, "src_hash": "72126eaf79b769f6",
                            "sources": ("ns_small.cu", "sm100_ptx.cuh", "muon_internal.h")},
    # large sweep: mean over the 112 apply launches of 4 steps (every chunk and
    # phase: X-space applies and the Gram-space ones), one-pass capture
    ("apply", "c5"): {"bytes": (1041320741376.0 + 98436361728.0) / 112, "src_hash": "573f9bb97c4b8a62",
                      "sources": ("ns_gemm.cu", "sm100_ptx.cuh", "muon_internal.h")},
}

def _traffic(kind, config):
    import hashlib
    rec = TRAFFIC.get((kind, config))
    if rec is None:
        return None
    h = hashlib.sha256()
    for f in rec["sources"]:
        with open(os.path.join(ROOT, "newton_schulz_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return rec["bytes"] if h.hexdigest()[:16] == rec["src_hash"] else None


def _shapes(groups):
    """(B, rows, cols, W bytes, G bytes, path) per group; path is the
    library's choice for the shape (0 small-m, 1 X space, 2 Gram space)."""
    from newton_schulz_gb300 import binding
    out = []
    for g in groups:
        w = g["W"]
        b, r, c = (1, *w.shape) if w.dim() == 2 else tuple(w.shape)
        out.append((b, r, c, w.element_size(), g["G"].element_size(), binding.muon_ns_path(r, c)))
    return out


def matrix_flops(r, c, path, steps=STEPS_NS, restart=None):
    """Algorithmic flops of one matrix's NS per GEMM kind, symmetric products
    formed once.  X space (and the small-m kernel, counted the same way):
    steps x (Gram m(m+1)n, polynomial m^2(m+1), apply 2m^2n).  Gram space,
    in phases of `restart` steps (the library's restart period, 0 = one
    phase): per phase the Gram and the apply once, and 4 (p - 1) + 2
    symmetric m x m products for a phase of p steps (B', Q, T, R per step;
    B' and Q only in the last; Q alone in a one-step phase)."""
    m, n = min(r, c), max(r, c)
    if path == 2:
        if restart is None:
            from newton_schulz_gb300 import binding
            restart = binding.muon_ns_gram_restart(m)
        period = restart
        period = period if period > 0 else steps
        phases = [min(period, steps - k0) for k0 in range(0, steps, period)]
        nsym = sum(1 if p == 1 else 4 * (p - 1) + 2 for p in phases)
        return {"gram": len(phases) * m * (m + 1) * n, "poly": nsym * m * m * (m + 1),
                "apply": len(phases) * 2 * m * m * n}
    return {"gram": steps * m * (m + 1) * n, "poly": steps * m * m * (m + 1),
            "apply": steps * 2 * m * m * n}


def ns_flops(r, c, steps=STEPS_NS):
    """Nominal flops of NS on one [r, c] matrix: steps (4 m^2 n + 2 m^3)."""
    m, n = min(r, c), max(r, c)
    return steps * (4 * m * m * n + 2 * m ** 3)


def nominal_flops(shapes, steps=STEPS_NS):
    return sum(s[0] * ns_flops(s[1], s[2], steps) for s in shapes)


def alg_flops(shapes, steps=STEPS_NS):
    """Algorithmic flops of the computation the library runs (matrix_flops)."""
    return sum(gemm_flops_per_kind(shapes, steps).values())


def algorithmic_bytes(shapes):
    """Per kernel kind: prep reads G, Mom and writes Mom and the bf16 NS
    operand (one layout); update reads W, the bf16 result and writes W; the
    fused small-m kernel moves only the compulsory bytes (G read, Mom and W
    read and written)."""
    prep = upd = fused = 0
    for b, r, c, we, ge, _ in shapes:
        e = b * r * c
        prep += e * (ge + 4 + 4 + 2)
        upd += e * (we + we + 2)
        fused += e * (ge + 4 + 4 + we + we)
    return {"prep": prep, "update": upd, "fused_small": fused}


def gemm_flops_per_kind(shapes, steps=STEPS_NS):
    """Algorithmic (symmetry-aware) flops of one step for each GEMM kind."""
    out = {"gram": 0, "poly": 0, "apply": 0}
    for b, r, c, _, _, path in shapes:
        for k, v in matrix_flops(r, c, path, steps).items():
            out[k] += b * v
    return out


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [l.strip().split(",") for l in self.file.read().splitlines() if l.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                for k, name in enumerate(names):
                    if r[5 + k].strip().lower() == "active":
                        reasons.add(name)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ---- workloads -------------------------------------------------------------------------
def make_workload(name, dev, args):
    from newton_schulz_gb300 import synth
    if name == "c4" and args.layers:
        return synth.config_c4(dev, layers=args.layers)
    if name == "c5" and args.scale_down > 1:
        return synth.config_c5(dev, scale_down=args.scale_down)
    if name == "c3" and args.experts:
        return synth.config_c3(dev, experts=args.experts)
    return synth.CONFIGS[name](dev)


def workload_name(name, args):
    from newton_schulz_gb300 import synth
    s = synth.WORKLOAD_NAMES[name]
    if name == "c4" and args.layers:
        s += f" [{args.layers} layers]"
    if name == "c3" and args.experts:
        s += f" [{args.experts} experts]"
    if name == "c5" and args.scale_down > 1:
        s += f" [dims / {args.scale_down}]"
    return s


# ---- float64 oracle baseline ---------------------------------------------------------
# Which matrices of each workload the oracle times inside the bench (its own
# matrices, copied to the host before the first step): all of the two small
# workloads, 8 experts of each MoE weight, one matrix per core shape of the
# Llama-3-8B shapes, and one [8192, 8192] matrix of the large sweep (one
# 16384^2 matrix alone is ~1.3e14 flops, minutes on the host cores).  The
# other matrices of a workload are extrapolated: the measured time of their
# core shape, or, for core shapes not timed, their nominal flops at the
# sample's rate.
def oracle_sample_index(name, groups):
    if name in ("c1", "c2"):
        return [(gi, b) for gi, g in enumerate(groups) for b in range(g["W"].shape[0])]
    if name == "c3":
        return [(gi, b) for gi in range(len(groups)) for b in range(0, groups[gi]["W"].shape[0], 16)]
    if name == "c4":
        pick, seen = [], set()
        for gi, g in enumerate(groups):
            r, c = g["W"].shape[-2:]
            core = (min(r, c), max(r, c))
            if core not in seen:
                seen.add(core)
                pick.append((gi, 0))
        return pick
    # c5: one matrix of the second group ([8192, 8192] at full size)
    return [(1, 0)]


def oracle_samples(name, groups):
    idx = oracle_sample_index(name, groups)
    out = []
    for gi, b in idx:
        g = groups[gi]
        out.append({k: (g[k][b] if g[k].dim() == 3 else g[k]).detach().double().cpu().numpy()
                    for k in ("W", "G", "Mom")})
    return out


def cpu_baseline(name, samples, shapes):
    """Oracle seconds on the sample, per core shape, extrapolated to the
    workload's ms per step and nominal TFLOP/s."""
    from oracle import muon_ref as R
    cores = len(os.sched_getaffinity(0))
    per_core = {}
    done_flops, t_total = 0, 0.0
    for x in samples:
        r, c = x["W"].shape
        t0 = time.perf_counter()
        R.muon_step_ref(x["W"], x["G"], x["Mom"], **HP)
        dt = time.perf_counter() - t0
        t_total += dt
        done_flops += ns_flops(r, c)
        per_core.setdefault((min(r, c), max(r, c)), []).append(dt)
    rate = done_flops / t_total                  # flop/s of the oracle on the sample
    total_mats = sum(sh[0] for sh in shapes)
    ms, timed_mats = 0.0, 0
    for b, r, c, _, _, _ in shapes:
        core = (min(r, c), max(r, c))
        if core in per_core:
            ms += b * statistics.mean(per_core[core]) * 1e3
            timed_mats += b
        else:
            ms += b * ns_flops(r, c) / rate * 1e3
    flops = nominal_flops(shapes)
    extrapolated = len(samples) < total_mats
    desc = ", ".join(f"{len(v)} x {k[0]}x{k[1]}" for k, v in per_core.items())
    return {"value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle", "extrapolated": extrapolated, "ms_per_step": ms,
            "sample": (f"{len(samples)} of {total_mats} matrices ({desc}), "
                       f"{t_total:.1f} s of float64 NumPy"
                       + ("; the rest extrapolated per core shape (untimed core shapes by "
                          "nominal flops at the sample's rate)" if extrapolated else ""))}


# ---- reference arm -------------------------------------------------------------------------
def _sample_groups_cpu(config):
    """CPU stand-ins with the workload's shapes and value distributions (the
    workload's own values come from the GPU's generator)."""
    import torch
    from newton_schulz_gb300 import synth
    if config in ("c1", "c2"):
        return synth.CONFIGS[config]("cpu")
    if config == "c3":
        return [synth.random_group((1, r, c), torch.bfloat16, torch.float32, "cpu", r, 1e-3)
                for r, c in ((2048, 768), (768, 2048))]
    if config == "c4":
        return [synth.random_group((1, 4096, 4096), torch.bfloat16, torch.bfloat16, "cpu", 4,
                                   1e-3)]
    return [synth.random_group((1, 8192, 8192), torch.bfloat16, torch.float32, "cpu", 5, 1.0)]


def run_reference(args, world, rank):
    """The float64 oracle on the host cores, on a bounded sample per step:
    c1 whole; c2 8 of its 74 matrices; c3 one expert of each weight; c4 one
    [4096, 4096] matrix; c5 one [8192, 8192] matrix with one of its five NS
    iterations (a whole matrix is ~30 s there).  The rate is the sample's
    nominal flops over its time."""
    from oracle import muon_ref as R
    if rank != 0:
        return
    name = args.config or HEADLINE
    cores = len(os.sched_getaffinity(0))
    groups = _sample_groups_cpu(name)
    ns_steps = 1 if name == "c5" else STEPS_NS
    keep = 8 if name == "c2" else None
    sample = []
    for g in groups:
        k = g["W"].shape[0] if keep is None else min(keep, g["W"].shape[0])
        sample.append({k2: g[k2][:k].double().numpy() for k2 in ("W", "G", "Mom")})
    flops = sum(x["W"].shape[0] * ns_flops(x["W"].shape[1], x["W"].shape[2], ns_steps)
                for x in sample)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        for x in sample:
            R.muon_step_ref(x["W"], x["G"], x["Mom"], steps=ns_steps, **HP)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    t = statistics.median(times)
    tf = flops / t / 1e12
    desc = "; ".join(f"{x['W'].shape[0]}x[{x['W'].shape[1]},{x['W'].shape[2]}]" for x in sample)
    if ns_steps != STEPS_NS:
        desc += f" with {ns_steps} of the {STEPS_NS} NS iterations"
    line = {
        "impl": "reference", "metric": METRIC, "value": tf, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(name, args), "config": name, "sample": desc},
        "cpu_baseline": {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": tf, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---- measurement of one workload ------------------------------------------------------
def measure(name, steps, warmup, args, world, dev, local, with_cpu):
    import torch
    from newton_schulz_gb300 import binding
    groups = make_workload(name, dev, args)
    samples = oracle_samples(name, groups) if with_cpu else None
    shapes = _shapes(groups)
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    arr = binding.make_groups(groups)

    def step():
        binding.muon_step_grouped(arr, stream=stream, **HP)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    st = binding.muon_query_status()
    if st != 0:
        raise SystemExit(f"{name}: device status {binding.muon_status_string(st)} after warm-up")
    launches_per_step = binding.muon_last_launch_count()

    # ---- device-resident timed region ------------------------------------------------
    sampler = ClockSampler(local)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    binding.muon_profile_enable(True)
    binding.muon_profile_read()      # reset
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    prof = binding.muon_profile_read()
    binding.muon_profile_enable(False)
    clocks = sampler.stop()
    t_ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    if world > 1:
        t = torch.tensor([t_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        t_ms = float(t.item())

    e2e = None if args.no_e2e else _end_to_end(groups, stream, flush, steps, warmup, world, dev)
    ns_only = None if args.no_ns_only else _ns_only(groups, stream, flush, steps, warmup, world,
                                                   dev, nominal_flops(shapes))
    st = binding.muon_query_status()
    if st != 0:
        raise SystemExit(f"{name}: device status {binding.muon_status_string(st)} after timing")
    line = _report(name, args, steps, warmup, world, shapes, t_ms, e2e, prof, clocks,
                   launches_per_step)
    line["ns_only"] = ns_only
    del groups, arr, flush
    torch.cuda.empty_cache()
    if samples is not None:
        line["cpu_baseline"] = cpu_baseline(name, samples, shapes)
    return line


def _ns_only(groups, stream, flush, steps, warmup, world, dev, flops):
    """Newton-Schulz alone through muon_ns_batched_ex (fp32 or bf16 input, the
    output in the input's dtype): the step's gradients, same-shape tensors
    stacked into one [B, M, N] batch per shape outside the timed region, one
    call per shape, timed like the step.  Not counted in gpu_launches (its
    own region)."""
    import torch
    from newton_schulz_gb300 import binding
    by_shape = {}
    for g in groups:
        x = g["G"] if g["G"].dim() == 3 else g["G"].unsqueeze(0)
        by_shape.setdefault((tuple(x.shape[1:]), x.dtype), []).append(x)
    xs = [torch.cat(v, 0).contiguous() for v in by_shape.values()]
    outs = [torch.empty_like(x) for x in xs]
    ms = []
    for i in range(warmup + steps):
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for x, o in zip(xs, outs):
            binding.muon_ns_batched_ex(x, out=o, stream=stream)
        b.record(stream)
        torch.cuda.synchronize()
        if i >= warmup:
            ms.append(a.elapsed_time(b))
    t = statistics.median(ms)
    del xs, outs
    if world > 1:
        import torch.distributed as dist
        tt = torch.tensor([t], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        t = float(tt.item())
    return {"ms_per_step": t, "value": world * flops / (t * 1e-3) / 1e12, "unit": "TFLOP/s",
            "calls_per_step": len(by_shape),
            "what": "muon_ns_batched_ex on the step's gradients, one call per shape"}


def _end_to_end(groups, stream, flush, steps, warmup, world, dev):
    """The step through the host-memory entry point: W, G and Mom start and
    end in pinned host memory; the library's copy-in, step and copy-out (the
    chunked pipeline of muon_step_grouped_host) are all inside the timed
    region."""
    import torch
    from newton_schulz_gb300 import binding
    host = []
    for g in groups:
        h = {}
        for k in ("W", "G", "Mom"):
            h[k] = torch.empty(g[k].shape, dtype=g[k].dtype, pin_memory=True)
            h[k].copy_(g[k])
        host.append(h)
    harr = binding.make_groups(host)
    h2d = sum(h[k].numel() * h[k].element_size() for h in host for k in ("W", "G", "Mom"))
    d2h = sum(h[k].numel() * h[k].element_size() for h in host for k in ("W", "Mom"))
    e2e_ms = []
    for i in range(warmup + max(3, steps // 2)):
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        binding.muon_step_grouped_host(harr, stream=stream, **HP)
        b.record(stream)
        torch.cuda.synchronize()
        if i >= warmup:
            e2e_ms.append(a.elapsed_time(b))
    e2e_t = statistics.median(e2e_ms)
    del host, harr
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([e2e_t], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_t = float(t.item())
    return {"ms": e2e_t, "h2d": h2d, "d2h": d2h, "steps": max(3, steps // 2)}


def _report(name, args, steps, warmup, world, shapes, t_ms, e2e, prof, clocks,
            launches_per_step):
    peaks = _peaks()
    flops = nominal_flops(shapes)
    # a timed region of seconds runs under the power cap like the sustained
    # GEMM measurement; shorter ones compare with the burst figure
    sustained = t_ms * steps > 1000.0
    tpeak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    peak_kind = "sustained" if sustained else "burst"
    # ---- roofline of the dominant kernel ------------------------------------------------
    kinds = {k: (ms / max(1, n), n) for k, (ms, n) in prof.items() if n}
    per_step_ms = {k: prof[k][0] / steps for k in prof}
    dom = max(per_step_ms, key=per_step_ms.get)
    avg_ms, n_launch = kinds[dom]
    byt = algorithmic_bytes(shapes)
    fl = gemm_flops_per_kind(shapes)
    launches_kind = n_launch / steps
    if dom in ("prep", "update", "fused_small"):
        per_launch = byt[dom] / launches_kind
        achieved = per_launch / (avg_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": _traffic(dom, name),
                "algorithmic_bytes": per_launch, "kernel": dom, "peak_source": peaks["source"]}
    else:
        per_launch = fl[dom] / launches_kind
        achieved = per_launch / (avg_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tpeak,
                "unit": "TFLOP/s", "frac": achieved / tpeak,
                "traffic": _traffic(dom, name), "algorithmic_flops": per_launch,
                "kernel": dom, "peak_source": peaks["source"], "peak_kind": peak_kind}
    per_kind = {}
    for k, (avg, n) in kinds.items():
        lk = n / steps
        if k in byt:
            a = byt[k] / lk / (avg * 1e-3) / 1e9
            per_kind[k] = {"avg_ms": avg, "GB/s": round(a, 1),
                           "frac": round(a / peaks["hbm_gbs"], 4)}
        elif k in fl:
            a = fl[k] / lk / (avg * 1e-3) / 1e12
            per_kind[k] = {"avg_ms": avg, "TFLOP/s": round(a, 1), "frac": round(a / tpeak, 4)}
    fa = alg_flops(shapes)
    alg = world * fa / (t_ms * 1e-3) / 1e12
    return {
        "metric": METRIC, "value": world * flops / (t_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
        "n_gpus": world, "steps": steps, "warmup": warmup, "ms_per_step": t_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": workload_name(name, args), "config": name,
                   "matrices": sum(s[0] for s in shapes), "nominal_gflop_per_step": flops / 1e9,
                   "alg_gflop_per_step": fa / 1e9,
                   "l2": "512 MiB L2 flush between timed steps (outside events)",
                   "parallelism": f"replica x{world}" if world > 1 else "single GPU"},
        "alg": {"value": alg, "unit": "TFLOP/s", "peak": tpeak, "peak_kind": peak_kind,
                "frac": alg / (world * tpeak),
                "what": "algorithmic flops of the products the library runs (symmetric "
                        "products once; Gram space where it is used) over the step time"},
        "e2e": None if e2e is None else {
            "value": world * flops / (e2e["ms"] * 1e-3) / 1e12, "unit": "TFLOP/s",
            "ms_per_step": e2e["ms"], "steps": e2e["steps"],
            "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"]},
        "gpu_launches": launches_per_step * steps,
        "launches_per_step": launches_per_step,
        "kernel_ms_per_step": {k: round(v, 5) for k, v in per_step_ms.items()},
        "roofline": roof,
        "kernels": per_kind,
        "clocks": clocks,
    }


# ---- extra reports -------------------------------------------------------------------------
def _owners_report(n_ranks):
    """Owner assignment across n_ranks with NS times measured per shape on
    this GPU (one assignment unit per matrix, byte cap eps = 0.1): the busiest
    rank's NS time over the mean, for LPT on the measured times, LPT on
    element counts, and round-robin in parameter order.  Two workloads: the
    224 Llama-3-8B matrices (32 layers x q, k, v, o, gate, up, down; layer
    spreading) and the 22 matrices of the large sweep."""
    from newton_schulz_gb300 import binding
    llama = [(4096, 4096), (1024, 4096), (1024, 4096), (4096, 4096),
             (14336, 4096), (14336, 4096), (4096, 14336)]
    sweep = [(8192, 28672)] * 8 + [(8192, 8192)] * 8 + [(16384, 16384)] * 4 + [(8192, 8192)] * 2
    distinct = sorted(set(llama) | set(sweep))
    ms = dict(zip(distinct, binding.muon_ns_cost_table(distinct, reps=3)))

    def report(units, layers):
        cost = [ms[s] for s in units]
        elems = [s[0] * s[1] for s in units]
        nbytes = [e * 10 for e in elems]          # bf16 W, bf16 G, fp32 Mom

        def ratio(owner):
            t = [0.0] * n_ranks
            for o, c in zip(owner, cost):
                t[o] += c
            return max(t) / (sum(t) / n_ranks)

        def bytes_ratio(owner):
            b = [0.0] * n_ranks
            for o, x in zip(owner, nbytes):
                b[o] += x
            return max(b) / (sum(b) / n_ranks)
        lpt = binding.muon_assign_owners(cost, n_ranks, nbytes, elems, layers, 0.1)
        free = binding.muon_assign_owners(cost, n_ranks, nbytes, elems, layers, 1e9)
        by_elems = binding.muon_assign_owners([float(e) for e in elems], n_ranks, nbytes, elems,
                                              layers, 0.1)
        rr = [i % n_ranks for i in range(len(units))]
        return {"lpt_measured": ratio(lpt), "lpt_measured_bytes": bytes_ratio(lpt),
                "lpt_no_byte_cap": ratio(free), "lpt_no_byte_cap_bytes": bytes_ratio(free),
                "lpt_element_count": ratio(by_elems), "round_robin": ratio(rr)}
    lu = [s for _ in range(32) for s in llama]
    rl = report(lu, [i // 7 for i in range(len(lu))])
    rs = report(sweep, [-1] * len(sweep))
    print(json.dumps({
        "metric": "owner assignment: busiest rank NS time / mean", "unit": "ratio",
        "n_ranks": n_ranks, "value": rs["lpt_measured"], "higher_is_better": False,
        "config": {"workload": "large sweep (22 matrices) and Llama-3-8B (224)", "eps": 0.1},
        "ms_per_matrix": {f"{r}x{c}": v for (r, c), v in ms.items()},
        "sweep": rs, "llama": rl}))


def _adamw_bench(args, local):
    """AdamW over the parameters Muon does not take in Llama-3-8B shapes: the
    embedding and the output head (128256 x 4096 each) and the 65 RMSNorm
    gains (4096): fp32 parameters and moments, bf16 gradients, synthetic
    values.  Algorithmic bytes per element: p r/w 8 + g 2 + m r/w 8 + v r/w 8."""
    import torch
    from newton_schulz_gb300 import binding
    dev = torch.device("cuda", local)
    rows = args.adamw_rows
    sizes = [rows * 4096, rows * 4096] + [4096] * 65
    gen = torch.Generator(device=dev).manual_seed(7)
    ts = []
    for n in sizes:
        ts.append({"param": torch.randn(n, device=dev, generator=gen) * 0.02,
                   "grad": (torch.randn(n, device=dev, generator=gen) * 1e-3).to(torch.bfloat16),
                   "exp_avg": torch.zeros(n, device=dev), "exp_avg_sq": torch.zeros(n, device=dev)})
    elems = sum(sizes)
    bytes_step = elems * 26
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    for i in range(args.warmup):
        binding.muon_adamw_grouped(ts, step=i + 1)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    ms = []
    for i in range(args.steps):
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        binding.muon_adamw_grouped(ts, step=args.warmup + i + 1)
        b.record(stream)
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    clocks = sampler.stop()
    t = statistics.median(ms)
    gbs = bytes_step / (t * 1e-3) / 1e9
    peaks = _peaks()
    print(json.dumps({
        "metric": "AdamW step over the non-matrix parameters (GB/s of algorithmic traffic)",
        "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t, "higher_is_better": True, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"Llama-3-8B non-matrix parameters: 2 x [{rows} x 4096] + 65 x [4096]",
                   "elements": elems, "l2": "512 MiB L2 flush between timed steps (outside events)"},
        "gpu_launches": args.steps * binding.muon_last_launch_count(),
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": None,
                     "algorithmic_bytes": bytes_step, "kernel": "adamw",
                     "peak_source": peaks["source"]},
        "clocks": clocks}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=None, choices=["c1", "c2", "c3", "c4", "c5"],
                    help="time one workload alone (default: all five, the large sweep as "
                         "the headline)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the host-buffer end-to-end pass")
    ap.add_argument("--no-ns-only", action="store_true",
                    help="skip the NS-only measurement (muon_ns_batched_ex on the same gradients)")
    ap.add_argument("--layers", type=int, default=None,
                    help="c4 only: number of Llama layers (default 32; a small profiling case)")
    ap.add_argument("--experts", type=int, default=None,
                    help="c3 only: experts per weight (default 128; a small profiling case)")
    ap.add_argument("--scale-down", type=int, default=1,
                    help="c5 only: divide every dimension (a small profiling case)")
    ap.add_argument("--adamw", action="store_true",
                    help="time the AdamW kernel on the Llama-3-8B non-matrix parameters instead")
    ap.add_argument("--adamw-rows", type=int, default=128256,
                    help="rows of the embedding and output head in the AdamW workload "
                         "(a smaller value gives a case small enough for a full profiler capture)")
    ap.add_argument("--owners", type=int, default=0,
                    help="report the owner-assignment balance of the Llama-3-8B matrices for N ranks")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = _dist_env()

    if args.impl == "reference":
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
        run_reference(args, world, rank)
        if world > 1:
            dist.destroy_process_group()
        return

    import torch
    from newton_schulz_gb300 import binding

    torch.cuda.set_device(local)
    binding.load()
    if args.adamw:
        _adamw_bench(args, local)
        return
    if args.owners:
        _owners_report(args.owners)
        return
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    with_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    if args.config is None and world == 1:
        per = {}
        for name in OTHERS:
            k, w = (min(args.steps, 10), 3) if name == "c4" else (args.steps, args.warmup)
            per[name] = measure(name, k, w, args, world, dev, local, with_cpu)
        line = measure(HEADLINE, args.steps, args.warmup, args, world, dev, local, with_cpu)
        line["per_config"] = per
    else:
        line = measure(args.config or HEADLINE, args.steps, args.warmup, args, world, dev, local,
                       with_cpu)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
