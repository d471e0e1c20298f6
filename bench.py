"""Benchmark of the owner-side Muon step on GB300: one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config llama7b]
                    [--method gram|standard] [--impl ours|reference]

A step is one muon_step over the whole packed group of the workload (momentum, norm,
five Newton-Schulz steps, decoupled decay and apply), plus the AdamW step of the
workload's routed-out parameters when it has any.  Inputs are synthetic (seeded,
transformer-shaped; see ``synth``) and already resident in HBM when the timed region
starts; the workload's state (tens of GB) is far larger than L2, so no flush is needed.

--impl reference times the float64 CPU oracle on a bounded sample of the same workload
and extrapolates to a full step by canonical flop count.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Muon optimizer step ms & NS TFLOP/s (frac of bf16 peak) on 1 GB300 vs CPU oracle"
NS_STEPS = 5


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


def _gram_counts(steps=NS_STEPS, every=2):
    """(products with X, square products) of the re-anchored gram form."""
    wide, cubes, q_identity = 1, 0, True
    for step in range(1, steps + 1):
        cubes += 1 if q_identity else 2
        q_identity = False
        if step < steps:
            if step % every == 0:
                wide += 2
                q_identity = True
            else:
                cubes += 2
    return wide + (0 if q_identity else 1), cubes


def _canonical_ns_flops(shapes, method):
    """Flops of the Newton-Schulz chain as the library runs it."""
    tot = 0
    wide, cubes = _gram_counts()
    for r, c in shapes:
        m, n = min(r, c), max(r, c)
        if method == "standard":
            tot += NS_STEPS * (4 * m * m * n + 2 * m ** 3)
        else:
            tot += 2 * wide * m * m * n + 2 * cubes * m ** 3
    return tot


def _describe(wl):
    shapes = sorted(set(wl.muon_shapes), key=lambda s: -s[0] * s[1])
    return {
        "workload": wl.name,
        "shapes": [f"{r}x{c}" for r, c in shapes],
        "matrices": len(wl.muon_shapes),
        "muon_elements": wl.muon_elements,
        "adam_elements": wl.adam_elements,
    }


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
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
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


def _dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_workload(name, rank):
    """The owner group rank `rank` runs: the workload's shapes with its own seed (weak
    scaling: every rank owns one group of the same size; no data crosses ranks)."""
    import synth
    wl = synth.workload(name)
    wl.seed = wl.seed + 7919 * rank
    return wl


def max_over_ranks(value, dist, device):
    """The largest of every rank's value (the step time the job sees)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# kernels whose timing work is flops (the others count bytes)
FLOP_KERNELS = ("k_ns_gemm", "k_ns_small")


def _traffic_record(method, workload):
    """Per-launch DRAM traffic of the dominant kernel from a committed ncu summary, if the
    kernel source is unchanged since the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    src = os.path.join(ROOT, "newton_schulz_orthogonalized_gb300", "csrc", "ns_gemm.cu")
    try:
        with open(path) as f:
            rec = json.load(f)
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        entry = rec.get(f"{workload}/{method}")
        if entry and entry.get("kernel_sha") == h:
            return entry.get("bytes_per_launch")
    except Exception:
        pass
    return None


def cpu_oracle_sample(wl, method, budget_s=20.0, max_flops=3e12):
    """Times the oracle on a bounded sample of the workload; returns (ms per full step
    extrapolated by canonical flops, description).  The sample is one matrix of each of
    the smallest shapes, as many as fit in max_flops canonical NS flops (at least one)."""
    import numpy as np
    import oracle
    import synth
    import torch

    order = sorted(range(len(wl.muon_shapes)), key=lambda i: wl.muon_shapes[i][0] * wl.muon_shapes[i][1])
    picked, seen = [], set()
    for i in order:
        if wl.muon_shapes[i] in seen:
            continue
        seen.add(wl.muon_shapes[i])
        if picked and _canonical_ns_flops([wl.muon_shapes[j] for j in picked + [i]], method) > max_flops:
            break
        picked.append(i)
    t_total = 0.0
    flops = 0
    for i in picked:
        r, c = wl.muon_shapes[i]
        g = synth.make_grad(r, c, wl.seed, i, "cpu", wl.lowrank).double().numpy()
        p = np.zeros((r, c))
        m = np.zeros((r, c))
        t0 = time.perf_counter()
        oracle.muon_step([g], [p], [m], wl.lr, wl.wd, wl.mu, method, storage="method")
        t_total += time.perf_counter() - t0
        flops += _canonical_ns_flops([(r, c)], method)
        if t_total > budget_s:
            break
    full = _canonical_ns_flops(wl.muon_shapes, method)
    ms = t_total * 1e3 * full / flops
    desc = (f"oracle.muon_step ({method}) on {len(picked)} matrices "
            f"({', '.join(f'{wl.muon_shapes[i][0]}x{wl.muon_shapes[i][1]}' for i in picked)}), "
            f"{t_total:.2f} s, extrapolated to the full {len(wl.muon_shapes)}-matrix step by canonical "
            f"NS flops ({flops:.3e} of {full:.3e})")
    return ms, desc


def run_reference(args):
    world, rank, local = _dist_setup(args)
    if rank != 0:
        return 0
    import synth
    wl = synth.workload(args.config)
    vals = []
    desc = ""
    for k in range(args.warmup + args.steps):
        # the cpu_baseline's sample, so that the two lines measure the same thing
        ms, desc = cpu_oracle_sample(wl, args.method, budget_s=20.0)
        if k >= args.warmup:
            vals.append(ms)
    value = statistics.median(vals)
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "ms", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": value,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": dict(_describe(wl), ns_method=args.method, ns_steps=NS_STEPS),
        "cpu_baseline": {"value": value, "unit": "ms", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_ours(args):
    import torch

    import newton_schulz_orthogonalized_gb300 as nsm
    import synth

    world, rank, local = _dist_setup(args)
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    nsm.lib()
    wl = rank_workload(args.config, rank)
    shapes = wl.muon_shapes
    method = args.method
    offsets, total = nsm.pack(shapes)
    grads = torch.empty(total, dtype=torch.bfloat16, device=dev)
    params = torch.zeros(total, dtype=torch.float32, device=dev)
    mom = torch.zeros(total, dtype=torch.float32, device=dev)
    synth.fill_packed_grads(wl, offsets, grads)
    synth.fill_packed_params(wl, offsets, params)
    ws = torch.empty(nsm.workspace_bytes(shapes, method, NS_STEPS), dtype=torch.uint8, device=dev)
    adam = None
    if wl.adam_elements:
        ag, ap = synth.make_adam_group(wl, dev)
        adam = (ag, ap, torch.zeros_like(ap), torch.zeros_like(ap))
    stream = torch.cuda.current_stream()
    adam_state = {"t": 0}

    def step():
        nsm.muon_step(grads, params, mom, offsets, shapes, wl.lr, wl.wd, wl.mu, method, NS_STEPS,
                      True, ws, stream)
        launches = nsm.last_launch_count()
        if adam is not None:
            adam_state["t"] += 1
            nsm.adamw_step(adam[0], adam[1], adam[2], adam[3], 3e-4, 0.9, 0.95, 1e-10, wl.wd,
                           adam_state["t"], stream)
            launches += nsm.last_launch_count()
        return launches

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if nsm.device_status() != nsm.NSM_OK:
        raise RuntimeError("a bounded device wait expired during warm-up")

    # ---- timed region (device events on the launching stream).  The step time comes from
    # an uninstrumented pass: events between the library's launches would serialise them
    # and hide the overlap of one kernel's tail with the next kernel's launch.
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    launches = 0
    with ClockSampler(local) as clk:
        t0.record(stream)
        for _ in range(args.steps):
            launches += step()
        t1.record(stream)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
    ms = t0.elapsed_time(t1) / args.steps
    # ---- the same number of steps again with an event pair around every launch: the
    # per-kernel times behind `kernels` and `roofline`
    nsm.timing_reset()
    nsm.timing_enable(True)
    torch.cuda.synchronize()
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    nsm.timing_enable(False)
    gemm_ms, gemm_launches, gemm_flops = nsm.timing_read(nsm.KIND_GEMM)
    per_kind = {}
    for kind, kname in nsm.KIND_NAMES.items():
        k_ms, k_n, k_work = nsm.timing_read(kind)
        if k_n:
            per_kind[kname] = (k_ms, k_n, k_work)
    if nsm.device_status() != nsm.NSM_OK:
        raise RuntimeError("a bounded device wait expired in the timed region")
    ms = max_over_ranks(ms, dist, dev)
    if dist is not None:
        dist.barrier()
    clocks = clk.summary()

    # ---- end to end through the public API with host buffers.  Every step copies its bf16
    # grads (the Muon group's and the AdamW group's) host -> device from pinned memory, runs
    # muon_step and adamw_step, and reads its result back: the bf16 copy of the updated
    # Muon parameters that the step writes (the buffer an owner broadcasts).  Two copy
    # streams and double-buffered device buffers let step k's copies overlap steps k-1 and
    # k+1.
    e2e = None
    try:
        # the same K steps as the device timing (at least 2, at most 20): the first
        # upload and the last read-back are the pipeline's only unhidden copies
        reps = max(2, min(args.steps, 20))
        h2d = torch.cuda.Stream()
        d2h = torch.cuda.Stream()
        h_grads = torch.empty(total, dtype=torch.bfloat16, pin_memory=True)
        h_grads.copy_(grads)
        h_out = torch.empty(total, dtype=torch.bfloat16, pin_memory=True)
        d_grads = [grads, torch.empty_like(grads)]
        d_out = [torch.empty(total, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        # the AdamW group's gradients are inputs of the step too
        h_agrads = d_agrads = None
        if adam is not None:
            h_agrads = torch.empty(adam[0].numel(), dtype=torch.bfloat16, pin_memory=True)
            h_agrads.copy_(adam[0])
            d_agrads = [adam[0], torch.empty_like(adam[0])]
        ev = lambda: torch.cuda.Event()

        def upload(slot):
            d_grads[slot].copy_(h_grads, non_blocking=True)
            if d_agrads is not None:
                d_agrads[slot].copy_(h_agrads, non_blocking=True)

        def pipeline():
            h2d_done, comp_done, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(h2d)
            with torch.cuda.stream(h2d):
                upload(0)
                h2d_done[0].record(h2d)
            for k in range(reps):
                cur, nxt = k % 2, (k + 1) % 2
                stream.wait_event(h2d_done[cur])
                if k >= 2:
                    stream.wait_event(d2h_done[cur])  # step k-2's result has left d_out[cur]
                nsm.muon_step(d_grads[cur], params, mom, offsets, shapes, wl.lr, wl.wd, wl.mu, method,
                              NS_STEPS, True, ws, stream, params_bf16=d_out[cur])
                if adam is not None:
                    adam_state["t"] += 1
                    nsm.adamw_step(d_agrads[cur], adam[1], adam[2], adam[3], 3e-4, 0.9, 0.95, 1e-10, wl.wd,
                                   adam_state["t"], stream)
                comp_done[cur].record(stream)
                if k + 1 < reps:
                    with torch.cuda.stream(h2d):
                        if k >= 1:
                            h2d.wait_event(comp_done[nxt])  # step k-1 is done with d_grads[nxt]
                        upload(nxt)
                        h2d_done[nxt].record(h2d)
                with torch.cuda.stream(d2h):
                    d2h.wait_event(comp_done[cur])
                    h_out.copy_(d_out[cur], non_blocking=True)
                    d2h_done[cur].record(d2h)
            h2d.wait_stream(d2h)
            e1.record(h2d)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / reps

        # Host<->device copy speed on these machines varies from pass to pass while the
        # GPU runs at its power cap, so one untimed pass warms the pinned buffers and the
        # median of three timed passes is reported (all three are listed).
        pipeline()
        passes = [pipeline() for _ in range(3)]
        h2d_bytes = total * 2 + (adam[0].numel() * 2 if adam is not None else 0)
        e2e = {"value": sorted(passes)[1], "unit": "ms",
               "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": total * 2,
               "steps": reps, "passes_ms": passes, "statistic": "median of 3 timed passes",
               "overlap": "copies on two streams, double-buffered"}
        del h_grads, h_out, d_grads, d_out, h_agrads, d_agrads
    except Exception as exc:  # pinned memory may be unavailable on a host
        e2e = {"value": None, "unit": "ms", "h2d_bytes_per_step": total * 2,
               "d2h_bytes_per_step": total * 2, "error": str(exc)[:200]}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peaks = _peaks()
    per_launch_ms = gemm_ms / max(gemm_launches, 1)
    per_launch_flops = gemm_flops / max(gemm_launches, 1)
    achieved_tflops = per_launch_flops / (per_launch_ms * 1e-3) / 1e12 if gemm_ms > 0 else None
    peak = peaks["bf16_tflops_sustained"]
    ns_flops = _canonical_ns_flops(shapes, method)
    ns_ms_per_step = gemm_ms / args.steps
    line = {
        "metric": METRIC,
        "value": ms * 1.0,
        "unit": "ms",
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if method == "standard" else "f16",
        "data": "synthetic",
        "config": dict(_describe(wl), ns_method=method, ns_steps=NS_STEPS,
                       l2="inputs larger than L2 (no flush)",
                       parallelism="replicas" if args.gpus > 1 else "single"),
        "ns_chain_ms_per_step": ns_ms_per_step,
        "ns_tflops": ns_flops / (ns_ms_per_step * 1e-3) / 1e12 if ns_ms_per_step > 0 else None,
        "ns_frac_of_peak": (ns_flops / (ns_ms_per_step * 1e-3) / 1e12) / peak if ns_ms_per_step > 0 else None,
        "matrices_per_s": len(shapes) / (ms * 1e-3) * args.gpus,
        "roofline": {
            "kernel": "k_ns_gemm",
            "bound": "tensor",
            "achieved": achieved_tflops,
            "peak": peak,
            "peak_kind": f"bf16 sustained ({peaks['source']}); fp16 nominal ratio 1:1" if method == "gram"
                         else f"bf16 sustained ({peaks['source']})",
            "unit": "TFLOP/s",
            "frac": achieved_tflops / peak if achieved_tflops else None,
            "traffic": _traffic_record(method, wl.name),
            "launches_timed": gemm_launches,
            "flops_per_launch": per_launch_flops,
            "ms_per_launch": per_launch_ms,
            "timing": "CUDA events around every launch, in a second timed pass of the same steps",
        },
        "kernels": {
            kname: {
                "launches": k_n,
                "ms_per_step": k_ms / args.steps,
                "achieved": (k_work / (k_ms * 1e-3) / (1e12 if kname in FLOP_KERNELS else 1e9)) if k_ms > 0 else None,
                "unit": "TFLOP/s" if kname in FLOP_KERNELS else "GB/s",
                "frac": ((k_work / (k_ms * 1e-3) / 1e12) / peak if kname in FLOP_KERNELS
                         else (k_work / (k_ms * 1e-3) / 1e9) / peaks["hbm_gbs"]) if k_ms > 0 else None,
            }
            for kname, (k_ms, k_n, k_work) in per_kind.items()
        },
        "gpu_launches": launches,
        "clocks": clocks,
        "e2e": e2e,
    }
    if not args.no_cpu_baseline:
        ms_cpu, desc = cpu_oracle_sample(wl, method, budget_s=20.0)
        line["cpu_baseline"] = {"value": ms_cpu, "unit": "ms", "cores": os.cpu_count(),
                                "kind": "oracle", "sample": desc}
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="llama7b")
    ap.add_argument("--method", default="gram", choices=["gram", "standard"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
