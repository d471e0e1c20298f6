"""Benchmark of the owner-side Muon step on GB300: one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config llama7b]
                    [--method gram|standard] [--impl ours|reference] [--no-other-configs]

A step is one muon_step over the whole packed group of the workload (momentum, norm,
five Newton-Schulz steps, decoupled decay and apply), plus the AdamW step of the
workload's routed-out parameters when it has any.  Inputs are synthetic (seeded,
transformer-shaped; see ``synth``) and already resident in HBM when the timed region
starts; the workload's state (tens of GB) is far larger than L2, so no flush is needed.
The line also carries, for the other workloads, a few timed steps each
(``other_configs``).

--impl reference times the float64 CPU oracle on a bounded sample of the same workload:
every step times the oracle on one matrix of one of the workload's distinct shapes (the
first step on all of them) and reports the full step that the latest time of every shape
implies, weighting each shape by its count in the table.
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
OTHER_CONFIGS = ("tiny", "layer1024", "gpt2small", "split_moe")


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


# the library re-anchors the gram form's R from the explicit iterate every 3 steps
GRAM_REANCHOR_EVERY = 3


def _gram_counts(steps=NS_STEPS, every=GRAM_REANCHOR_EVERY):
    """(products with X, square products) of the gram form re-anchored every `every`
    steps (every = 0: never)."""
    wide, cubes, q_identity = 1, 0, True
    for step in range(1, steps + 1):
        cubes += 1 if q_identity else 2
        q_identity = False
        if step < steps:
            if every and step % every == 0:
                wide += 2
                q_identity = True
            else:
                cubes += 2
    return wide + (0 if q_identity else 1), cubes


def _chain_flops(shapes, method, every):
    tot = 0
    wide, cubes = _gram_counts(NS_STEPS, every)
    for r, c in shapes:
        m, n = min(r, c), max(r, c)
        if method == "standard":
            tot += NS_STEPS * (4 * m * m * n + 2 * m ** 3)
        else:
            tot += 2 * wide * m * m * n + 2 * cubes * m ** 3
    return tot


def _canonical_ns_flops(shapes, method):
    """The method's canonical flop count: 5 (4 m^2 n + 2 m^3) per matrix for the standard
    form, 4 m^2 n + 34 m^3 for the gram form iterated on R without re-anchoring."""
    return _chain_flops(shapes, method, every=0)


def _dense_ns_flops(shapes, method):
    """Flops of the chain as the library runs it (the gram form re-anchored every 3
    steps), counted as if every tile of every product were computed."""
    return _chain_flops(shapes, method, every=GRAM_REANCHOR_EVERY)


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


def owner_workload(nsm, name, rank, world, method):
    """The matrices rank `rank` owns when one table is split by dedicated ownership
    (DMuon: LPT on Newton-Schulz flops, `nsm_assign_owners`): strong scaling, every matrix
    on exactly one rank, the AdamW group on rank 0.  Matrix names, shapes and the
    workload's hyperparameters are kept; the seed is the table's."""
    import dataclasses

    import synth
    wl = synth.workload(name)
    owner, _ = nsm.assign_owners(wl.muon_shapes, world, method)
    idx = [i for i, o in enumerate(owner) if int(o) == rank]
    return dataclasses.replace(
        wl, name=f"{wl.name}/owner{rank}of{world}",
        muon_names=[wl.muon_names[i] for i in idx], muon_shapes=[wl.muon_shapes[i] for i in idx],
        adam_names=wl.adam_names if rank == 0 else [], adam_shapes=wl.adam_shapes if rank == 0 else [])


def synth_table(name):
    import synth
    return synth.workload(name).muon_shapes


def max_over_ranks(value, dist, device):
    """The largest of every rank's value (the step time the job sees)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# kernels whose timing work is flops (the others count bytes)
FLOP_KERNELS = ("k_ns_gemm",)


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


# ---------------------------------------------------------------- the oracle on the host

def _shape_counts(wl):
    """Distinct shapes of the table, smallest first, with the index of their first matrix
    and their count."""
    counts, first = {}, {}
    for i, sh in enumerate(wl.muon_shapes):
        counts[sh] = counts.get(sh, 0) + 1
        first.setdefault(sh, i)
    order = sorted(counts, key=lambda s: s[0] * s[1])
    return [(sh, first[sh], counts[sh]) for sh in order]


def _time_oracle_matrix(wl, method, sh, index):
    """Seconds the float64 oracle takes for one whole step of one matrix of shape sh."""
    import numpy as np
    import oracle
    import synth
    r, c = sh
    g = synth.make_grad(r, c, wl.seed, index, "cpu", wl.lowrank).double().numpy()
    p = np.zeros((r, c))
    m = np.zeros((r, c))
    t0 = time.perf_counter()
    oracle.muon_step([g], [p], [m], wl.lr, wl.wd, wl.mu, method)
    return time.perf_counter() - t0


def _time_oracle_adamw(wl, max_elems=16 * 1024 * 1024):
    """Seconds the oracle's AdamW takes on the workload's whole AdamW group, timed on up to
    max_elems of it and scaled linearly (every element costs the same); 0 without one."""
    import numpy as np
    import oracle
    import synth
    n = wl.adam_elements
    if not n:
        return 0.0
    k = min(n, max_elems)
    g16, p = synth.make_adam_group(wl, "cpu")
    g = g16[:k].double().numpy()
    pp = p[:k].double().numpy()
    z = np.zeros(k)
    t0 = time.perf_counter()
    oracle.adamw_step(g, pp, z, z, 3e-4, 0.9, 0.95, 1e-10, wl.wd, 1)
    return (time.perf_counter() - t0) * n / k


def cpu_oracle_sample(wl, method, budget_s=30.0):
    """Times the float64 oracle (the exact iteration) on one matrix of each distinct shape
    of the workload, smallest shapes first, until the budget is spent (at least one); the
    full step is the sum over shapes of count x time, scaled by the share of the table's
    matrices whose shape was timed when the budget ran out.  Returns (ms per full step,
    description)."""
    shapes = _shape_counts(wl)
    times = {}
    spent = 0.0
    for sh, idx, _ in shapes:
        if times and spent > budget_s:
            break
        t = _time_oracle_matrix(wl, method, sh, idx)
        times[sh] = t
        spent += t
    covered = sum(cnt for sh, _, cnt in shapes if sh in times)
    est = sum(cnt * times[sh] for sh, _, cnt in shapes if sh in times) * len(wl.muon_shapes) / covered
    adam = _time_oracle_adamw(wl)
    desc = (f"oracle.muon_step ({method}, exact float64 iteration) on one matrix of each of "
            f"{len(times)} of the {len(shapes)} distinct shapes "
            f"({', '.join(f'{r}x{c} {times[(r, c)]:.2f} s' for (r, c) in times)}); the full "
            f"{len(wl.muon_shapes)}-matrix step is extrapolated as the sum over shapes of count x time"
            + (f"; plus oracle.adamw_step on the {wl.adam_elements}-element AdamW group ({adam:.2f} s, "
               f"timed on up to 16M elements and scaled)" if wl.adam_elements else ""))
    return (est + adam) * 1e3, desc


def run_reference(args):
    world, rank, local = _dist_setup(args)
    if rank != 0:
        return 0
    import synth
    wl = synth.workload(args.config)
    shapes = _shape_counts(wl)
    latest = {}
    vals = []
    adam = 0.0
    for k in range(args.warmup + args.steps):
        if k == 0:
            for sh, idx, _ in shapes:
                latest[sh] = _time_oracle_matrix(wl, args.method, sh, idx)
            adam = _time_oracle_adamw(wl)
        else:
            sh, idx, _ = shapes[(k - 1) % len(shapes)]
            latest[sh] = _time_oracle_matrix(wl, args.method, sh, idx)
        ms = 1e3 * (sum(cnt * latest[sh] for sh, _, cnt in shapes) + adam)
        if k >= args.warmup:
            vals.append(ms)
    value = statistics.median(vals)
    cores = os.cpu_count()
    desc = (f"oracle.muon_step ({args.method}, exact float64 iteration): the first step times one "
            f"matrix of each of the {len(shapes)} distinct shapes, every later step re-times one "
            f"shape in turn; each step reports the sum over shapes of count x latest time "
            f"(median of {args.steps} timed steps)"
            + (f", plus oracle.adamw_step on the {wl.adam_elements}-element AdamW group timed once "
               f"({adam:.2f} s)" if wl.adam_elements else ""))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "ms", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": value,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": dict(_describe(wl), ns_method=args.method, ns_steps=NS_STEPS),
        "cpu_baseline": {"value": value, "unit": "ms", "cores": cores, "kind": "oracle", "sample": desc,
                         "extrapolated": True},
        "e2e": {"value": value, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- the GPU path

class Setup:
    """Device buffers of one workload's step."""

    def __init__(self, nsm, wl, method, dev):
        import torch
        import synth
        self.wl, self.method, self.dev = wl, method, dev
        self.shapes = wl.muon_shapes
        self.offsets, self.total = nsm.pack(self.shapes)
        self.grads = torch.empty(self.total, dtype=torch.bfloat16, device=dev)
        self.params = torch.zeros(self.total, dtype=torch.float32, device=dev)
        self.mom = torch.zeros(self.total, dtype=torch.float32, device=dev)
        synth.fill_packed_grads(wl, self.offsets, self.grads)
        synth.fill_packed_params(wl, self.offsets, self.params)
        self.ws = torch.empty(nsm.workspace_bytes(self.shapes, method, NS_STEPS), dtype=torch.uint8, device=dev)
        self.adam = None
        if wl.adam_elements:
            ag, ap = synth.make_adam_group(wl, dev)
            self.adam = (ag, ap, torch.zeros_like(ap), torch.zeros_like(ap))
        self.t = 0

    def step(self, nsm, stream, grads=None, params_bf16=None, adam_grads=None):
        nsm.muon_step(self.grads if grads is None else grads, self.params, self.mom, self.offsets, self.shapes,
                      self.wl.lr, self.wl.wd, self.wl.mu, self.method, NS_STEPS, True, self.ws, stream,
                      params_bf16=params_bf16)
        launches = nsm.last_launch_count()
        if self.adam is not None:
            self.t += 1
            nsm.adamw_step(self.adam[0] if adam_grads is None else adam_grads, self.adam[1], self.adam[2],
                           self.adam[3], 3e-4, 0.9, 0.95, 1e-10, self.wl.wd, self.t, stream)
            launches += nsm.last_launch_count()
        return launches


def _timed_steps(nsm, S, stream, steps):
    """Device ms per step over `steps` uninstrumented steps (CUDA events on the stream)."""
    import torch
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    launches = 0
    t0.record(stream)
    for _ in range(steps):
        launches += S.step(nsm, stream)
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps, launches


def _orthogonalize_block(nsm, S, stream, calls, executed_per_call, peak):
    """muon_orthogonalize alone over the step's table (the Newton-Schulz-only number):
    device ms per call over `calls` uninstrumented calls after one warm call (CUDA events
    on the stream), and its rates on the chain's canonical and executed flops."""
    import torch
    out = torch.empty_like(S.grads)

    def call():
        nsm.muon_orthogonalize(S.grads, out, S.offsets, S.shapes, S.method, NS_STEPS, S.ws, stream)

    call()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(calls):
        call()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / calls
    del out
    executed = executed_per_call / (ms * 1e-3) / 1e12 if executed_per_call else None
    return {"ms": ms, "calls": calls,
            "tflops_canonical": _canonical_ns_flops(S.shapes, S.method) / (ms * 1e-3) / 1e12,
            "tflops_executed": executed,
            "frac_executed": executed / peak if executed else None,
            "includes": "the layout pass from the bf16 input, the whole chain and the export of O as bf16"}


def _kernel_times(nsm, S, stream, steps):
    """Per kernel kind: (ms, launches, work) over `steps` steps with an event pair around
    every launch."""
    import torch
    nsm.timing_reset()
    nsm.timing_enable(True)
    torch.cuda.synchronize()
    for _ in range(steps):
        S.step(nsm, stream)
    torch.cuda.synchronize()
    nsm.timing_enable(False)
    per_kind = {}
    for kind, kname in nsm.KIND_NAMES.items():
        k_ms, k_n, k_work = nsm.timing_read(kind)
        if k_n:
            per_kind[kname] = (k_ms, k_n, k_work)
    return per_kind


def _kernels_block(per_kind, steps, peaks):
    peak_t = peaks["bf16_tflops_sustained"]
    out = {}
    for kname, (k_ms, k_n, k_work) in per_kind.items():
        flops = kname in FLOP_KERNELS
        # work 0: a pass whose bytes depend on the data (the step's second layout pass,
        # which rewrites only matrices whose exponent was out of range)
        ach = (k_work / (k_ms * 1e-3) / (1e12 if flops else 1e9)) if k_ms > 0 and k_work > 0 else None
        out[kname] = {"launches": k_n, "ms_per_step": k_ms / steps, "achieved": ach,
                      "unit": "TFLOP/s" if flops else "GB/s",
                      "frac": (ach / (peak_t if flops else peaks["hbm_gbs"])) if ach else None}
    return out


def _e2e(nsm, S, stream, reps, upload_by="mapped", sm_ctas=16):
    """The step end to end through the public API with host buffers: every step moves
    its bf16 grads (and the AdamW group's) from pinned host memory to the GPU, runs the
    step, and reads back the bf16 copy of the updated Muon parameters that the step
    writes.  upload_by "mapped" (the default): the step's first pass reads the pinned
    grads in place, over the host link, once; "engine" / "sm": a copy before the step, by
    the copy engine or by SM loads, on its own stream, triple-buffered so that uploads run
    up to two steps ahead of the compute.  The read-back runs one step behind the compute
    on a second copy stream.  Every copy and every step is bracketed by events on its own
    stream, so the line records where the time went."""
    import torch
    dev = S.dev
    h2d = torch.cuda.Stream()
    d2h = torch.cuda.Stream()
    # the host copy of the grads is filled by the CPU (a device-to-host copy into pageable
    # memory, then a host memcpy), as a data loader would leave it
    h_grads = torch.empty(S.total, dtype=torch.bfloat16, pin_memory=True)
    h_grads.copy_(S.grads.cpu())
    h_out = torch.empty(S.total, dtype=torch.bfloat16, pin_memory=True)
    nbuf = 3
    d_grads = [S.grads] + [torch.empty_like(S.grads) for _ in range(nbuf - 1)]
    d_out = [torch.empty(S.total, dtype=torch.bfloat16, device=dev) for _ in range(nbuf)]
    h_agrads = d_agrads = None
    if S.adam is not None:
        h_agrads = torch.empty(S.adam[0].numel(), dtype=torch.bfloat16, pin_memory=True)
        h_agrads.copy_(S.adam[0].cpu())
        d_agrads = [S.adam[0]] + [torch.empty_like(S.adam[0]) for _ in range(nbuf - 1)]
    ev = lambda: torch.cuda.Event(enable_timing=True)

    mapped = upload_by == "mapped"
    if mapped:
        # the step reads the pinned grads through their device mapping; where the host
        # memory has none (nsm_copy_to_device checks the same thing), the copy engine
        # uploads them instead and the line says so
        try:
            probe = torch.empty(8, dtype=torch.bfloat16, device=dev)
            nsm.copy_to_device(probe, h_grads[:8], stream)
            torch.cuda.synchronize()
        except nsm.NsmError:
            mapped, upload_by = False, "engine"

    def upload(slot):
        # the library's SM-load upload (nsm_copy_to_device) or the copy engine; mapped:
        # nothing to copy, the step's first pass reads the page-locked grads in place
        if mapped:
            return
        if upload_by == "sm":
            nsm.copy_to_device(d_grads[slot], h_grads, h2d, sm_ctas)
            if d_agrads is not None:
                nsm.copy_to_device(d_agrads[slot], h_agrads, h2d, sm_ctas)
        else:
            d_grads[slot].copy_(h_grads, non_blocking=True)
            if d_agrads is not None:
                d_agrads[slot].copy_(h_agrads, non_blocking=True)

    def pipeline():
        up = [(ev(), ev()) for _ in range(reps)]
        cp = [(ev(), ev()) for _ in range(reps)]
        dn = [(ev(), ev()) for _ in range(reps)]
        torch.cuda.synchronize()
        e0, e1 = ev(), ev()
        e0.record(h2d)

        def issue_upload(j):
            with torch.cuda.stream(h2d):
                if j >= nbuf:
                    h2d.wait_event(cp[j - nbuf][1])  # step j - nbuf is done with the slot
                up[j][0].record(h2d)
                upload(j % nbuf)
                up[j][1].record(h2d)

        for j in range(min(nbuf - 1, reps)):
            issue_upload(j)
        for k in range(reps):
            cur = k % nbuf
            stream.wait_event(up[k][1])
            if k >= nbuf:
                stream.wait_event(dn[k - nbuf][1])  # step k - nbuf's result has left d_out[cur]
            cp[k][0].record(stream)
            S.step(nsm, stream, grads=h_grads if mapped else d_grads[cur], params_bf16=d_out[cur],
                   adam_grads=None if d_agrads is None else (h_agrads if mapped else d_agrads[cur]))
            cp[k][1].record(stream)
            if k + nbuf - 1 < reps:
                issue_upload(k + nbuf - 1)
            with torch.cuda.stream(d2h):
                d2h.wait_event(cp[k][1])
                dn[k][0].record(d2h)
                h_out.copy_(d_out[cur], non_blocking=True)
                dn[k][1].record(d2h)
        h2d.wait_stream(d2h)
        e1.record(h2d)
        torch.cuda.synchronize()
        dur = lambda p: p[0].elapsed_time(p[1])
        return {"ms_per_step": e0.elapsed_time(e1) / reps,
                "h2d_ms_per_step": statistics.mean(dur(p) for p in up),
                "compute_ms_per_step": statistics.mean(dur(p) for p in cp),
                "d2h_ms_per_step": statistics.mean(dur(p) for p in dn),
                "first_upload_ms": dur(up[0]), "last_download_ms": dur(dn[-1])}

    # Host<->device copy speed varies between machines of the pool (and, on some, from
    # pass to pass), so one untimed pass warms the pinned buffers and the median of three
    # timed passes is reported, with every pass's breakdown.
    pipeline()
    passes = [pipeline() for _ in range(3)]
    med = sorted(passes, key=lambda p: p["ms_per_step"])[1]
    h2d_bytes = S.total * 2 + (S.adam[0].numel() * 2 if S.adam is not None else 0)
    res = {"value": med["ms_per_step"], "unit": "ms",
           "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": S.total * 2,
           "steps": reps, "statistic": "median of 3 timed passes",
           "overlap": "copies on two streams, triple-buffered (uploads up to two steps ahead)",
           "upload": (f"SM loads over the host link (nsm_copy_to_device, {sm_ctas} CTAs)" if upload_by == "sm"
                      else "read in place from page-locked host memory by the step's first pass (inside compute)"
                      if mapped else "copy engine (cudaMemcpyAsync)"),
           "download": "copy engine (cudaMemcpyAsync)",
           "breakdown": {k: med[k] for k in med if k != "ms_per_step"},
           "h2d_gbs": None if mapped else h2d_bytes / (med["h2d_ms_per_step"] * 1e-3) / 1e9,
           "d2h_gbs": S.total * 2 / (med["d2h_ms_per_step"] * 1e-3) / 1e9,
           "passes_ms": [p["ms_per_step"] for p in passes]}
    # the bound: the slowest of the three streams per step
    res["bound"] = max(("compute", med["compute_ms_per_step"]), ("h2d", med["h2d_ms_per_step"]),
                       ("d2h", med["d2h_ms_per_step"]), key=lambda t: t[1])[0]
    return res


def _graph_steps(nsm, S, steps):
    """Device ms per step of the step captured in a CUDA graph (10 steps per graph) and
    replayed: the launch-bound small tables' remedy (the plan is cached first, so a
    captured step launches kernels only)."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        S.step(nsm, side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for _ in range(10):
            S.step(nsm, side)
    graph.replay()
    torch.cuda.synchronize()
    reps = max(1, steps // 10)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        graph.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / (10 * reps)


def _other_configs(nsm, names, method, dev, stream, peaks):
    """A few timed steps of each other workload (device step ms, kernel rates)."""
    import torch
    out = {}
    for name in names:
        try:
            import synth
            wl = synth.workload(name)
            S = Setup(nsm, wl, method, dev)
            steps = 20 if wl.muon_elements < 1e9 else 5
            for _ in range(3):
                S.step(nsm, stream)
            ms, launches = _timed_steps(nsm, S, stream, steps)
            per_kind = _kernel_times(nsm, S, stream, steps)
            if nsm.device_status() != nsm.NSM_OK:
                raise RuntimeError("a bounded device wait expired")
            kb = _kernels_block(per_kind, steps, peaks)
            graph_ms = _graph_steps(nsm, S, 50) if wl.muon_elements < 1e9 else None
            g_ms, g_launches, g_flops = per_kind.get("k_ns_gemm", (0.0, 0, 0.0))
            ortho = _orthogonalize_block(nsm, S, stream, max(2, min(steps, 10)), g_flops / steps,
                                         peaks["bf16_tflops_sustained"]) if wl.muon_shapes else None
            out[name] = {"ms_per_step": ms, "steps": steps, "matrices": len(wl.muon_shapes),
                         "graph_ms_per_step": graph_ms,
                         "orthogonalize_ms": ortho["ms"] if ortho else None,
                         "ns_tflops_canonical": ortho["tflops_canonical"] if ortho else None,
                         "muon_elements": wl.muon_elements, "adam_elements": wl.adam_elements,
                         "gpu_launches_per_step": launches / steps,
                         "gemm_frac_executed": kb.get("k_ns_gemm", {}).get("frac"),
                         "adamw_gbs": kb.get("k_adamw", {}).get("achieved"),
                         "adamw_frac": kb.get("k_adamw", {}).get("frac"),
                         "kernels": kb}
            del S
        except Exception as exc:
            out[name] = {"error": str(exc)[:200]}
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch

    import newton_schulz_orthogonalized_gb300 as nsm

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
    owners = args.split == "owners"
    wl = owner_workload(nsm, args.config, rank, world, args.method) if owners else rank_workload(args.config, rank)
    if not wl.muon_shapes:
        raise RuntimeError(f"rank {rank} owns no matrix of {args.config} at {world} ranks")
    method = args.method
    S = Setup(nsm, wl, method, dev)
    shapes = S.shapes
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        S.step(nsm, stream)
    torch.cuda.synchronize()
    if nsm.device_status() != nsm.NSM_OK:
        raise RuntimeError("a bounded device wait expired during warm-up")

    # ---- timed region (device events on the launching stream).  The step time comes from
    # an uninstrumented pass: events between the library's launches would serialise them.
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ms, launches = _timed_steps(nsm, S, stream, args.steps)
        if dist is not None:
            dist.barrier()
    # ---- the same number of steps again with an event pair around every launch: the
    # per-kernel times behind `kernels` and `roofline`
    per_kind = _kernel_times(nsm, S, stream, args.steps)
    gemm_ms, gemm_launches, gemm_flops = per_kind.get("k_ns_gemm", (0.0, 0, 0.0))
    if nsm.device_status() != nsm.NSM_OK:
        raise RuntimeError("a bounded device wait expired in the timed region")
    ms = max_over_ranks(ms, dist, dev)
    if dist is not None:
        dist.barrier()
    clocks = clk.summary()

    # ---- end to end through the public API with host buffers
    try:
        e2e = _e2e(nsm, S, stream, max(2, min(args.steps, 20)), args.upload)
    except Exception as exc:  # pinned memory may be unavailable on a host
        e2e = {"value": None, "unit": "ms", "h2d_bytes_per_step": S.total * 2,
               "d2h_bytes_per_step": S.total * 2, "error": str(exc)[:200]}

    peaks = _peaks()
    kernels = _kernels_block(per_kind, args.steps, peaks)
    # ---- the orthogonalisation alone (muon_orthogonalize) over the same table
    try:
        ortho = _orthogonalize_block(nsm, S, stream, max(2, min(args.steps, 5)),
                                     gemm_flops / max(args.steps, 1), peaks["bf16_tflops_sustained"])
    except Exception as exc:
        ortho = {"error": str(exc)[:200]}
    del S
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    others = None
    if rank == 0 and not args.no_other_configs:
        others = _other_configs(nsm, [c for c in OTHER_CONFIGS if c != args.config], method, dev, stream, peaks)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    per_launch_ms = gemm_ms / max(gemm_launches, 1)
    per_launch_flops = gemm_flops / max(gemm_launches, 1)
    achieved_tflops = per_launch_flops / (per_launch_ms * 1e-3) / 1e12 if gemm_ms > 0 else None
    peak = peaks["bf16_tflops_sustained"]
    ns_ms_per_step = gemm_ms / args.steps
    tflops = lambda f: f / (ns_ms_per_step * 1e-3) / 1e12 if ns_ms_per_step > 0 else None
    line = {
        "metric": METRIC,
        "value": ms * 1.0,
        "unit": "ms",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": False,
        "scaling": "strong" if owners else "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic",
        "config": dict(_describe(wl), ns_method=method, ns_steps=NS_STEPS,
                       storage="fp16 iterates, fp32 tensor-core accumulation; bf16 grads, fp32 params/momentum",
                       l2="inputs larger than L2 (no flush)",
                       parallelism=(f"dmuon-owners{world}" if owners else "replicas") if world > 1 else "single"),
        "ns_chain_ms_per_step": ns_ms_per_step,
        # the chain's canonical flops (standard 5(4m^2n+2m^3), gram 4m^2n+34m^3 per matrix)
        # and the dense flops of the chain as run (gram re-anchored), over the GEMM time
        "ns_tflops_canonical": tflops(_canonical_ns_flops(shapes, method)),
        "ns_tflops_dense": tflops(_dense_ns_flops(shapes, method)),
        "ns_frac_executed": achieved_tflops / peak if achieved_tflops else None,
        # matrices of the whole job per second: every rank's table (replicas), or the one
        # table the ranks share (owners)
        "matrices_per_s": (len(synth_table(args.config)) if owners else len(shapes) * world) / (ms * 1e-3),
        "roofline": {
            "kernel": "k_ns_gemm",
            "bound": "tensor",
            "achieved": achieved_tflops,
            "peak": peak,
            "peak_kind": f"bf16 sustained ({peaks['source']}); fp16 at the nominal 1:1 ratio",
            "unit": "TFLOP/s",
            "frac": achieved_tflops / peak if achieved_tflops else None,
            "traffic": _traffic_record(method, wl.name),
            "launches_timed": gemm_launches,
            "flops_per_launch": per_launch_flops,
            "flops_counted": "executed: the tiles launched, clipped to the matrix edges; upper-triangle tiles of symmetric outputs",
            "ms_per_launch": per_launch_ms,
            "timing": "CUDA events around every launch, in a second timed pass of the same steps",
        },
        "kernels": kernels,
        "orthogonalize": ortho,
        "gpu_launches": launches,
        "clocks": clocks,
        "e2e": e2e,
    }
    if others is not None:
        line["other_configs"] = others
    if not args.no_cpu_baseline:
        ms_cpu, desc = cpu_oracle_sample(wl, method)
        line["cpu_baseline"] = {"value": ms_cpu, "unit": "ms", "cores": os.cpu_count(),
                                "kind": "oracle", "sample": desc, "extrapolated": True}
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
    ap.add_argument("--no-other-configs", action="store_true")
    ap.add_argument("--upload", default="mapped", choices=["mapped", "engine", "sm"],
                    help="e2e: grads read in place from page-locked host memory by the step's first pass "
                         "(mapped, the default), or uploaded before the step by the copy engine or by SM "
                         "loads (nsm_copy_to_device)")
    ap.add_argument("--split", default="replicas", choices=["replicas", "owners"],
                    help="N > 1: every rank runs its own copy of the table (replicas, weak scaling), "
                         "or one table is split among the ranks by dedicated ownership (owners, "
                         "strong scaling)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
