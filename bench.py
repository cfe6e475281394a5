"""Benchmark of the owner-side Muon step on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl reference] [--no-e2e] [--no-cpu-baseline]

Prints one JSON line.  `value` is the Muon step time (ms, lower is better) of
the whole projection set with inputs resident in HBM; `e2e` is the same step
through `dmuon_muon_step` with the gradients copied in from pinned host memory
and the updated weights copied back inside the timed region.  The roofline
entry covers the Newton-Schulz product kernel (tcgen05, bf16), which takes
more than 90% of the step.  `--impl reference` times the fp64 CPU oracle on a
bounded sample of the same workload instead.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "llama-3.1-8b"
METRIC = "Muon step ms & NS TFLOP/s per model projection set (1 GB300); % bf16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 2 ** 20


def _rank_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region.  Each
    sample keeps its host arrival time, so that a short timed region can be
    summarised from its own samples only (`stop(window=(t0, t1))`, times from
    time.monotonic()) rather than from idle ones around it."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def stop(self, window=None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)
        sm, smax, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, ln in self.lines:
            if window is not None and not (window[0] <= t <= window[1]):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                pw.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_median": statistics.median(pw) if pw else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def blas_name() -> str:
    """The BLAS library numpy (and so the oracle) runs on."""
    try:
        import numpy as np
        b = np.show_config(mode="dicts").get("Build Dependencies", {}).get("blas", {})
        return f"{b.get('name', '?')} {b.get('version', '')}".strip()
    except Exception:
        return "unknown"


def traffic_record():
    """DRAM bytes per launch of the product kernel from the committed ncu summary,
    valid only while the kernel source is unchanged (else None)."""
    rec = os.path.join(ROOT, "profiles", "ns_gemm_traffic.json")
    src = os.path.join(ROOT, "newton_schulz_owner_gb300", "csrc", "ns_gemm.cu")
    if not os.path.exists(rec):
        return None
    with open(rec) as f:
        d = json.load(f)
    with open(src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()
    if d.get("source_sha256") != h:
        return None
    return d


def ns_flops(shapes, ns_steps: int) -> float:
    """Algorithmic flops of the standard iteration: per step X X^T (m^2 n,
    symmetric, counted half), A A (m^3, half) and B X (2 m^2 n)."""
    return float(sum((3.0 * min(s) ** 2 * max(s) + float(min(s)) ** 3) * ns_steps
                     for s in shapes))


def nominal_flops(shapes, ns_steps: int) -> float:
    """Nominal dense flops of the standard iteration, every product counted in
    full (X X^T 2 m^2 n, A A 2 m^3, B X 2 m^2 n): the count a dense GEMM library
    would report for the same products."""
    return float(sum((4.0 * min(s) ** 2 * max(s) + 2.0 * float(min(s)) ** 3) * ns_steps
                     for s in shapes))


def gram_flops(shapes, ns_steps: int) -> float:
    """Algorithmic flops of the Gram iteration: A0 = X0 X0^T (m^2 n, half) and
    O = Q X0 (2 m^2 n), and per step the symmetric m^3 products A A, P Q (not
    at the first step, where Q = P), P P and A P^2 (not at the last step)."""
    if ns_steps <= 0:
        return 0.0
    per = 4 * ns_steps - 3          # m^3 products over the whole iteration
    return float(sum(3.0 * min(s) ** 2 * max(s) + per * float(min(s)) ** 3 for s in shapes))


# ---------------------------------------------------------------- CPU oracle
def oracle_sample(workload_name: str, ns_steps: int = 5, warm: bool = False):
    """Time the fp64 oracle on a bounded sample of the workload and extrapolate
    to one full Muon step (`ns_steps` NS steps, every matrix).

    The sample is one matrix of every distinct shape of the set -- the large
    MLP shapes that carry most of the flops included -- each run through
    momentum, one Newton-Schulz step and the update.  Each shape's own
    measured NS time scales by its multiplicity and `ns_steps` (one NS step of
    a shape costs the same every step); momentum and update scale by elements.
    `warm` runs only the cheapest shape (warm-up of the BLAS threads).
    Returns (ms_per_full_step, description, seconds_spent)."""
    import numpy as np
    import oracle
    from newton_schulz_owner_gb300 import workloads as wl

    def nominal(s):   # dense fp64 flops of one NS step: 4 m^2 n + 2 m^3
        m, n = min(s), max(s)
        return 4.0 * m * m * n + 2.0 * m ** 3

    w = wl.WORKLOADS[workload_name]
    shapes = w.shapes()
    distinct = sorted(set(shapes), key=nominal)
    if warm:
        distinct = distinct[:1]
    rng = np.random.default_rng(0)
    t_ew = e_ew = 0.0
    t_ns = {}
    t_all = time.perf_counter()
    for s in distinct:
        G = rng.standard_normal(s) * 1e-3
        M = np.zeros(s)
        W = rng.standard_normal(s) * 0.02
        t0 = time.perf_counter()
        M1, U = oracle.nesterov_momentum(G, M, 0.95)
        t1 = time.perf_counter()
        O = oracle.newton_schulz(U, 1)
        t2 = time.perf_counter()
        oracle.apply_update(W, O, 0.02)
        t3 = time.perf_counter()
        t_ew += (t1 - t0) + (t3 - t2)
        e_ew += s[0] * s[1]
        t_ns[s] = t2 - t1
    spent = time.perf_counter() - t_all
    if warm:
        return None, "warm-up", spent
    total_s = sum(t_ns[s] * ns_steps for s in shapes) + \
        sum(r * c for r, c in shapes) * (t_ew / e_ew)
    desc = (f"fp64 oracle, one matrix of each of the {len(distinct)} distinct shapes of "
            f"{workload_name} ({', '.join(f'{r}x{c}' for r, c in distinct)}), one NS step "
            f"each, timed directly; extrapolated to all {len(shapes)} matrices x {ns_steps} NS "
            f"steps by each shape's own time (NS) and by elements (momentum, update)")
    return total_s * 1e3, desc, spent


def trace_summary(rec, step_ms: float):
    """Where the CTA pairs of the product kernel spend one traced step.

    `rec` holds one record per CTA of every product launch of the step
    (dmuon_trace_begin).  Pair time over the product window (first product
    entry to last product exit) splits into MMA-active (a pair's first MMA
    issue to its last MMA completion, per launch), fill/drain (resident but
    before its first or after its last MMA) and not resident (launch gaps,
    last-wave tails, pairs without a tile).  A whole-step persistent kernel
    could recover at most the last two."""
    lead = rec["cta"] % 2 == 0
    entry, exit_ = rec["t_entry"], rec["t_exit"]
    t0, t1 = int(entry.min()), int(exit_.max())
    window = (t1 - t0) * 1e-6
    pairs = int(rec["cta"].max().item()) // 2 + 1   # pairs of the widest launch
    has = lead & (rec["t_mma_first"] > 0)
    busy = float((rec["t_mma_last"][has] - rec["t_mma_first"][has]).sum().item()) * 1e-6
    resident = float((exit_[lead] - entry[lead]).sum().item()) * 1e-6
    total = pairs * window
    launches = sorted(set(rec["launch"].tolist()))
    spans = []
    for L in launches:
        m = rec["launch"] == L
        spans.append((int(entry[m].min()), int(exit_[m].max())))
    gaps = sum(max(0, spans[k + 1][0] - spans[k][1]) for k in range(len(spans) - 1)) * 1e-6
    # the leaders' MMA threads: share of their MMA span spent waiting, per product kind
    waits = {}
    if "mma_span_cycles" in rec:
        names = {0: "sym_k", 1: "sym_mn", 2: "full_wide", 3: "full_tall"}
        for kd, nm in names.items():
            sel = has & (rec["kind"] == kd)
            span = float(rec["mma_span_cycles"][sel].sum().item())
            if span > 0:
                waits[nm] = {"operand": float(rec["wait_operand_cycles"][sel].sum().item()) / span,
                             "accumulator": float(rec["wait_accum_cycles"][sel].sum().item()) / span}
    return {"launches": len(launches), "pairs": pairs, "step_ms": step_ms,
            "mma_thread_wait_frac": waits,
            "product_window_ms": window,
            "mma_active_frac": busy / total, "fill_drain_frac": (resident - busy) / total,
            "not_resident_frac": (total - resident) / total,
            "launch_gaps_ms": gaps,
            "recoverable_ms_upper_bound": (total - busy) / pairs,
            "note": "pair time over the product window of one traced dmuon_muon_step: MMA-active "
                    "(first MMA issue to last MMA completion of each pair and launch), fill/drain "
                    "(resident, outside that span), not resident (launch gaps, last-wave tails, "
                    "pairs without a tile); a whole-step persistent kernel could recover at most "
                    "the time outside MMA-active"}


def e2e_group_bounds(layers: int, groups: int, taper: bool):
    """Layer ranges of the end-to-end loop's groups.  Only the first group's copy
    in and the last group's copy out are not hidden behind another group's
    compute, so with `taper` the groups grow towards the middle (weights
    1, 2, 4, ..., 4, 2, 1) and those two stay small; otherwise equal groups."""
    groups = max(1, min(groups, layers))
    if taper and groups >= 3:
        half = [2 ** min(k, 2) for k in range((groups + 1) // 2)]
        wts = half + half[:groups // 2][::-1]
    else:
        wts = [1] * groups
    tot = float(sum(wts))
    cuts, acc = [0], 0.0
    for wgt in wts[:-1]:
        acc += wgt
        cuts.append(max(cuts[-1] + 1, min(layers - (len(wts) - len(cuts)), round(layers * acc / tot))))
    cuts.append(layers)
    return [(cuts[k], cuts[k + 1]) for k in range(len(wts)) if cuts[k] < cuts[k + 1]]


def owner_times(dmuon, shapes, owner, variant, ns_steps, stream, barrier, grouped_ns_ms):
    """Each LPT owner's Newton-Schulz as its own call on its segments of the
    packed buffer, back to back, against all owners in one grouped call: the
    single-GPU picture of the pages' balanced ownership (the slowest owner
    bounds a distributed step)."""
    import torch
    n = len(shapes)
    n_owners = max(owner.owner_of) + 1
    groups = [[i for i in range(n) if owner.owner_of[i] == k] for k in range(n_owners)]
    groups = [gk for gk in groups if gk]
    ws_max = max(dmuon.workspace_bytes([shapes[i] for i in gk], variant) for gk in groups)
    ws_o = torch.zeros(ws_max, dtype=torch.uint8, device=owner.packed.device)

    def owner_ns(gk):
        dmuon.ns_batched([shapes[i] for i in gk], owner.packed, [owner.offsets[i] for i in gk],
                         ws_o, ns_steps=ns_steps, variant=variant, stream=stream)

    for gk in groups:
        owner_ns(gk)
    barrier()
    oev = [torch.cuda.Event(enable_timing=True) for _ in range(len(groups) + 1)]
    with torch.cuda.stream(stream):
        oev[0].record(stream)
        for k, gk in enumerate(groups):
            owner_ns(gk)
            oev[k + 1].record(stream)
    barrier()
    st = dmuon.stream_status(ws_o, stream)
    if st != dmuon.OK:
        raise RuntimeError(f"per-owner NS failed: {dmuon.status_string(st)}")
    o_ms = [oev[k].elapsed_time(oev[k + 1]) for k in range(len(groups))]
    o_elems = [sum(shapes[i][0] * shapes[i][1] for i in gk) for gk in groups]
    return {"n_owners": len(groups), "ns_ms": o_ms, "elements": o_elems,
            "back_to_back_ms": sum(o_ms), "grouped_ns_ms": grouped_ns_ms,
            "max_over_mean": max(o_ms) / (sum(o_ms) / len(o_ms)),
            "note": "each owner's Newton-Schulz alone (norms from the packed values), "
                    "back to back, vs all owners in one grouped call"}


# The benchmark's other projection-set configurations, measured after the main
# workload when it runs at its default: (workload, variant, ns_steps).
OTHER_CONFIGS = [("single-256x1024", 0, 5), ("qwen2.5-1.5b", 0, 5), ("llama-3.2-3b", 0, 5),
                 ("qwen2.5-7b", 0, 3), ("qwen2.5-7b", 1, 3), ("qwen2.5-7b", 0, 5),
                 ("qwen2.5-7b", 1, 5), ("qwen2.5-7b", 0, 8), ("qwen2.5-7b", 1, 8)]


def config_point(dmuon, wl, name, variant, ns_steps, dev, gpu_index, peak, steps=3, warmup=3,
                 min_region_s=0.5, max_steps=2000):
    """One configuration, measured like the main workload but shorter: the whole
    step through dmuon_muon_step (median of the timed steps), then the same step
    as three calls with events between them for the Newton-Schulz phase;
    per-owner times where the set has an owner partition.  Short steps are
    repeated (up to `max_steps`) until each of the two timed regions lasts
    about `min_region_s`, and the clocks are summarised from the samples taken
    inside them only."""
    import torch
    w = wl.WORKLOADS[name]
    shapes = w.shapes()
    owner = dmuon.MuonOwner(shapes, n_owners=w.n_owners, variant=variant, device=dev)
    G = wl.alloc_flat(shapes, w.grad_dtype, dev)
    M = wl.alloc_flat(shapes, torch.float32, dev)
    W = wl.alloc_flat(shapes, w.weight_dtype, dev)
    wl.fill_grads(w, G, step=0)
    wl.fill_weights(w, W)
    stream = torch.cuda.Stream(device=dev)
    gs = [s for s in shapes if dmuon.ns_variant_for(s, ns_steps, variant) == 1]
    ss = [s for s in shapes if dmuon.ns_variant_for(s, ns_steps, variant) != 1]
    flops = gram_flops(gs, ns_steps) + ns_flops(ss, ns_steps)

    def barrier():
        torch.cuda.synchronize(dev)

    def step():
        owner.step(G.views, M.views, W.views, lr=0.02, beta=0.95, ns_steps=ns_steps,
                   stream=stream)

    for _ in range(warmup):
        step()
    barrier()
    t_one = time.perf_counter()
    step()
    barrier()
    t_one = time.perf_counter() - t_one
    steps = max(steps, min(max_steps, int(math.ceil(min_region_s / max(t_one, 1e-6)))))
    sampler = ClockSampler(gpu_index)
    sampler.start()
    time.sleep(0.3)
    t_region0 = time.monotonic()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for k in range(steps):
        step()
        ev[k + 1].record(stream)
    barrier()
    ph = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    with torch.cuda.stream(stream):
        for k in range(steps):
            ph[k][0].record(stream)
            dmuon.pack(shapes, G.views, M.views, 0.95, owner.packed, owner.offsets,
                       owner.workspace, stream=stream)
            ph[k][1].record(stream)
            dmuon.ns_batched(shapes, owner.packed, owner.offsets, owner.workspace,
                             ns_steps=ns_steps, variant=variant, use_pack_norms=True,
                             stream=stream)
            ph[k][2].record(stream)
            dmuon.unpack_update(shapes, W.views, 0.02, owner.packed, owner.offsets,
                                owner.workspace, stream=stream)
            ph[k][3].record(stream)
    barrier()
    clocks = sampler.stop(window=(t_region0, time.monotonic()))
    st = dmuon.stream_status(owner.workspace, stream)
    if st != dmuon.OK:
        raise RuntimeError(f"{name}: {dmuon.status_string(st)}")
    step_ms = statistics.median(ev[k].elapsed_time(ev[k + 1]) for k in range(steps))
    ns_ms = statistics.median(p[1].elapsed_time(p[2]) for p in ph)
    out = {"workload": name, "variant": {0: "standard", 1: "gram", 2: "gram-all"}[variant],
           "ns_steps": ns_steps, "matrices": len(shapes),
           "gram_matrices": len(gs), "step_ms": step_ms, "ns_ms": ns_ms,
           "pack_ms": statistics.median(p[0].elapsed_time(p[1]) for p in ph),
           "update_ms": statistics.median(p[2].elapsed_time(p[3]) for p in ph),
           "ns_tflops_algorithmic": flops / (ns_ms * 1e-3) / 1e12,
           "ns_tflops_nominal_dense": None if gs else
           nominal_flops(shapes, ns_steps) / (ns_ms * 1e-3) / 1e12,
           "ns_frac_of_peak": flops / (ns_ms * 1e-3) / 1e12 / peak,
           "matrices_per_s": len(shapes) / (step_ms * 1e-3), "steps": steps, "warmup": warmup,
           "clocks": clocks}
    if w.n_owners > 1:
        out["owners"] = owner_times(dmuon, shapes, owner, variant, ns_steps, stream, barrier,
                                    ns_ms)
    del owner, G, M, W
    torch.cuda.empty_cache()
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    cores = os.cpu_count()
    for _ in range(args.warmup):
        oracle_sample(args.workload, args.ns_steps, warm=True)
    vals, spent = [], []
    for _ in range(args.steps):
        ms, desc, sec = oracle_sample(args.workload, args.ns_steps)
        vals.append(ms)
        spent.append(sec)
    v = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "ms",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": v,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": args.workload, "ns_steps": args.ns_steps,
                                        "variant": "standard"},
        "extrapolated": True,
        "note": "each timed step is a bounded sample (one matrix of every distinct shape, one "
                "NS step); value is that sample extrapolated to one whole Muon step, not a "
                "timed whole step",
        "cpu_baseline": {"value": v, "unit": "ms", "cores": cores, "kind": "oracle",
                         "sample": desc, "blas": blas_name(), "extrapolated": True,
                         "sample_seconds": statistics.median(spent)},
        "e2e": {"value": v, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm
def max_over_ranks(value: float, dist=None, device="cpu") -> float:
    """Largest value over all ranks (the job's time is its slowest rank's)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def owned_matrices(shapes, rank: int, world: int):
    """Indices of the matrices rank `rank` owns when `world` ranks split the set
    with the library's owner plan (each matrix has exactly one owner)."""
    from newton_schulz_owner_gb300 import dmuon
    owner_of, _, _ = dmuon.plan(shapes, world)
    return [i for i, o in enumerate(owner_of) if o == rank]


def run_gpu(args, rank, world, local_rank):
    import numpy as np
    import torch

    from newton_schulz_owner_gb300 import build_lib
    if not os.path.exists(build_lib.LIB):
        build_lib.build()
    from newton_schulz_owner_gb300 import dmuon
    from newton_schulz_owner_gb300 import workloads as wl

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)

    w = wl.WORKLOADS[args.workload]
    shapes = w.shapes()
    n = len(shapes)
    owner = dmuon.MuonOwner(shapes, n_owners=w.n_owners, variant=args.variant, device=dev)
    packed_elems = owner.packed.numel()
    G = wl.alloc_flat(shapes, w.grad_dtype, dev)
    M = wl.alloc_flat(shapes, torch.float32, dev)
    W = wl.alloc_flat(shapes, w.weight_dtype, dev)
    wl.fill_grads(w, G, step=0)
    wl.fill_weights(w, W)
    stream = torch.cuda.Stream(device=dev)
    # Gram where the library's rule admits it; the standard form on the rest
    gs = [s for s in shapes if dmuon.ns_variant_for(s, args.ns_steps, args.variant) == 1]
    ss = [s for s in shapes if dmuon.ns_variant_for(s, args.ns_steps, args.variant) != 1]
    flops = gram_flops(gs, args.ns_steps) + ns_flops(ss, args.ns_steps)
    # nominal dense count (standard form only): both symmetric products counted in full
    flops_nominal = nominal_flops(shapes, args.ns_steps) if not gs else None
    elems = sum(r * c for r, c in shapes)

    def step_phases(ev=None):
        with torch.cuda.stream(stream):
            if ev is not None:
                ev[0].record(stream)
            dmuon.pack(shapes, G.views, M.views, 0.95, owner.packed, owner.offsets,
                       owner.workspace, stream=stream)
            if ev is not None:
                ev[1].record(stream)
            dmuon.ns_batched(shapes, owner.packed, owner.offsets, owner.workspace,
                             ns_steps=args.ns_steps, variant=args.variant,
                             use_pack_norms=True, stream=stream)
            if ev is not None:
                ev[2].record(stream)
            dmuon.unpack_update(shapes, W.views, 0.02, owner.packed, owner.offsets,
                                owner.workspace, stream=stream)
            if ev is not None:
                ev[3].record(stream)

    def barrier():
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    def whole_step():
        owner.step(G.views, M.views, W.views, lr=0.02, beta=0.95, ns_steps=args.ns_steps,
                   stream=stream)

    for _ in range(args.warmup):
        whole_step()
        step_phases()
    barrier()
    st = dmuon.stream_status(owner.workspace, stream)
    if st != dmuon.OK:
        raise RuntimeError(f"warm-up failed: {dmuon.status_string(st)}")

    sampler = ClockSampler(local_rank if world > 1 else int(os.environ.get("GPU_INDEX", "0")))
    sampler.start()
    time.sleep(0.3)
    # timed region 1 -- `value`: the product call, dmuon_muon_step, once per step
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    barrier()
    t_region0 = time.monotonic()
    dmuon.launch_count(reset=True)
    torch.cuda.nvtx.range_push("whole_step")   # for profiler selection (ncu --nvtx-include)
    step_ev[0].record(stream)
    for k in range(args.steps):
        whole_step()
        step_ev[k + 1].record(stream)
    torch.cuda.nvtx.range_pop()
    timed_launches = dmuon.launch_count(reset=True)   # the library's own count
    barrier()
    # timed region 2 -- the same step as its three calls (pack, Newton-Schulz,
    # update) with events between them: the per-phase times and the roofline
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    barrier()
    torch.cuda.nvtx.range_push("three_call")
    for k in range(args.steps):
        step_phases(evs[k])
    torch.cuda.nvtx.range_pop()
    barrier()
    clocks = sampler.stop(window=(t_region0, time.monotonic()))
    st = dmuon.stream_status(owner.workspace, stream)
    if st != dmuon.OK:
        raise RuntimeError(f"timed steps failed: {dmuon.status_string(st)}")
    step_ms = [step_ev[k].elapsed_time(step_ev[k + 1]) for k in range(args.steps)]
    pack_ms = [e[0].elapsed_time(e[1]) for e in evs]
    ns_ms = [e[1].elapsed_time(e[2]) for e in evs]
    upd_ms = [e[2].elapsed_time(e[3]) for e in evs]
    t_total = max_over_ranks(sum(step_ms), dist, dev)
    ms = t_total / args.steps
    ns_mean = sum(ns_ms) / len(ns_ms)
    achieved_tflops = flops / (ns_mean * 1e-3) / 1e12

    # ---- one more dmuon_muon_step, outside the timed regions, with the
    # product launches traced (per-CTA timestamps): what a whole-step
    # persistent kernel could recover at most
    ns_trace = None
    if not args.no_trace:
        tbuf = torch.zeros(4 << 20, dtype=torch.uint8, device=dev)
        ns_trace, raw = {}, {}
        # the whole step (the value's call), then its Newton-Schulz phase alone
        for label, fn in (("whole_step", whole_step),
                          ("ns_phase_alone", lambda: dmuon.ns_batched(
                              shapes, owner.packed, owner.offsets, owner.workspace,
                              ns_steps=args.ns_steps, variant=args.variant, stream=stream))):
            te = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            barrier()
            dmuon.trace_begin(tbuf)
            te[0].record(stream)
            fn()
            te[1].record(stream)
            barrier()
            rec = dmuon.trace_end(tbuf)
            st = dmuon.stream_status(owner.workspace, stream)
            if st != dmuon.OK:
                raise RuntimeError(f"traced step failed: {dmuon.status_string(st)}")
            if rec["cta"].numel():
                ns_trace[label] = trace_summary(rec, te[0].elapsed_time(te[1]))
                raw[label] = {k: v.numpy() for k, v in rec.items()}
        if args.trace_out:
            import numpy as np
            np.savez(args.trace_out, **{f"{lab}.{k}": v for lab, d in raw.items()
                                        for k, v in d.items()})
        del tbuf

    # ---- owners (workloads with an LPT owner partition): each owner's
    # Newton-Schulz as its own call on its segments of the packed buffer, back
    # to back, against the grouped call above -- the single-GPU picture of the
    # pages' balanced ownership (the slowest owner bounds a distributed step).
    owners = None
    if w.n_owners > 1:
        owners = owner_times(dmuon, shapes, owner, args.variant, args.ns_steps, stream, barrier,
                             ns_mean)

    # ---- AdamW for the parameters outside the Muon set (embedding, head, norms),
    # timed on its own: bf16 parameters and gradients, fp32 moments.
    adamw = None
    ashapes = w.adamw_shapes()
    if ashapes and not args.no_adamw:
        ap_ = wl.alloc_flat(ashapes, torch.bfloat16, dev)
        ag_ = wl.alloc_flat(ashapes, torch.bfloat16, dev)
        am_ = wl.alloc_flat(ashapes, torch.float32, dev)
        av_ = wl.alloc_flat(ashapes, torch.float32, dev)
        ap_.flat.normal_(0.0, 0.02)
        ag_.flat.normal_(0.0, 1e-3)
        aws = torch.zeros(dmuon.adamw_workspace_bytes(len(ashapes)), dtype=torch.uint8, device=dev)
        for t in range(1, args.warmup + 1):
            dmuon.adamw(ap_.views, ag_.views, am_.views, av_.views, t, aws, stream=stream)
        barrier()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for t in range(args.warmup + 1, args.warmup + 1 + args.steps):
            dmuon.adamw(ap_.views, ag_.views, am_.views, av_.views, t, aws, stream=stream)
        a1.record(stream)
        barrier()
        st = dmuon.stream_status(aws, stream)
        if st != dmuon.OK:
            raise RuntimeError(f"adamw failed: {dmuon.status_string(st)}")
        a_ms = a0.elapsed_time(a1) / args.steps
        a_elems = sum(r * c for r, c in ashapes)
        a_bytes = a_elems * 22   # p r/w 2+2, g 2, m r/w 4+4, v r/w 4+4
        adamw = {"ms": a_ms, "elements": a_elems, "bytes_per_elem": 22,
                 "gbs": a_bytes / (a_ms * 1e-3) / 1e9, "tensors": len(ashapes)}
        del ap_, ag_, am_, av_, aws

    # ---- end to end through dmuon_muon_step with host buffers.  Every step copies
    # its gradients in from pinned host memory and its updated weights back out.
    # The copies are pipelined with the compute the way a training loop would,
    # per group of consecutive layers (one owner and one dmuon_muon_step call
    # per group): a group's gradients are copied in while the previous group
    # computes, its updated weights are snapshotted on the device and copied
    # out while the next group computes, and the next step's copies in use a
    # second device buffer.  Only the first group's copy in and the last
    # group's copy out are not hidden.  All copies sit inside the timed region.
    e2e = None
    if not args.no_e2e:
        G_host = wl.alloc_flat(shapes, w.grad_dtype, "cpu", pin=True, zero=False)
        W_host = wl.alloc_flat(shapes, w.weight_dtype, "cpu", pin=True, zero=False)
        G_host.flat.copy_(G.flat)
        h2d = G.flat.numel() * G.flat.element_size()
        d2h = W.flat.numel() * W.flat.element_size()
        G_dev = [G, wl.alloc_flat(shapes, w.grad_dtype, dev, zero=False)]
        W_snap = [wl.alloc_flat(shapes, w.weight_dtype, dev, zero=False) for _ in range(2)]
        h2d_stream = torch.cuda.Stream(device=dev)
        d2h_stream = torch.cuda.Stream(device=dev)
        # groups of whole layers, each a contiguous range of every flat buffer
        per_layer = max(1, n // max(1, w.layers))
        gsets = [(a * per_layer, min(n, b * per_layer))
                 for a, b in e2e_group_bounds(n // per_layer, args.e2e_groups, args.e2e_taper)]
        gsets[-1] = (gsets[-1][0], n)
        owner = None   # the groups' owners take its place
        torch.cuda.empty_cache()
        g_owner = [dmuon.MuonOwner(shapes[i0:i1], n_owners=w.n_owners, variant=args.variant,
                                   device=dev) for i0, i1 in gsets]

        def span(fs, i0, i1):
            o1 = fs.offsets[i1] if i1 < n else fs.flat.numel()
            return fs.flat[fs.offsets[i0]:o1]

        def e2e_steps(nsteps, spans=None):
            # spans: per step (h2d start, h2d end, step start, step end, d2h start, d2h end)
            done = [[None] * len(gsets) for _ in range(2)]   # last step that read G_dev[b], group j
            out = [[None] * len(gsets) for _ in range(2)]    # last copy out of W_snap[b], group j
            last = None
            ev = lambda: torch.cuda.Event(enable_timing=spans is not None)
            for k in range(nsteps):
                b = k % 2
                sp = [ev() for _ in range(6)]
                for j, (i0, i1) in enumerate(gsets):
                    with torch.cuda.stream(h2d_stream):
                        if done[b][j] is not None:
                            h2d_stream.wait_event(done[b][j])
                        if j == 0:
                            sp[0].record(h2d_stream)
                        span(G_dev[b], i0, i1).copy_(span(G_host, i0, i1), non_blocking=True)
                        g_in = ev()
                        g_in.record(h2d_stream)
                    stream.wait_event(g_in)
                    if j == 0:
                        sp[2].record(stream)
                    g_owner[j].step(G_dev[b].views[i0:i1], M.views[i0:i1], W.views[i0:i1],
                                    lr=0.02, beta=0.95, ns_steps=args.ns_steps, stream=stream)
                    d = ev()
                    d.record(stream)
                    done[b][j] = d
                    with torch.cuda.stream(stream):
                        if out[b][j] is not None:
                            stream.wait_event(out[b][j])
                        span(W_snap[b], i0, i1).copy_(span(W, i0, i1), non_blocking=True)
                        snap = torch.cuda.Event()
                        snap.record(stream)
                    with torch.cuda.stream(d2h_stream):
                        d2h_stream.wait_event(snap)
                        if j == 0:
                            sp[4].record(d2h_stream)
                        span(W_host, i0, i1).copy_(span(W_snap[b], i0, i1), non_blocking=True)
                        o = ev()
                        o.record(d2h_stream)
                        out[b][j] = o
                    last = o
                sp[1] = g_in
                sp[3] = d
                sp[5] = last
                if spans is not None:
                    spans.append(sp)
            return last

        e2e_steps(max(2, min(args.warmup, 3)))
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(h2d_stream)
        stream.wait_event(e0)
        spans = []
        last = e2e_steps(args.steps, spans)
        stream.wait_event(last)
        e1.record(stream)
        barrier()
        for go in g_owner:
            st = dmuon.stream_status(go.workspace, stream)
            if st != dmuon.OK:
                raise RuntimeError(f"e2e steps failed: {dmuon.status_string(st)}")
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dist, dev)
        mean = lambda i, j: sum(sp[i].elapsed_time(sp[j]) for sp in spans) / len(spans)
        h2d_ms, step_ms_e2e, d2h_ms = mean(0, 1), mean(2, 3), mean(4, 5)
        e2e = {"value": e2e_ms, "unit": "ms", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h),
               "groups": len(gsets),
               "note": f"{len(gsets)} groups of consecutive layers, one dmuon_muon_step call "
                       "each; a group's copies in and out overlap the other groups' compute; "
                       "only the first group's copy in and the last group's copy out are not "
                       "hidden; h2d/d2h/step times span the groups of one step",
               "h2d_ms": h2d_ms, "h2d_gbs": h2d / (h2d_ms * 1e-3) / 1e9,
               "d2h_ms": d2h_ms, "d2h_gbs": d2h / (d2h_ms * 1e-3) / 1e9,
               "step_ms": step_ms_e2e}
        del G_host, W_host, G_dev, W_snap, g_owner


    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    tr = traffic_record()
    if tr is not None and (tr.get("workload") != args.workload or tr.get("ns_steps") != args.ns_steps
                           or args.variant != 0):
        tr = None   # the ncu figure covers one workload and configuration only
    # one roofline unit = one Newton-Schulz phase: all product launches of one step
    roofline = {"bound": "tensor", "kernel": "ns_gemm_kernel (all Newton-Schulz products)",
                "unit_of_work": "one Newton-Schulz phase (all product launches of one step)",
                "achieved": achieved_tflops, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved_tflops / peak, "peak_source": f"{peak_src} bf16 sustained",
                "traffic": None if tr is None else tr.get("dram_bytes_per_ns_phase"),
                # per matrix and iteration: X read twice and X' written (6mn bytes),
                # A and B each written once and read once (8m^2 bytes), bf16
                "algorithmic_bytes": None if args.variant != 0 else float(args.ns_steps * sum(
                    6 * min(r, c) * max(r, c) + 8 * min(r, c) ** 2 for r, c in shapes)),
                "flops_per_step": flops}
    elem_bytes = {"pack": (2 if w.grad_dtype == torch.bfloat16 else 4) + 4 + 4 + 2,
                  "update": 2 + 2 * (2 if w.weight_dtype == torch.bfloat16 else 4)}
    pack_mean = sum(pack_ms) / len(pack_ms)
    upd_mean = sum(upd_ms) / len(upd_ms)
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    phases = {
        "note": "three-call decomposition (pack, ns_batched, unpack_update) timed in a second "
                "region, each phase alone; dmuon_muon_step (the value) overlaps the "
                "memory-bound phases with the products on a second stream",
        "pack_ms": pack_mean, "ns_ms": ns_mean, "update_ms": upd_mean,
        "three_call_step_ms": sum(e[0].elapsed_time(e[3]) for e in evs) / len(evs),
        "pack_gbs": elems * elem_bytes["pack"] / (pack_mean * 1e-3) / 1e9,
        "update_gbs": elems * elem_bytes["update"] / (upd_mean * 1e-3) / 1e9,
        "hbm_peak_gbs": hbm_peak,
    }
    resident = (G.flat.numel() * G.flat.element_size() + M.flat.numel() * 4 +
                W.flat.numel() * W.flat.element_size() + packed_elems * 2)
    line = {
        "metric": METRIC, "value": ms, "unit": "ms", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False,
        "step_ms_median": statistics.median(step_ms), "step_ms_min": min(step_ms),
        "step_ms_max": max(step_ms),
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded normal gradients/weights shaped like the model's projections)",
        "config": {"workload": args.workload, "matrices": n, "elements": elems,
                   "ns_steps": args.ns_steps,
                   "variant": {0: "standard", 1: "gram", 2: "gram-all"}[args.variant],
                   "grad_dtype": str(w.grad_dtype).replace("torch.", ""),
                   "weight_dtype": str(w.weight_dtype).replace("torch.", ""),
                   "momentum_dtype": "float32", "parallelism": f"replicas x{world}",
                   "l2": f"no flush: resident inputs {resident / 1e9:.1f} GB >> L2 "
                         f"{L2_BYTES / 2**20:.0f} MB"},
        "ns_tflops": achieved_tflops,
        "ns_tflops_nominal_dense": None if flops_nominal is None else
        flops_nominal / (ns_mean * 1e-3) / 1e12,
        "matrices_per_s": n * world / (ms * 1e-3),
        "phases": phases,
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": timed_launches,
        "adamw": adamw,
        "owners": owners,
        "ns_trace": ns_trace,
        "clocks": clocks,
    }
    # ---- the benchmark's other configurations (one GPU, default workload only),
    # each measured on its own after the main workload's buffers are freed
    if world == 1 and args.workload == DEFAULT_WORKLOAD and not args.no_other_configs:
        owner = G = M = W = None
        torch.cuda.empty_cache()
        gpu_index = int(os.environ.get("GPU_INDEX", "0"))
        line["other_configs"] = [config_point(dmuon, wl, name, variant, k, dev, gpu_index, peak)
                                 for name, variant, k in OTHER_CONFIGS]
    if rank == 0 and not args.no_cpu_baseline:
        cms, desc, sec = oracle_sample(args.workload, args.ns_steps)
        line["cpu_baseline"] = {"value": cms, "unit": "ms", "cores": os.cpu_count(),
                                "kind": "oracle", "sample": desc, "blas": blas_name(),
                                "extrapolated": True, "sample_seconds": sec}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--ns-steps", type=int, default=5)
    ap.add_argument("--variant", type=int, default=0,
                    help="0 standard, 1 Gram where the library's rule admits it, "
                         "2 Gram on every matrix with n > m")
    ap.add_argument("--impl", default="dmuon", choices=["dmuon", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-groups", type=int, default=4,
                    help="layer groups of the end-to-end loop (one dmuon_muon_step call each)")
    ap.add_argument("--e2e-taper", type=int, default=0,
                    help="1: end-to-end groups grow towards the middle (small first and last "
                         "groups, whose copies are not hidden)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-launch-count", action="store_true",
                    help="accepted for older command lines; the launch count now comes "
                         "from the library and costs nothing")
    ap.add_argument("--no-trace", action="store_true",
                    help="skip the traced step (per-CTA timestamps of the product launches)")
    ap.add_argument("--trace-out", default="",
                    help="also save the traced records (numpy .npz) to this file")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip the measurements of the other projection-set configurations "
                         "that follow the default workload's")
    ap.add_argument("--no-adamw", action="store_true",
                    help="skip the AdamW measurement of the non-Muon parameters")
    args = ap.parse_args()
    rank, world, local_rank = _rank_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_gpu(args, rank, world, local_rank)


if __name__ == "__main__":
    sys.exit(main())
