#!/usr/bin/env python3
"""Throughput of batched draft-token verification on one GB300.

One step = one pass of the whole verification path over one batch:
  1. spec_verify_sample      B=64 sequences, k=4 drafts, V=128256, bf16, T=1.0
  2. spec_verify_greedy      same logits shape, 70% of drafts forced to argmax
  3. spec_verify_tree_greedy 16 trees of 60 nodes, depth <= 6, V=128256, bf16
The three calls verify independent batches: a step forks them onto three
streams (one workspace each) and joins them before the next step begins
(`serial_ms_per_step` times the same steps with the calls one after another).
Metric: verified draft positions per second (B*k + B*k + B*(N-1) = 1456 per
step) and the achieved HBM bandwidth on the logits the method must read.

Inputs are generated once on the host (seeded) and copied to 4 device sets used
in rotation; every tree call reads 246 MB (> the 129 MB L2) between two uses of
any set, so every read comes from HBM.  `value` is timed with CUDA events on the
launching stream with inputs resident in HBM, the steps replayed from CUDA graphs
(so that Python does not pace the launches); `e2e` repeats the step through the
same public API with inputs copied from pinned host memory and results copied
back inside the timed region.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun each rank verifies its own batches (sequences are independent:
no collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("verified draft positions/sec and achieved HBM GB/s (% of GB300 peak) "
          "at B=64,k=4,V=128k")
UNIT = "positions/s"
NSETS = 4
FALLBACK_HBM_GBS = 6800.0
# the files holding the verification kernels (the recorded traffic is valid
# while they are unchanged)
KERNEL_SOURCES = ["speculative_decoding_verification_56_gb300/csrc/sv_device.cuh",
                  "speculative_decoding_verification_56_gb300/csrc/sv_kernels.cuh"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="budget of the oracle CPU baseline (0 disables it)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--profile-case", choices=["lm_head_greedy", "tree_grow", "sample", "step"],
                    default=None,
                    help="only run that kernel --calls times, untimed (for ncu)")
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--skip-next-rows", action="store_true",
                    help="leave out the kernels around the draft tree (next_rows)")
    ap.add_argument("--skip-large", action="store_true",
                    help="leave out the large-batch measurement (at_scale)")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def replica_seed(seed, rank):
    """Each rank verifies its own batches (sequences are independent): the
    workload of rank r is drawn from seed + 1000 r."""
    return seed + 1000 * rank


def max_over_ranks(x, device):
    """The largest of every rank's x (the step time of the slowest rank); x
    itself on one rank.  `device` holds the reduction tensor: a CUDA device
    under NCCL, the CPU under gloo."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, steps, units_per_step, total_ms):
    """Whole-job units/s: every rank ran `steps` steps of `units_per_step`
    units; the job takes the slowest rank's `total_ms`."""
    return world * steps * units_per_step / (total_ms / 1e3)


def workload(seed):
    from speculative_decoding_verification_56_gb300 import synth
    samp = synth.zipf128k(seed=seed)
    greedy = synth.greedy_variant(samp, 0.7)
    tree = synth.tree(seed=seed)
    return samp, greedy, tree


def positions(samp, greedy, tree):
    return samp.B * samp.k + greedy.B * greedy.k + tree.B * (tree.N - 1)


def kernel_source_hash():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_tflops():
    """Dense bf16 tensor peak for a kernel timed in short bursts."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops)"
    except Exception:
        return 1900.0, "fallback 1.9 PFLOP/s"


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(kernel):
    """Per-launch DRAM bytes of ``kernel`` from the committed ncu summary, or
    None when the summary is missing or the kernel sources changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    cur = kernel_source_hash()
    for line in open(path):
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel \
                and parts[1] == cur:
            return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) taken while timing."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, t0, t1):
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts + frac, float(parts[1]), float(parts[2]), parts[5:9]))
            except Exception:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        use = inside if inside else rows
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in use:
            for n, v in zip(names, r[3]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in use),
                "sm_max_mhz": max(r[2] for r in use),
                "reasons": sorted(reasons), "samples": len(use),
                "samples_in_timed_region": len(inside)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args, rank, world, local_rank):
    import torch
    import speculative_decoding_verification_56_gb300 as sv
    from speculative_decoding_verification_56_gb300 import build

    build.build_library()
    lib = sv.load_library()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    samp, greedy, tree = workload(replica_seed(args.seed, rank))
    pos_step = positions(samp, greedy, tree)
    seqs_step = samp.B + greedy.B + tree.B  # sequences and trees verified per step
    eb = samp.elem_bytes
    B, k, V = samp.B, samp.k, samp.V
    Bt, N, Vt = tree.B, tree.N, tree.V

    # pinned host copies (e2e) and NSETS device sets (rotation)
    def pinned(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return t.pin_memory()

    h = dict(t=pinned(samp.target.view(np.int16)), d=pinned(samp.draft.view(np.int16)),
             tok=pinned(samp.tokens), ua=pinned(samp.u_accept), us=pinned(samp.u_sample),
             gtok=pinned(greedy.tokens), tt=pinned(tree.target.view(np.int16)),
             ttok=pinned(tree.tokens), tpar=pinned(tree.parents))
    sets = []
    for _ in range(NSETS):
        sets.append({key: val.to(dev, non_blocking=False) for key, val in h.items()})
    i32 = dict(dtype=torch.int32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    outs = dict(n=torch.empty(B, **i32), tok=torch.empty(B, k + 1, **i32),
                p=torch.empty(B, k, **f32), q=torch.empty(B, k, **f32), R=torch.empty(B, **f32),
                gn=torch.empty(B, **i32), gtok=torch.empty(B, k + 1, **i32),
                tn=torch.empty(Bt, **i32), tpath=torch.empty(Bt, tree.max_depth + 1, **i32),
                ttok=torch.empty(Bt, tree.max_depth + 1, **i32))
    # one workspace per call type: the three calls of a step run concurrently
    wsb = {"sample": sv.spec_verify_workspace_bytes(sv.SPEC_MODE_SAMPLE, B, k, V, 1),
           "greedy": sv.spec_verify_workspace_bytes(sv.SPEC_MODE_GREEDY, B, k, V, 1),
           "tree": sv.spec_verify_workspace_bytes(sv.SPEC_MODE_TREE_GREEDY, Bt, N, Vt, 1)}
    wss = {key: torch.zeros(n, dtype=torch.uint8, device=dev) for key, n in wsb.items()}
    stream = torch.cuda.Stream(device=dev)   # the step's stream (and the sampling call's)
    side = {"greedy": torch.cuda.Stream(device=dev), "tree": torch.cuda.Stream(device=dev)}
    sp = stream.cuda_stream
    O = {key: v.data_ptr() for key, v in outs.items()}
    W = {key: v.data_ptr() for key, v in wss.items()}
    T = float(samp.temperature)

    def call_sample(s, st_ptr=None):
        st = lib.spec_verify_sample(s["t"].data_ptr(), s["d"].data_ptr(), 1, s["tok"].data_ptr(),
                                    s["ua"].data_ptr(), s["us"].data_ptr(), T, B, k, V, O["n"],
                                    O["tok"], O["p"], O["q"], O["R"], W["sample"],
                                    wsb["sample"], st_ptr or sp)
        assert st == 0, st

    def call_greedy(s, st_ptr=None):
        st = lib.spec_verify_greedy(s["t"].data_ptr(), 1, s["gtok"].data_ptr(), B, k, V,
                                    O["gn"], O["gtok"], W["greedy"], wsb["greedy"], st_ptr or sp)
        assert st == 0, st

    def call_tree(s, st_ptr=None):
        st = lib.spec_verify_tree_greedy(s["tt"].data_ptr(), 1, s["ttok"].data_ptr(),
                                         s["tpar"].data_ptr(), Bt, N, Vt, tree.max_depth,
                                         O["tn"], O["tpath"], O["ttok"], W["tree"], wsb["tree"],
                                         st_ptr or sp)
        assert st == 0, st

    calls = {"sample": call_sample, "greedy": call_greedy, "tree": call_tree}

    def step_serial(i):
        """The step's three calls one after another on the step's stream."""
        call_sample(sets[(2 * i) % NSETS])
        call_greedy(sets[(2 * i + 1) % NSETS])
        call_tree(sets[i % NSETS])

    ev_fork = torch.cuda.Event()
    ev_join = {key: torch.cuda.Event() for key in side}

    def step(i):
        """The step's three calls (independent batches) forked onto three
        streams and joined before the step ends: each call's serial tail (the
        finish and resolve kernels) overlaps the other calls' streaming."""
        ev_fork.record(stream)
        for key, sd in side.items():
            sd.wait_event(ev_fork)
        call_sample(sets[(2 * i) % NSETS])
        call_greedy(sets[(2 * i + 1) % NSETS], side["greedy"].cuda_stream)
        call_tree(sets[i % NSETS], side["tree"].cuda_stream)
        for key, sd in side.items():
            ev_join[key].record(sd)
            stream.wait_event(ev_join[key])

    # second-pass bytes depend on each set's accept outcomes (same data in all sets)
    with torch.cuda.stream(stream):
        call_sample(sets[0])
    stream.synchronize()
    n_acc = outs["n"].cpu().numpy()
    pass2_rows = int(np.where(n_acc < k, 2, 1).sum())
    bytes_sample = (B * (2 * k + 1) + pass2_rows) * V * eb
    bytes_greedy = B * (k + 1) * V * eb
    bytes_tree = Bt * N * Vt * eb
    bytes_step = bytes_sample + bytes_greedy + bytes_tree

    for i in range(args.warmup):
        step(i)
    stream.synchronize()

    # ---- headline: K whole steps replayed from CUDA graphs, events only
    # around the timed region.  One graph holds one rotation period of the
    # input sets (NSETS steps), so replays continue the rotation; a second
    # graph holds the K % NSETS steps left over.  Python and ctypes would
    # otherwise pace the launches: the host needs about as long to enqueue a
    # step's three calls as the GPU needs to run them. ----
    K = args.steps
    with torch.cuda.stream(stream):
        launches0 = sv.spec_verify_launch_count()
        step(0)
        launches_per_step = sv.spec_verify_launch_count() - launches0
    stream.synchronize()
    g_main = capture_graph(lambda: [step(i) for i in range(NSETS)], stream)
    g_tail = capture_graph(lambda: [step(i) for i in range(K % NSETS)], stream) \
        if K % NSETS else None
    with torch.cuda.stream(stream):
        for _ in range(3):
            g_main.replay()
    stream.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(K // NSETS):
            g_main.replay()
        if g_tail is not None:
            g_tail.replay()
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    launches = int(round(launches_per_step * K))
    if world > 1:
        torch.distributed.barrier()
    total_ms = ev0.elapsed_time(ev1)

    # ---- the same K steps with the three calls serialised on one stream
    # (reported beside the headline) ----
    g_serial = capture_graph(lambda: [step_serial(i) for i in range(NSETS)], stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g_serial.replay()
        es0 = torch.cuda.Event(enable_timing=True)
        es1 = torch.cuda.Event(enable_timing=True)
        es0.record(stream)
        for _ in range(max(1, K // NSETS)):
            g_serial.replay()
        es1.record(stream)
    stream.synchronize()
    serial_ms_step = es0.elapsed_time(es1) / (max(1, K // NSETS) * NSETS)

    # ---- spread of single steps: up to 200 steps, each a replay of a
    # one-step graph between its own pair of events (a step's calls stay
    # chained inside it) ----
    NS = min(200, K)
    g_one = [capture_graph(lambda i=i: step(i), stream) for i in range(NSETS)]
    sev = [torch.cuda.Event(enable_timing=True) for _ in range(NS + 1)]
    with torch.cuda.stream(stream):
        sev[0].record(stream)
        for i in range(NS):
            g_one[i % NSETS].replay()
            sev[i + 1].record(stream)
    stream.synchronize()
    step_samples = np.array([sev[i].elapsed_time(sev[i + 1]) for i in range(NS)])

    # ---- per-call durations: each call type alone, in its own loop of at
    # least max(K, 200) calls and 0.5 s, same rotation, from CUDA graphs of
    # NSETS calls (events between calls chained by programmatic dependent
    # launch distort the chain, so the mean comes from one event pair around
    # the whole loop; the spread from a second loop with one event pair per
    # graph replay of NSETS calls) ----
    per_call = {}
    for name in ("sample", "greedy", "tree"):
        fn = calls[name]
        per_call[name] = time_call_loop(
            lambda fn=fn: [fn(sets[i]) for i in range(NSETS)], NSETS, stream,
            min_calls=max(K, 200), min_seconds=0.5)
    mean_ms = np.array([per_call[n]["mean_ms"] for n in ("sample", "greedy", "tree")])
    t_wall1 = time.time()
    clk = clocks.stop(t_wall0, t_wall1) if clocks else None
    next_rows = measure_next_rows(dev, stream, tree, K) \
        if rank == 0 and not args.skip_next_rows else None
    at_scale = measure_at_scale(dev, stream, max(K, 200), measured_peak()[0]) \
        if rank == 0 and not args.skip_large else None
    total_ms = max_over_ranks(total_ms, dev)
    ms_step = total_ms / K
    value = job_rate(world, K, pos_step, total_ms)

    # ---- e2e through the public API: pinned host in, results back each step ----
    E = args.e2e_steps
    out_host = {key: torch.empty(v.shape, dtype=v.dtype).pin_memory() for key, v in outs.items()}
    h2d = sum(v.numel() * v.element_size() for v in h.values())
    d2h = sum(v.numel() * v.element_size() for v in outs.values())
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    def e2e_step(s):
        for key in h:
            s[key].copy_(h[key], non_blocking=True)
        sv.spec_verify_sample(s["t"].view(torch.bfloat16).view(B, k + 1, V),
                              s["d"].view(torch.bfloat16).view(B, k, V), s["tok"],
                              s["ua"], s["us"], T, outs["n"], outs["tok"], outs["p"],
                              outs["q"], outs["R"], wss["sample"], stream)
        sv.spec_verify_greedy(s["t"].view(torch.bfloat16).view(B, k + 1, V), s["gtok"],
                              outs["gn"], outs["gtok"], wss["greedy"], stream)
        sv.spec_verify_tree_greedy(s["tt"].view(torch.bfloat16).view(Bt, N, Vt),
                                   s["ttok"], s["tpar"], tree.max_depth, outs["tn"],
                                   outs["tpath"], outs["ttok"], wss["tree"], stream)
        for key in outs:
            out_host[key].copy_(outs[key], non_blocking=True)

    e2e = None
    if E > 0:
        with torch.cuda.stream(stream):
            for _ in range(2):
                e2e_step(sets[0])
            stream.synchronize()
            e0.record(stream)
            for _ in range(E):
                e2e_step(sets[0])
            e1.record(stream)
            stream.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
        e2e = {"value": round(job_rate(world, E, pos_step, e2e_ms), 1), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": E}

    # ---- roofline of the dominant kernel ----
    names = ["stream_stats + sample_finish (4-CTA clusters) kernels",
             "stream_argmax + argmax_resolve kernels (greedy)",
             "stream_argmax + argmax_resolve kernels (tree)"]
    byts = [bytes_sample, bytes_greedy, bytes_tree]
    peak, peak_kind = measured_peak()
    dom = int(np.argmax(mean_ms))
    dom_name = ["spec_verify_sample (stream_stats, sample_finish)",
                "spec_verify_greedy (stream_argmax, argmax_resolve)",
                "spec_verify_tree_greedy (stream_argmax, argmax_resolve)"][dom]
    achieved = byts[dom] / (mean_ms[dom] / 1e3) / 1e9
    traffic = recorded_traffic(["sample", "greedy", "tree"][dom])
    breakdown = {}
    for j, nm in enumerate(names):
        key = ["sample", "greedy", "tree"][j]
        pc = per_call[key]
        gbs = byts[j] / (mean_ms[j] / 1e3) / 1e9
        breakdown[key] = {
            "kernels": nm, "ms": round(float(mean_ms[j]), 5),
            "algorithmic_bytes": int(byts[j]), "gb_s": round(gbs, 1),
            "frac_of_peak": round(gbs / peak, 4),
            "calls_timed": pc["calls"],
            "ms_p10_p50_p90": [round(pc["p10_ms"], 5), round(pc["p50_ms"], 5),
                               round(pc["p90_ms"], 5)],
            "spread": f"{pc['spread_calls']} calls, one event pair per graph replay of "
                      f"{NSETS} calls"}
    step_gbs = bytes_step / (ms_step / 1e3) / 1e9

    headline_calls = {
        name: {"us_per_call": round(float(mean_ms[j]) * 1e3, 2),
               "positions_per_s": round(B * k / (mean_ms[j] / 1e3), 1),
               "gb_s": breakdown[name]["gb_s"], "frac_of_peak": breakdown[name]["frac_of_peak"],
               "calls_timed": per_call[name]["calls"]}
        for j, name in ((0, "sample"), (1, "greedy"))}
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT,
        "calls_B64_k4": headline_calls, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded Zipf-biased Gaussian logits; random draft trees)",
        "config": {"workload": "sample+greedy B=64 k=4 V=128256 bf16 T=1.0; "
                               "tree greedy B=16 N=60 depth<=6 V=128256 bf16",
                   "positions_per_step": pos_step, "algorithmic_bytes_per_step": bytes_step,
                   "logits": "bf16 in HBM; exponentials, sums and comparisons in f32 "
                             "(double-float sums, float64 final probabilities)",
                   "l2": f"{NSETS} rotating input sets; every set is reused only after a "
                         "246 MB tree read (> 129 MB L2)",
                   "parallelism": f"replicas x{world} (sequences shard, no collective)",
                   "streams": "each step forks its sampling, greedy and tree calls (independent "
                              "batches, one workspace each) onto three streams and joins them "
                              "before the next step"},
        "serial_ms_per_step": round(serial_ms_step, 5),
        "hbm_gbs": round(step_gbs, 1), "hbm_frac_of_peak": round(step_gbs / peak, 4),
        "sequences_per_s": round(job_rate(world, K, seqs_step, total_ms), 1),
        "step_ms_percentiles": {"p10": round(float(np.percentile(step_samples, 10)), 5),
                                "p50": round(float(np.percentile(step_samples, 50)), 5),
                                "p90": round(float(np.percentile(step_samples, 90)), 5),
                                "steps": int(NS), "timed": "one event pair per step (a one-step graph replay)"},
        "roofline": {"bound": "hbm", "kernel": dom_name, "timed": "whole call, its own loop of K calls (CUDA-graph replay)",
                     "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "traffic": traffic, "algorithmic_bytes_per_launch": int(byts[dom])},
        "breakdown": breakdown,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": clk,
        "next_rows": next_rows,
        "at_scale": at_scale,
    }
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        result["cpu_baseline"] = cpu_baseline(samp, greedy, tree, args.cpu_seconds)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


def measure_at_scale(dev, stream, K, peak):
    """The sampling and greedy calls on the large-batch workload (B=256
    sequences of k=7 drafts over V=151936, bf16, T=0.7; 1.17 GB of target and
    draft rows per sampling call, far above L2): each call type in its own
    loop of K calls, inputs resident in HBM."""
    import torch
    import speculative_decoding_verification_56_gb300 as sv
    from speculative_decoding_verification_56_gb300 import synth
    c = synth.zipf152k(seed=0)
    g = synth.greedy_variant(c, 0.7)
    B, k, V = c.B, c.k, c.V
    t = sv.to_device_logits(c.target, c.dtype, dev)
    d = sv.to_device_logits(c.draft, c.dtype, dev)
    tok = torch.from_numpy(c.tokens).to(dev)
    gtok = torch.from_numpy(g.tokens).to(dev)
    ua = torch.from_numpy(c.u_accept).to(dev)
    us = torch.from_numpy(c.u_sample).to(dev)
    del c, g
    i32 = dict(dtype=torch.int32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    n, otok = torch.empty(B, **i32), torch.empty(B, k + 1, **i32)
    p, q, R = torch.empty(B, k, **f32), torch.empty(B, k, **f32), torch.empty(B, **f32)
    ws = sv.alloc_workspace(sv.SPEC_MODE_SAMPLE, B, k, V, sv.SPEC_DTYPE_BF16, dev)
    wg = sv.alloc_workspace(sv.SPEC_MODE_GREEDY, B, k, V, sv.SPEC_DTYPE_BF16, dev)

    def call_sample():
        sv.spec_verify_sample(t, d, tok, ua, us, 0.7, n, otok, p, q, R, ws, stream)

    def call_greedy():
        sv.spec_verify_greedy(t, gtok, n, otok, wg, stream)

    out = {"workload": f"sample and greedy B={B} k={k} V={V} bf16 T=0.7 (Zipf-biased Gaussian "
                       "target, draft = target + N(0, 1.5^2))",
           "timed": f"each call type in its own loop of at least {K} calls (CUDA-graph "
                    "replays of 4 calls; spread from one event pair per replay)"}
    with torch.cuda.stream(stream):
        call_sample()
    stream.synchronize()
    pass2 = int(np.where(n.cpu().numpy() < k, 2, 1).sum())
    for name, fn, byts, pos in (
            ("sample", call_sample, (B * (2 * k + 1) + pass2) * V * 2, B * k),
            ("greedy", call_greedy, B * (k + 1) * V * 2, B * k)):
        pc = time_call_loop(lambda fn=fn: [fn() for _ in range(4)], 4, stream, min_calls=K,
                            min_seconds=0.0)
        ms = pc["mean_ms"]
        gbs = byts / (ms / 1e3) / 1e9
        out[name] = {"us_per_call": round(ms * 1e3, 2), "algorithmic_bytes": int(byts),
                     "gb_s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
                     "positions_per_s": round(pos / (ms / 1e3), 1), "calls_timed": pc["calls"],
                     "us_p10_p50_p90": [round(pc["p10_ms"] * 1e3, 2),
                                        round(pc["p50_ms"] * 1e3, 2),
                                        round(pc["p90_ms"] * 1e3, 2)]}
    del t, d, ws, wg
    torch.cuda.empty_cache()
    return out


def capture_graph(body, stream):
    """A CUDA graph of whatever `body` enqueues on `stream` (after one eager
    run of it, so every lazily initialised resource exists)."""
    import torch
    with torch.cuda.stream(stream):
        body()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        body()
    return g


def time_call_loop(body, calls_per_body, stream, min_calls=200, min_seconds=0.5):
    """Per-call time of whatever `body` enqueues (`calls_per_body` calls) on
    `stream`, replayed from one CUDA graph.

    mean: one event pair around a continuous loop of replays covering at
    least `min_calls` calls and `min_seconds` (after 3 untimed replays);
    spread: a second loop of as many replays, each between its own pair of
    events, whose per-call times give p10/p50/p90."""
    import torch
    g = capture_graph(body, stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(10):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    est = e0.elapsed_time(e1) / 10 / 1e3               # seconds per replay
    reps = max(-(-min_calls // calls_per_body), int(np.ceil(min_seconds / max(est, 1e-7))))
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    mean_ms = e0.elapsed_time(e1) / (reps * calls_per_body)
    nrep = max(-(-min_calls // calls_per_body), 50)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(nrep + 1)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(nrep):
            g.replay()
            ev[i + 1].record(stream)
    stream.synchronize()
    per = np.array([ev[i].elapsed_time(ev[i + 1]) for i in range(nrep)]) / calls_per_body
    return {"mean_ms": float(mean_ms), "calls": int(reps * calls_per_body),
            "p10_ms": float(np.percentile(per, 10)), "p50_ms": float(np.percentile(per, 50)),
            "p90_ms": float(np.percentile(per, 90)), "spread_calls": int(nrep * calls_per_body)}


def _time_loop(fn, stream, K, per_graph=20):
    """Mean ms of one fn() call on `stream`: `per_graph` calls are captured in
    a CUDA graph and the graph is replayed until K calls have run (3 untimed
    replays first), so host-side call overhead does not pace small kernels."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(3):
            fn()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(per_graph):
            fn()
    reps = max(1, K // per_graph)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1) / (reps * per_graph)


def _time_pair(fa, fb, stream, K, per_graph=4, rounds=8):
    """Mean ms of one fa() call and of one fb() call, timed in alternating
    rounds (each a CUDA-graph replay of about K / rounds calls) so that both
    see the same clock and thermal state; the median round of each is
    returned.  Used where a fused call is compared with its unfused
    equivalent: under the power cap the clock drifts over seconds."""
    import torch
    graphs = []
    for fn in (fa, fb):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(per_graph):
                fn()
        graphs.append(g)
    reps = max(1, K // (per_graph * rounds))
    out = [[], []]
    with torch.cuda.stream(stream):
        for g in graphs:
            for _ in range(2):
                g.replay()
        for _ in range(rounds):
            for i, g in enumerate(graphs):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(reps):
                    g.replay()
                e1.record(stream)
                out[i].append((e0, e1))
    stream.synchronize()
    med = []
    for pairs in out:
        ms = sorted(a.elapsed_time(b) / (reps * per_graph) for a, b in pairs)
        med.append(ms[len(ms) // 2])
    return med[0], med[1]


def lm_head_case(dev):
    """LM head fused with greedy verification on the greedy workload's shape:
    B=64, k=4 (320 target rows), hidden 4096, V=128256, bf16."""
    import torch
    import speculative_decoding_verification_56_gb300 as sv
    from speculative_decoding_verification_56_gb300 import synth
    Bl, kl, d, Vl = 64, 4, 4096, 128256
    Hb, Wb, tokl, _ = synth.make_lm_head_case(B=Bl, k=kl, d=d, V=Vl, seed=1)
    c = {"B": Bl, "k": kl, "d": d, "V": Vl, "rows": Bl * (kl + 1)}
    c["H"] = torch.from_numpy(Hb.view(np.int16)).view(torch.bfloat16).to(dev)
    c["W"] = torch.from_numpy(Wb.view(np.int16)).view(torch.bfloat16).to(dev)
    del Hb, Wb
    c["tokens"] = torch.from_numpy(tokl).to(dev)
    c["acc"] = torch.empty(Bl, dtype=torch.int32, device=dev)
    c["out"] = torch.empty(Bl, kl + 1, dtype=torch.int32, device=dev)
    c["ws"] = sv.alloc_workspace(sv.SPEC_MODE_LM_HEAD_GREEDY, Bl, kl, Vl, sv.SPEC_DTYPE_BF16, dev)
    c["call"] = lambda stream: sv.spec_lm_head_verify_greedy(c["H"], c["W"], c["tokens"], c["acc"],
                                                             c["out"], c["ws"], stream)
    return c


def grow_case(dev):
    """EAGLE-2 tree growth producing the tree workload's shape (16 trees of 60
    nodes): 6 layers of 8 frontier rows over V=128256 bf16 draft rows."""
    import torch
    import speculative_decoding_verification_56_gb300 as sv
    from speculative_decoding_verification_56_gb300 import synth
    Bg, Dg, Kg, Mg, Vg = 16, 6, 8, 59, 128256
    zg = synth.make_grow_logits(B=Bg, D=Dg, K=Kg, V=Vg, seed=2)
    c = {"B": Bg, "D": Dg, "K": Kg, "M": Mg, "V": Vg}
    c["z"] = sv.to_device_logits(zg, "bf16", dev)
    del zg
    gi = dict(dtype=torch.int32, device=dev)
    c["out"] = [torch.empty(Bg, Mg + 1, **gi) for _ in range(3)] + \
        [torch.empty(Bg, Mg + 1, dtype=torch.float32, device=dev)]
    c["ws"] = sv.alloc_workspace(sv.SPEC_MODE_TREE_GROW, Bg, Kg, Vg, sv.SPEC_DTYPE_BF16, dev)
    c["call"] = lambda stream: sv.spec_tree_grow(c["z"], 1.0, Mg, *c["out"], c["ws"], stream)
    return c


def sample_case(dev):
    """Sampling verification on the headline workload (B=64, k=4, V=128256,
    bf16) over four device copies of the logits used in turn, as in the
    per-call loops: each call reads logits that the previous three did not."""
    import torch
    import speculative_decoding_verification_56_gb300 as sv
    from speculative_decoding_verification_56_gb300 import synth
    cs = synth.zipf128k(seed=0)
    c = {"sets": [(sv.to_device_logits(cs.target, cs.dtype, dev),
                   sv.to_device_logits(cs.draft, cs.dtype, dev)) for _ in range(NSETS)],
         "i": 0}
    tok = torch.from_numpy(cs.tokens).to(dev)
    ua = torch.from_numpy(cs.u_accept).to(dev)
    us = torch.from_numpy(cs.u_sample).to(dev)
    ws = sv.alloc_workspace(sv.SPEC_MODE_SAMPLE, cs.B, cs.k, cs.V, sv.SPEC_DTYPE_BF16, dev)

    def call(stream):
        t, d = c["sets"][c["i"] % NSETS]
        c["i"] += 1
        sv.verify_sample(t, d, tok, ua, us, cs.temperature, workspace=ws, stream=stream)
    c["call"] = call
    return c


def step_case(dev):
    """One verification step per call, its three calls one after another on
    one stream: sampling and greedy (B=64, k=4, V=128256) and tree greedy
    (16 trees of 60 nodes), bf16, over four device copies of the inputs."""
    import torch
    import speculative_decoding_verification_56_gb300 as sv
    samp, greedy, tree = workload(0)
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    sets = [dict(t=sv.to_device_logits(samp.target, samp.dtype, dev),
                 d=sv.to_device_logits(samp.draft, samp.dtype, dev),
                 tt=sv.to_device_logits(tree.target, tree.dtype, dev)) for _ in range(NSETS)]
    tok, ua, us, gtok = up(samp.tokens), up(samp.u_accept), up(samp.u_sample), up(greedy.tokens)
    ttok, tpar = up(tree.tokens), up(tree.parents)
    ws = sv.alloc_workspace(sv.SPEC_MODE_SAMPLE, samp.B, samp.k, samp.V, sv.SPEC_DTYPE_BF16, dev)
    wg = sv.alloc_workspace(sv.SPEC_MODE_GREEDY, greedy.B, greedy.k, greedy.V, sv.SPEC_DTYPE_BF16,
                            dev)
    wt = sv.alloc_workspace(sv.SPEC_MODE_TREE_GREEDY, tree.B, tree.N, tree.V, sv.SPEC_DTYPE_BF16,
                            dev)
    c = {"i": 0}

    def call(stream):
        x = sets[c["i"] % NSETS]
        c["i"] += 1
        sv.verify_sample(x["t"], x["d"], tok, ua, us, samp.temperature, workspace=ws,
                         stream=stream)
        sv.verify_greedy(x["t"], gtok, workspace=wg, stream=stream)
        sv.verify_tree_greedy(x["tt"], ttok, tpar, tree.max_depth, workspace=wt, stream=stream)
    c["call"] = call
    return c


def profile_case(name, calls):
    """Run one call type `calls` times, untimed: the program ncu profiles
    (`--profile-case`)."""
    import torch
    dev = torch.device("cuda", 0)
    c = {"lm_head_greedy": lm_head_case, "tree_grow": grow_case, "sample": sample_case,
         "step": step_case}[name](dev)
    for _ in range(calls):
        c["call"](None)
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": name, "calls": calls}), flush=True)


def measure_next_rows(dev, stream, tree, K):
    """The kernels around the draft tree (each timed alone, outside the step):
    tree attention mask of the tree workload's trees, and the KV commit of
    the paths tree verification accepts on it."""
    import torch
    import speculative_decoding_verification_56_gb300 as sv
    out = {}
    Bt, N = tree.parents.shape
    W = (N + 31) // 32
    par = torch.from_numpy(tree.parents).to(dev)
    mask = torch.empty(Bt, N, W, dtype=torch.int32, device=dev)
    depth = torch.empty(Bt, N, dtype=torch.int32, device=dev)
    wsm = sv.alloc_workspace(sv.SPEC_MODE_TREE_MASK, Bt, N, 1, sv.SPEC_DTYPE_F32, dev)
    ms = _time_loop(lambda: sv.spec_tree_attention_mask(par, mask, depth, wsm, stream), stream, K)
    out["tree_mask"] = {"workload": f"B={Bt} N={N} trees (the tree-verification workload)",
                        "us_per_call": round(ms * 1e3, 3),
                        "bytes": int(Bt * N * 4 + Bt * N * W * 4 + Bt * N * 4),
                        "bound": "launch latency (one kernel, a few KB)",
                        "timed": "CUDA-graph replay of 20 calls"}

    # KV commit of the paths that tree verification accepts on that workload:
    # 32 layers x (K, V) planes, 8 KV heads x 128 bf16 per entry, 400+ prefix
    res = sv.verify_tree_greedy(sv.to_device_logits(tree.target, tree.dtype, dev),
                                torch.from_numpy(tree.tokens).to(dev), par, tree.max_depth)
    path, acc = res["path_nodes"], res["accepted_len"]
    planes, E, L = 64, 1024, 512
    # successive calls use 12 prefix lengths 100, 130, ..., 430, so the entries
    # they move (12 x ~12.6 MB) do not stay in the 129 MB L2 between calls
    bases = [(100 + 30 * j + torch.arange(Bt, dtype=torch.int32, device=dev) % 2).contiguous()
             for j in range(12)]
    cache = torch.empty(planes, Bt, L, E, dtype=torch.bfloat16, device=dev).normal_()
    new_len = torch.empty(Bt, dtype=torch.int32, device=dev)
    wsk = sv.alloc_workspace(sv.SPEC_MODE_KV_COMMIT, Bt, N, 1, sv.SPEC_DTYPE_F32, dev)
    p_np, a_np = path.cpu().numpy(), acc.cpu().numpy()
    moves = sum(int((p_np[b, 1:a_np[b] + 1] != np.arange(1, a_np[b] + 1)).sum()) for b in range(Bt))
    turn = [0]

    def kv_call():
        sv.spec_kv_commit_path(cache, bases[turn[0] % 12], acc, path, N, new_len, wsk, stream)
        turn[0] += 1
    ms = _time_loop(kv_call, stream, K, per_graph=24)
    byts = 2 * moves * planes * E * 2
    out["kv_commit"] = {"workload": f"B={Bt} accepted tree paths ({int(a_np.sum())} nodes, "
                                    f"{moves} moved), {planes} planes x {E} bf16 per entry; "
                                    "12 rotating prefix lengths (151 MB touched > L2)",
                        "us_per_call": round(ms * 1e3, 3), "bytes": int(byts),
                        "gb_s": round(byts / (ms / 1e3) / 1e9, 1),
                        "bound": "HBM gather, latency at this size",
                        "timed": "CUDA-graph replay of 24 calls"}
    del cache

    # LM head fused with greedy verification: the greedy workload's shape
    # (B=64, k=4 -> 320 target rows) with hidden size 4096 and V=128256,
    # against the unfused path (cuBLAS GEMM writing the logits, then greedy
    # verification of the logits)
    lm = lm_head_case(dev)
    Bl, kl, d, Vl, rows = lm["B"], lm["k"], lm["d"], lm["V"], lm["rows"]
    H, Wm, tk, acc_l, out_l, wsl = lm["H"], lm["W"], lm["tokens"], lm["acc"], lm["out"], lm["ws"]
    wsg = sv.alloc_workspace(sv.SPEC_MODE_GREEDY, Bl, kl, Vl, sv.SPEC_DTYPE_BF16, dev)
    logits = torch.empty(rows, Vl, dtype=torch.bfloat16, device=dev)
    def unfused():
        torch.matmul(H, Wm.t(), out=logits)
        sv.spec_verify_greedy(logits.view(Bl, kl + 1, Vl), tk, acc_l, out_l, wsg, stream)
    ms_f, ms_u = _time_pair(
        lambda: sv.spec_lm_head_verify_greedy(H, Wm, tk, acc_l, out_l, wsl, stream), unfused,
        stream, max(64, K // 10), per_graph=4)
    flops = 2.0 * rows * d * Vl
    w_bytes = Vl * d * 2
    peak_tf, peak_kind_tf = measured_tflops()
    out["lm_head_greedy"] = {
        "workload": f"B={Bl} k={kl} ({rows} rows), hidden {d}, V={Vl}, bf16 in, fp32 accumulate",
        "us_per_call": round(ms_f * 1e3, 2),
        "tflops": round(flops / (ms_f / 1e3) / 1e12, 1),
        "tensor_peak_tflops": peak_tf, "tensor_frac": round(flops / (ms_f / 1e3) / 1e12 / peak_tf, 4),
        "peak_source": peak_kind_tf,
        "w_lm_gb_s": round(w_bytes / (ms_f / 1e3) / 1e9, 1),
        "unfused_us_per_call": round(ms_u * 1e3, 2),
        "unfused": "torch.matmul (cuBLAS) writing bf16 logits, then spec_verify_greedy",
        "bound": "tensor cores on SM pairs (M=256 x N=160 MMAs from one issuing thread per pair), "
                 "W_LM streamed once",
        "timed": "fused and unfused in 8 alternating rounds of CUDA-graph replays (4 calls "
                 "per graph); median round of each"}

    # LM head fused with sampling verification on the same shape: 320 target
    # rows, 256 drafted features (the target's first k hidden states of each
    # sequence plus N(0, 0.3^2) noise), T = 1; the unfused path writes both
    # logits matrices with cuBLAS and runs spec_verify_sample
    g = torch.Generator(device=dev).manual_seed(3)
    Hd = (H.view(Bl, kl + 1, d)[:, :kl].float()
          + 0.3 * torch.randn(Bl, kl, d, device=dev, generator=g)).to(torch.bfloat16)
    Hd = Hd.reshape(Bl * kl, d).contiguous()
    ua = torch.rand(Bl, kl, device=dev, generator=g)
    us = torch.rand(Bl, device=dev, generator=g)
    wss = sv.alloc_workspace(sv.SPEC_MODE_LM_HEAD_SAMPLE, Bl, kl, Vl, sv.SPEC_DTYPE_BF16, dev)
    wsu = sv.alloc_workspace(sv.SPEC_MODE_SAMPLE, Bl, kl, Vl, sv.SPEC_DTYPE_BF16, dev)
    i32 = dict(dtype=torch.int32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    so = dict(n=torch.empty(Bl, **i32), tok=torch.empty(Bl, kl + 1, **i32),
              p=torch.empty(Bl, kl, **f32), q=torch.empty(Bl, kl, **f32), R=torch.empty(Bl, **f32))
    logits_d = torch.empty(Bl * kl, Vl, dtype=torch.bfloat16, device=dev)

    def fused_sample():
        sv.spec_lm_head_verify_sample(H, Hd, Wm, tk, ua, us, 1.0, so["n"], so["tok"], so["p"],
                                      so["q"], so["R"], wss, stream)

    def unfused_sample():
        torch.matmul(H, Wm.t(), out=logits)
        torch.matmul(Hd, Wm.t(), out=logits_d)
        sv.spec_verify_sample(logits.view(Bl, kl + 1, Vl), logits_d.view(Bl, kl, Vl), tk, ua, us,
                              1.0, so["n"], so["tok"], so["p"], so["q"], so["R"], wsu, stream)
    ms_fs, ms_us = _time_pair(fused_sample, unfused_sample, stream, max(32, K // 20), per_graph=2)
    flops_s = 2.0 * (rows + Bl * kl) * d * Vl
    out["lm_head_sample"] = {
        "workload": f"B={Bl} k={kl}: {rows} target rows and {Bl * kl} drafted features, hidden {d}, "
                    f"V={Vl}, bf16 in, fp32 accumulate, T=1",
        "us_per_call": round(ms_fs * 1e3, 2),
        "tflops_statistics_gemm_equivalent": round(flops_s / (ms_fs / 1e3) / 1e12, 1),
        "unfused_us_per_call": round(ms_us * 1e3, 2),
        "unfused": "torch.matmul (cuBLAS) writing bf16 target and draft logits, then "
                   "spec_verify_sample",
        "launches": 4,
        "bound": "the statistics GEMM (576 rows) and a second pass over W_LM for the 2B drawn rows",
        "timed": "fused and unfused in 8 alternating rounds of CUDA-graph replays (2 calls "
                 "per graph); median round of each"}
    del H, Wm, logits, lm, Hd, logits_d, wss, wsu

    # EAGLE-2 tree growth producing the tree workload's shape (16 trees of 60
    # nodes): 6 layers of 8 frontier rows over V=128256 bf16 draft rows
    gr = grow_case(dev)
    Bg, Dg, Kg, Mg, Vg = gr["B"], gr["D"], gr["K"], gr["M"], gr["V"]
    ms_g = _time_loop(lambda: gr["call"](stream), stream, max(40, K // 10), per_graph=8)
    rows_read = Bg * (1 + (Dg - 1) * Kg)
    gbytes = rows_read * Vg * 2
    out["tree_grow"] = {"workload": f"B={Bg} trees, {Dg} layers x {Kg} frontier rows, V={Vg} "
                                    f"bf16, budget {Mg} nodes",
                        "us_per_call": round(ms_g * 1e3, 2), "bytes": int(gbytes),
                        "gb_s": round(gbytes / (ms_g / 1e3) / 1e9, 1),
                        "launches": 2,
                        "bound": "streaming top-k: issue and CTA-barrier latency (HBM at 1/3); "
                                 "per-tree bookkeeping: latency chain on 16 CTAs",
                        "timed": "CUDA-graph replay of 8 calls"}
    del gr
    return out


def cpu_baseline(samp, greedy, tree, budget_s):
    """The float64 oracle as it stands, single-threaded, on whole steps of the
    same workload until the budget is spent."""
    import oracle
    oracle.build()
    pos = positions(samp, greedy, tree)
    t0 = time.perf_counter()
    steps = 0
    while True:
        oracle.verify_sample(samp.target, samp.draft, samp.tokens, samp.u_accept, samp.u_sample,
                             samp.temperature, dtype=samp.dtype)
        oracle.verify_greedy(greedy.target, greedy.tokens, dtype=greedy.dtype)
        oracle.verify_tree_greedy(tree.target, tree.tokens, tree.parents, tree.max_depth,
                                  dtype=tree.dtype)
        steps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    out = {"value": round(steps * pos / el, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": f"{steps} whole step(s) of the same workload (sample+greedy 64 seqs, "
                     f"16 trees) in {el:.1f} s, single thread, float64 C oracle"}
    out["all_cores"] = cpu_baseline_all_cores(samp, greedy, tree, budget_s / 2)
    return out


def cpu_baseline_all_cores(samp, greedy, tree, budget_s):
    """The same oracle on every host core: one task per sequence or tree of a
    whole step, run by a pool of os.cpu_count() threads (the C oracle keeps no
    shared state, and ctypes releases the interpreter lock during each call)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    pos = positions(samp, greedy, tree)
    cores = os.cpu_count() or 1

    def task(unit):
        mode, b = unit
        s = slice(b, b + 1)
        if mode == 0:
            oracle.verify_sample(samp.target[s], samp.draft[s], samp.tokens[s], samp.u_accept[s],
                                 samp.u_sample[s], samp.temperature, dtype=samp.dtype)
        elif mode == 1:
            oracle.verify_greedy(greedy.target[s], greedy.tokens[s], dtype=greedy.dtype)
        else:
            oracle.verify_tree_greedy(tree.target[s], tree.tokens[s], tree.parents[s],
                                      tree.max_depth, dtype=tree.dtype)

    units = ([(0, b) for b in range(samp.B)] + [(1, b) for b in range(greedy.B)] +
             [(2, b) for b in range(tree.B)])
    with ThreadPoolExecutor(max_workers=cores) as ex:
        t0 = time.perf_counter()
        steps = 0
        while True:
            list(ex.map(task, units))
            steps += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                break
    return {"value": round(steps * pos / el, 1), "unit": UNIT, "cores": cores,
            "sample": f"{steps} whole step(s) in {el:.1f} s, one task per sequence or tree on "
                      f"{cores} threads"}


# ---------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    samp, greedy, tree = workload(args.seed)
    # one step = one sequence (or tree) of one mode, cycling through the modes
    units = [("sample", samp.k), ("greedy", greedy.k), ("tree", tree.N - 1)]

    def ref_step(i):
        mode, _ = units[i % 3]
        if mode == "sample":
            b = (i // 3) % samp.B
            s = slice(b, b + 1)
            oracle.verify_sample(samp.target[s], samp.draft[s], samp.tokens[s], samp.u_accept[s],
                                 samp.u_sample[s], samp.temperature, dtype=samp.dtype)
        elif mode == "greedy":
            b = (i // 3) % greedy.B
            s = slice(b, b + 1)
            oracle.verify_greedy(greedy.target[s], greedy.tokens[s], dtype=greedy.dtype)
        else:
            b = (i // 3) % tree.B
            s = slice(b, b + 1)
            oracle.verify_tree_greedy(tree.target[s], tree.tokens[s], tree.parents[s],
                                      tree.max_depth, dtype=tree.dtype)
        return units[i % 3][1]

    for i in range(args.warmup):
        ref_step(i)
    pos = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        pos += ref_step(i)
    el = time.perf_counter() - t0
    value = pos / el
    out = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(el * 1e3 / max(args.steps, 1), 4), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "impl": "reference",
           "config": {"workload": "sample+greedy B=64 k=4 V=128256 bf16 T=1.0; "
                                  "tree greedy B=16 N=60 depth<=6 V=128256 bf16",
                      "reference": "float64 CPU oracle (the method written out from the "
                                   "pages); one sequence or tree per step, cycling modes"},
           "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": 1,
                            "kind": "oracle",
                            "sample": "one sequence (sample, greedy) or one tree per step"},
           "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    args = parse_args()
    rank, world, local_rank = dist_env()
    if args.profile_case:
        profile_case(args.profile_case, args.calls)
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
