"""Benchmark of one speculative cycle (Markov-head draft + lossless verify).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C2]
                    [--impl ours|reference] [--no-cpu-baseline]

A step is one full cycle over one batch: spec_markov_draft (gamma sequential
draft steps) then spec_verify, through the C ABI, on synthetic seeded inputs
of the named workload.  The metric is verified draft positions per second
(sum over requests of the verify length L_b per cycle / cycle time); rank 0
prints ONE JSON line.  Under torchrun every rank runs its own batch on its
own GPU (independent replicas, weak scaling, no data-path collective).

--impl reference times the float64 CPU oracle on the host cores on a bounded
sample of the same workload (the pages define no runnable reference system).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified draft positions/sec and achieved HBM GB/s (% of GB300 peak) at 1 GPU"
UNIT = "verified draft positions/s"
NOMINAL_HBM_GBS = 8000.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="C2")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--eager", action="store_true",
                    help="launch the timed cycles one call at a time instead of replaying a CUDA graph")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the scheduled, RNN-head and tree passes (profiling runs)")
    ap.add_argument("--other-configs", default="C1,C3,C4",
                    help="other named workloads timed at full size beside the headline ('' = none)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", 6800.0)), float(d.get("bf16_tflops", 1900.0)), "measured"
    return 6800.0, 1900.0, "fallback"


def recorded_traffic(kernel, config):
    """DRAM bytes per launch of `kernel` from its committed ncu summary
    (profiles/<kernel>_<config>.md), or None when there is none or when the
    kernel's sources changed since the counters were taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", f"{kernel}_{config}.md")
    if not os.path.exists(p):
        return None
    fields = {}
    for line in open(p):
        line = line.strip()
        for key in ("traffic_bytes_per_launch:", "sources:", "source_sha256:"):
            if line.startswith(key):
                fields[key[:-1]] = line[len(key):].strip()
    if len(fields) != 3:
        return None
    h = hashlib.sha256()
    for f in fields["sources"].split():
        fp = os.path.join(ROOT, f)
        if not os.path.exists(fp):
            return None
        with open(fp, "rb") as fh:
            h.update(fh.read())
    if h.hexdigest() != fields["source_sha256"]:
        return None
    return float(fields["traffic_bytes_per_launch"])


# Target decode step used for the draft cost ratio c: the pages' estimate of a
# 70B bf16 decode step (about 140 GB of weights read at 3.35 TB/s: ~42 ms).
TARGET_STEP_MS = 42.0


def operating_point(d, bufs, draft_prof, steps):
    """The analytic speed-up report from this run's measured acceptance (device
    statistics of the last cycle's outputs) and the draft time per cycle."""
    import torch
    from speculative_decoding_draft_04_gb300 import _lib
    out = torch.zeros(4, dtype=torch.float64, device=bufs.alpha.device)
    _lib.spec_acceptance_stats(bufs.alpha, d.verify_len, bufs.accept_len, out)
    s = out.cpu().numpy()
    alpha = float(s[0] / s[1]) if s[1] else float("nan")
    tau = float(s[2] / s[3]) if s[3] else float("nan")
    draft_ms = draft_prof[0] / max(steps, 1)
    c = draft_ms / (d.gamma * TARGET_STEP_MS) if draft_ms > 0 else float("nan")
    rep = _lib.spec_operating_point(min(max(alpha, 0.0), 1.0), c, d.gamma, 256) \
        if alpha == alpha and c == c and c > 0 else {}
    return {"measured_alpha": alpha, "measured_tau": tau, "draft_ms_per_cycle": draft_ms,
            "c": c, "c_source": f"draft time / (gamma x {TARGET_STEP_MS} ms 70B decode step, the pages' estimate)",
            **{k: v for k, v in rep.items()}}


def scheduled_pass(args, w, d, bufs, stream, flush, rank, dev):
    """The confidence-scheduled cycle on the same workload: draft, confidence
    head, prefix scheduler, then verification at the scheduled lengths.  Timed
    like the main pass (events around each cycle, L2 flushed outside them),
    then once more with per-kernel events for the scheduler's stages."""
    import torch
    from speculative_decoding_draft_04_gb300 import _lib, engine
    from speculative_decoding_draft_04_gb300 import workloads as W
    si = W.make_schedule_inputs(W.config(args.config), trial=rank)
    s = engine.DeviceSchedule.from_inputs(si, w.B, w.gamma, w.dtype, dev)

    def step():
        engine.scheduled_cycle(d, bufs, s, stream)
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    ms = float(sum(a.elapsed_time(b) for a, b in evs) / args.steps)
    _lib.spec_profile_enable(True)
    _lib.spec_profile_read()
    for _ in range(args.steps):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    prof = _lib.spec_profile_read()
    _lib.spec_profile_enable(False)
    tot = s.totals.cpu().numpy()
    positions = int(s.verify_len.sum().item())
    esz = 2 if w.dtype == "bf16" else 4
    conf_bytes = w.B * w.gamma * (si.d + w.r) * esz + (si.d + w.r) * 4 + w.B * w.gamma * 8
    c_ms, c_n = prof.get("confidence", (0.0, 0))
    c_avg = c_ms / max(c_n, 1)
    hbm_peak, _, peak_src = measured_peaks()
    return {
        "ms_per_step": ms, "value": positions / (ms * 1e-3), "unit": UNIT,
        "positions_per_step": positions, "B": int(tot[0]), "tau": float(tot[1]) * 2.0 ** -36,
        "stop_reason": int(tot[3]), "theta": float(s.theta.item()),
        "hidden_width": si.d, "cost_table": "1000/sqrt(42^2 + (B t1)^2) steps/s, knee at B(1+gamma/2)",
        "stages_ms_per_step": {k: v[0] / args.steps for k, v in prof.items() if v[1]},
        "confidence_roofline": {"bound": "hbm", "algorithmic_bytes_per_launch": conf_bytes,
                                "avg_launch_ms": c_avg,
                                "achieved": conf_bytes / (c_avg * 1e-3) / 1e9 if c_avg else None,
                                "peak": hbm_peak, "peak_source": peak_src, "unit": "GB/s"},
    }


def rnn_pass(args, w, d, bufs, stream, flush, rank, dev):
    """The cycle with the RNN head drafting on the same workload (its factor
    rows feed the verification), timed like the main pass."""
    import torch
    from speculative_decoding_draft_04_gb300 import _lib, engine
    from speculative_decoding_draft_04_gb300 import workloads as W
    ri = W.make_rnn_inputs(W.config(args.config), trial=rank)
    h = engine.DeviceRnn.from_inputs(ri, d, dev)

    def step():
        engine.rnn_cycle(d, bufs, h, stream)
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    ms = float(sum(a.elapsed_time(b) for a, b in evs) / args.steps)
    _lib.spec_profile_enable(True)
    _lib.spec_profile_read()
    for _ in range(args.steps):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    prof = _lib.spec_profile_read()
    _lib.spec_profile_enable(False)
    positions = int(w.verify_len.sum())
    return {"ms_per_step": ms, "value": positions / (ms * 1e-3), "unit": UNIT,
            "positions_per_step": positions,
            "draft_status": engine.status_words(bufs.dstatus),
            "stages_ms_per_step": {k: v[0] / args.steps for k, v in prof.items() if v[1]}}


def config_pass(name, args, flush, dev, warmup=3, steps=10):
    """One other named workload at its full size: cycles with L2 flushed
    between them (cold, events around each cycle) and back to back (warm),
    then once more with per-kernel events for the draft / verification split.
    Returns the times and the cycle's algorithmic HBM rate."""
    import torch
    from speculative_decoding_draft_04_gb300 import _lib, engine
    from speculative_decoding_draft_04_gb300 import workloads as W
    w = W.make_workload(W.config(name), trial=0)
    d = engine.DeviceWorkload.from_workload(w, dev)
    b = engine.Buffers.for_workload(d, dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        flush.zero_()
        engine.cycle(d, b, stream)
    torch.cuda.synchronize()

    def timed(cold):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for i in range(steps):
            if cold:
                flush.zero_()
            evs[i][0].record(stream)
            engine.cycle(d, b, stream)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return float(sum(a.elapsed_time(e) for a, e in evs) / steps)
    cold, warm = timed(True), timed(False)
    _lib.spec_profile_enable(True)
    _lib.spec_profile_read()
    for _ in range(steps):
        flush.zero_()
        engine.cycle(d, b, stream)
    torch.cuda.synchronize()
    prof = _lib.spec_profile_read()
    _lib.spec_profile_enable(False)
    stages = {k: v[0] / steps for k, v in prof.items() if v[1]}
    draft_ms = stages.get("draft_persistent", 0.0) + stages.get("draft_slice", 0.0)
    verify_ms = sum(v for k, v in stages.items() if not k.startswith("draft"))
    hbm_peak, _, _ = measured_peaks()
    db, vb, _ = algorithmic_bytes(w)
    gbs = (db + vb) / (cold * 1e-3) / 1e9
    positions = int(w.verify_len.sum())
    out = {"workload": name + ": " + W.CONFIG_DESCRIPTIONS[name],
           "draft_kernel": "slice-resident" if "draft_slice" in stages else "tile-strided",
           "ms_per_cycle_cold": cold, "ms_per_cycle_warm": warm,
           "draft_ms": draft_ms, "verify_ms": verify_ms,
           "value": positions / (cold * 1e-3), "unit": UNIT, "positions_per_cycle": positions,
           "cycle_algorithmic_bytes": db + vb, "cycle_gbs_cold": gbs,
           "frac_of_8TBs": gbs / NOMINAL_HBM_GBS, "frac_of_measured": gbs / hbm_peak,
           "draft_gbs": db / (draft_ms * 1e-3) / 1e9 if draft_ms else None,
           "stages_ms_per_cycle": stages,
           "status": [engine.status_words(b.dstatus), engine.status_words(b.vstatus)]}
    del d, b
    torch.cuda.empty_cache()
    return out


TREE_SLOTS, TREE_BUDGET = 24, 12


def tree_pass(args, w, d, flush, rank, dev):
    """The tree path on the same requests: select the top-12 of 24 candidate
    slots per request, draft them, verify the tree.  Timed with events around
    each cycle (L2 flushed outside them), then with per-kernel events."""
    import torch
    from speculative_decoding_draft_04_gb300 import _lib, engine
    from speculative_decoding_draft_04_gb300 import workloads as W
    ti = W.make_tree_inputs(W.config(args.config), w, TREE_SLOTS, trial=rank)
    t = engine.DeviceTree.from_inputs(ti, d, TREE_BUDGET, dev)
    stream = torch.cuda.current_stream(dev)
    steps = max(1, min(args.steps, 5))

    def step():
        engine.tree_cycle(d, t, stream)
    for _ in range(2):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    ms = float(sum(a.elapsed_time(b) for a, b in evs) / steps)
    _lib.spec_profile_enable(True)
    _lib.spec_profile_read()
    flush.zero_()
    step()
    torch.cuda.synchronize()
    prof = _lib.spec_profile_read()
    _lib.spec_profile_enable(False)
    acc = t.accept_len.cpu().numpy()
    return {"ms_per_step": ms, "steps": steps, "slots": TREE_SLOTS, "budget": TREE_BUDGET,
            "accepted_per_request": float(acc.mean()),
            "tokens_per_s": float((acc + 1).sum()) / (ms * 1e-3),
            "status": engine.status_words(t.status),
            "stages_ms": {k: v[0] for k, v in prof.items() if v[1]},
            "arithmetic": "double-float throughout (direct formulation, not tiled)"}


def algorithmic_bytes(w):
    """Bytes a cycle must move at least (logits + W2 once per call): draft = B*g*V*s + r*V*s; verify = sum(L+1)*V*s (target
    rows) + sum(L)*V*s (U rows re-read to rebuild q) + r*V*s."""
    s = 2 if w.dtype == "bf16" else 4
    L = w.verify_len.astype(np.int64)
    draft = w.B * w.gamma * w.V * s + w.r * w.V * s
    verify = int((L + 1).sum()) * w.V * s + int(L.sum()) * w.V * s + w.r * w.V * s
    per_stage = {
        "draft_persistent": draft,                                  # per launch (whole draft)
        "draft_slice": draft,                                       # the same, slice-resident kernel
        "target_stats": int((L + 1).sum()) * w.V * s,
        "verify_tile": int(L.sum()) * w.V * s + w.r * w.V * s,
        "verify_slice": int(L.sum()) * w.V * s + w.r * w.V * s,   # the same, slice-resident tiles
    }
    return draft, verify, per_stage


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.f = None

    def __enter__(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.f is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.f.flush()
        self.f.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in self.f.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names[1:], parts[5:9]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(n)
        os.unlink(self.f.name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def oracle_timing(name, trial, warmup, steps, seconds):
    """Time the float64 oracle (as it stands) in a single-threaded subprocess:
    `warmup` untimed then `steps` timed samples, each a bounded run of whole
    requests (draft + verify) of the named workload; returns per-step
    (requests, positions, seconds)."""
    code = f"""
import os, sys, time, json
sys.path.insert(0, {ROOT!r})
import numpy as np
from speculative_decoding_draft_04_gb300 import workloads as W
from oracle import spec_oracle as O
w = W.make_workload(W.config({name!r}), trial={trial})
W1, W2 = w.f64("W1"), w.f64("W2")
b = 0
def sample(limit):
    global b
    t0 = time.perf_counter(); done = 0; pos = 0
    while True:
        tb = W.to_f64(w.target[b], w.dtype); ub = W.to_f64(w.U[b], w.dtype)
        O.cycle_request(tb, ub, W1, W2, w.anchor[b], float(w.temperature[b]),
                        w.u_draft[b].astype(np.float64), int(w.verify_len[b]),
                        w.u_accept[b].astype(np.float64), float(w.u_final[b]))
        done += 1; pos += int(w.verify_len[b]); b = (b + 1) % w.B
        el = time.perf_counter() - t0
        if el > limit: return (done, pos, el)
for _ in range({warmup}): sample({seconds} / 4)
print(json.dumps([sample({seconds}) for _ in range({steps})]))
"""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                         timeout=(warmup + steps) * seconds * 4 + 900)
    if out.returncode != 0:
        raise RuntimeError("oracle timing failed: " + out.stderr[-500:])
    return json.loads(out.stdout.strip().splitlines()[-1])


def oracle_timing_all_cores(name, seconds, procs=None, steps=1):
    """The same oracle on every host core: `procs` single-threaded processes
    (spawned once), each drawing the workload; then `steps` timed samples,
    each started by all processes together and ended when every process has
    run whole requests (request b, b + procs, ...) for about `seconds`.
    Returns per step (requests, positions, wall seconds of the slowest), and
    the process count."""
    procs = procs or (os.cpu_count() or 1)
    code = f"""
import os, sys, time, json
import multiprocessing as mp
sys.path.insert(0, {ROOT!r})
def work(i, n, bar, q):
    import numpy as np
    from speculative_decoding_draft_04_gb300 import workloads as W
    from oracle import spec_oracle as O
    w = W.make_workload(W.config({name!r}), trial=0)
    W1, W2 = w.f64("W1"), w.f64("W2")
    b = i % w.B
    for step in range({steps}):
        bar.wait()
        t0 = time.perf_counter(); done = 0; pos = 0
        while True:
            tb = W.to_f64(w.target[b], w.dtype); ub = W.to_f64(w.U[b], w.dtype)
            O.cycle_request(tb, ub, W1, W2, w.anchor[b], float(w.temperature[b]),
                            w.u_draft[b].astype(np.float64), int(w.verify_len[b]),
                            w.u_accept[b].astype(np.float64), float(w.u_final[b]))
            done += 1; pos += int(w.verify_len[b]); b = (b + n) % w.B
            el = time.perf_counter() - t0
            if el > {seconds}: break
        q.put((step, done, pos, el))
if __name__ == "__main__":
    ctx = mp.get_context("spawn")
    n = {procs}
    bar = ctx.Barrier(n, timeout=300); q = ctx.Queue()
    ps = [ctx.Process(target=work, args=(i, n, bar, q)) for i in range(n)]
    for p in ps: p.start()
    res = [q.get(timeout={seconds} * 4 + 300) for _ in range(n * {steps})]
    for p in ps: p.join()
    print(json.dumps(res))
"""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    # spawned children import the script's functions by file, so it runs from a file
    with tempfile.NamedTemporaryFile("w", suffix=".py", delete=False) as f:
        f.write(code)
        script = f.name
    try:
        out = subprocess.run([sys.executable, script], capture_output=True, text=True, env=env,
                             timeout=(seconds + 60) * steps + 700)
    finally:
        os.unlink(script)
    if out.returncode != 0:
        raise RuntimeError("all-core oracle timing failed: " + out.stderr[-500:])
    res = json.loads(out.stdout.strip().splitlines()[-1])
    per = []
    for st in range(steps):
        rs = [r for r in res if r[0] == st]
        per.append((sum(r[1] for r in rs), sum(r[2] for r in rs), max(r[3] for r in rs)))
    return per, procs


def cpu_baseline(name, seconds):
    """The float64 oracle on all host cores (one process per core, whole
    requests), with the single-core figure beside it."""
    (req1, pos1, el1), = oracle_timing(name, 0, 0, 1, seconds / 2)
    ((req, pos, el),), n = oracle_timing_all_cores(name, seconds / 2)
    return {"value": pos / el, "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": f"{req} whole requests of {name} (draft + verify, float64 numpy) on {n} "
                      f"single-threaded processes in {el:.1f} s; host cpus={os.cpu_count()}",
            "one_core": {"value": pos1 / el1, "unit": UNIT, "cores": 1,
                         "sample": f"{req1} whole requests in {el1:.1f} s, 1 thread"}}


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return
    from speculative_decoding_draft_04_gb300 import workloads as W
    per_step = min(20.0, max(0.5, 120.0 / max(1, args.steps + args.warmup)))
    # warm-up steps (untimed) then the timed steps, in one set of processes
    samples, ncores = oracle_timing_all_cores(args.config, per_step, steps=args.warmup + args.steps)
    samples = samples[args.warmup:]
    req = sum(x[0] for x in samples)
    pos = sum(x[1] for x in samples)
    el = sum(x[2] for x in samples)
    v = pos / el
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.config + ": " + W.CONFIG_DESCRIPTIONS[args.config],
                       "step": f"a bounded sample of about {per_step:.1f} s of whole requests"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": ncores, "kind": "oracle",
                             "sample": f"{req} whole requests over {args.steps} steps in {el:.1f} s "
                                       f"on {ncores} single-threaded processes; host cpus={os.cpu_count()}"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl")

    from speculative_decoding_draft_04_gb300 import _lib, build, engine
    from speculative_decoding_draft_04_gb300 import workloads as W
    build.build()
    w = W.make_workload(W.config(args.config), trial=rank)
    d = engine.DeviceWorkload.from_workload(w, dev)
    bufs = engine.Buffers.for_workload(d, dev)
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # The cycle's launches (3 memsets, the cooperative draft, 7 verification
    # kernels) are captured once into a CUDA graph and replayed: the calls
    # never synchronize or allocate, so the same calls serve both ways.
    graph, launch_mode = None, "eager"
    if not args.eager:
        try:
            side = torch.cuda.Stream(dev)
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                engine.cycle(d, bufs, side)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                engine.cycle(d, bufs, side)
            torch.cuda.synchronize()
            graph, launch_mode = g, "cuda graph (one captured cycle, replayed)"
        except Exception as exc:          # capture refused: time the eager launches
            launch_mode = f"eager (graph capture failed: {str(exc)[:80]})"

    def step():
        if graph is not None:
            graph.replay()
        else:
            engine.cycle(d, bufs, stream)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize()

    # ---- timed region: K cycles, L2 flushed between cycles (outside the events).
    # Clocks are sampled every 200 ms over the timed region, repeated untimed
    # until the sampler has seen at least 5 samples under load.
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            flush.zero_()
            evs[i][0].record(stream)
            step()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        t_end = time.time() + 1.2
        while time.time() < t_end:
            flush.zero_()
            step()
            torch.cuda.synchronize()
    barrier()
    times = [a.elapsed_time(b) for a, b in evs]
    ms = float(sum(times) / len(times))
    clocks = clk.summary()
    # the same cycles back to back without the flush (warm L2), for context
    wev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for i in range(args.steps):
        wev[i][0].record(stream)
        step()
        wev[i][1].record(stream)
    torch.cuda.synchronize()
    warm_ms = float(sum(a.elapsed_time(b) for a, b in wev) / args.steps)

    # ---- second timed pass with per-kernel events (roofline of the top kernel)
    _lib.spec_profile_enable(True)
    _lib.spec_profile_read()
    for i in range(args.steps):
        flush.zero_()
        engine.cycle(d, bufs, stream)
    torch.cuda.synchronize()
    prof = _lib.spec_profile_read()
    _lib.spec_profile_enable(False)

    # ---- end to end through spec_cycle_host: the step's inputs start in
    # page-locked host memory; the library copies them in (the target logits
    # on a second stream, overlapping the draft), runs the cycle and copies
    # accept_len / out_tokens back
    hs = engine.HostStep.like(d)
    copy_stream = torch.cuda.Stream(device=dev)
    h2d, d2h = hs.h2d_bytes(), hs.d2h_bytes()
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    for _ in range(2):
        engine.cycle_host(d, bufs, hs, stream, copy_stream)
    torch.cuda.synchronize()
    barrier()
    for i in range(args.steps):
        flush.zero_()
        e2e_ev[i][0].record(stream)
        engine.cycle_host(d, bufs, hs, stream, copy_stream)
        e2e_ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = float(sum(a.elapsed_time(b) for a, b in e2e_ev) / args.steps)
    # the same host-to-device copies alone (U, then the target logits, one
    # stream): the link rate, and how much of the copy the overlap hides
    link_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    big = (hs.U.numel() * hs.U.element_size() + hs.target.numel() * hs.target.element_size())
    with torch.cuda.stream(stream):
        for _ in range(2):
            d.U.copy_(hs.U, non_blocking=True)
            d.target.copy_(hs.target, non_blocking=True)
        torch.cuda.synchronize()
        flush.zero_()
        link_ev[0].record(stream)
        for _ in range(args.steps):
            d.U.copy_(hs.U, non_blocking=True)
            d.target.copy_(hs.target, non_blocking=True)
        link_ev[1].record(stream)
    torch.cuda.synchronize()
    link_ms = float(link_ev[0].elapsed_time(link_ev[1]) / args.steps)

    draft_prof = tuple(a + b for a, b in zip(prof.get("draft_persistent", (0.0, 0)),
                                               prof.get("draft_slice", (0.0, 0))))
    op = operating_point(d, bufs, draft_prof, args.steps) \
        if rank == 0 else None
    sched = rnn = tree = None
    others = {}
    if rank == 0 and world == 1:
        for name in [c for c in args.other_configs.split(",") if c and c != args.config]:
            others[name] = config_pass(name, args, flush, dev)
    if not args.no_extras:
        sched = scheduled_pass(args, w, d, bufs, stream, flush, rank, dev)
        rnn = rnn_pass(args, w, d, bufs, stream, flush, rank, dev)
        tree = tree_pass(args, w, d, flush, rank, dev)

    positions = int(w.verify_len.sum())
    if world > 1:
        t = torch.tensor([ms, e2e_ms, float(positions)], device=dev)
        mx = t.clone()
        torch.distributed.all_reduce(mx, op=torch.distributed.ReduceOp.MAX)
        tot = t.clone()
        torch.distributed.all_reduce(tot, op=torch.distributed.ReduceOp.SUM)
        ms_all, e2e_all, pos_all = float(mx[0]), float(mx[1]), float(tot[2])
    else:
        ms_all, e2e_all, pos_all = ms, e2e_ms, float(positions)

    if rank == 0:
        hbm_peak, _, peak_src = measured_peaks()
        draft_b, verify_b, per_stage = algorithmic_bytes(w)
        cyc_gbs = (draft_b + verify_b) / (ms * 1e-3) / 1e9
        tot_ms = sum(v[0] for v in prof.values())
        top = max(per_stage, key=lambda k: prof.get(k, (0.0, 0))[0])
        t_ms, n_l = prof[top]
        avg_ms = t_ms / max(n_l, 1)
        ach = per_stage[top] / (avg_ms * 1e-3) / 1e9
        launches = sum(v[1] for v in prof.values()) // max(args.steps, 1)
        line = {
            "metric": METRIC, "value": pos_all / (ms_all * 1e-3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_all,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": args.config + ": " + W.CONFIG_DESCRIPTIONS[args.config],
                       "l2": f"flushed between steps ({flush.numel() >> 20} MiB write, outside the events)",
                       "launch": launch_mode,
                       "positions_per_step": positions},
            "warm_l2": {"ms_per_step": warm_ms, "value": float(positions) / (warm_ms * 1e-3),
                        "note": "the same cycles back to back, no L2 flush (context only)"},
            "hbm": {"cycle_algorithmic_bytes": draft_b + verify_b, "cycle_gbs": cyc_gbs,
                    "frac_of_8TBs": cyc_gbs / NOMINAL_HBM_GBS,
                    "frac_of_measured": cyc_gbs / hbm_peak},
            "roofline": {"kernel": top, "bound": "hbm", "achieved": ach, "peak": hbm_peak,
                         "peak_source": peak_src, "unit": "GB/s", "frac": ach / hbm_peak,
                         "traffic": recorded_traffic(top, args.config),
                         "algorithmic_bytes_per_launch": per_stage[top],
                         "avg_launch_ms": avg_ms, "share_of_step": t_ms / tot_ms if tot_ms else None},
            "stages_ms_per_step": {k: v[0] / args.steps for k, v in prof.items() if v[1]},
            "e2e": {"value": pos_all / (e2e_all * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_all,
                    "call": "spec_cycle_host (pinned host inputs and results; the target "
                            "logits copied on a second stream during the draft)",
                    "link": {"h2d_ms_alone": link_ms, "h2d_gbs": big / (link_ms * 1e6),
                             "bytes": big,
                             "hidden_ms": link_ms + ms - e2e_ms,
                             "note": "U and target logits copied alone, back to back on one "
                                     "stream; hidden_ms = copy alone + device cycle - e2e"}},
            "gpu_launches": int(launches * args.steps),
            "clocks": clocks,
        }
        if others:
            line["other_configs"] = others
        if not args.no_extras:
            line["scheduled_cycle"] = sched
            line["rnn_cycle"] = rnn
            line["tree_cycle"] = tree
        line["operating_point"] = op
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args.config, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
