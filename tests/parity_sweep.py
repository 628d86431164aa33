"""Parity sweep of the token parity gate at scale.

The gate: on every workload, every request whose GPU tokens or accept length
differ from the float64 oracle must have a consumed uniform within 1e-6 of a
decision boundary, and such mismatched requests must be fewer than 0.01% of
all requests.  Resolving 0.01% needs at least 10^4 requests per workload,
so this runs many seeded trials of each at full size, in two halves:

  gpu      (on the GPU machine)  for each trial: draw the seeded workload
           (workloads.make_workload, a thread pool), run one cycle through the
           C ABI (spec_markov_draft + spec_verify), keep the outputs and a
           checksum of every input array; one .npz per workload.
  compare  (any machine, CPU only)  for each saved trial: draw the same
           workload again, check the checksums (so both sides saw identical
           inputs), run the oracle on every request (a process pool) and
           compare request by request as the parity tests do; write the
           counts per workload (requests, near-boundary requests, mismatched,
           mismatched away from every boundary, largest errors of q(x), lse,
           alpha and p(x), re-decisions) to a JSON record.

    python tests/parity_sweep.py gpu --config C2 --trials 0:1000 --out DIR
    python tests/parity_sweep.py compare --dir DIR --record FILE [--workers 8]

Test infrastructure: the compare half runs the oracle; nothing in the
package imports this file.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
for p in (ROOT, HERE):
    if p not in sys.path:
        sys.path.insert(0, p)

INPUT_FIELDS = ("target", "U", "W1", "W2", "anchor", "temperature", "verify_len", "u_draft",
                "u_accept", "u_final")
OUTPUT_FIELDS = ("draft_tokens", "q_tok", "lse_q", "accept_len", "out_tokens", "alpha", "p_tok")


def parse_trials(s: str) -> list[int]:
    a, b = s.split(":")
    return list(range(int(a), int(b)))


def checksum(w) -> str:
    h = hashlib.blake2b(digest_size=16)
    for f in INPUT_FIELDS:
        a = np.ascontiguousarray(getattr(w, f))
        h.update(f.encode())
        h.update(str(a.dtype).encode())
        h.update(str(a.shape).encode())
        h.update(a.tobytes())
    return h.hexdigest()


# ----------------------------------------------------------------------------- GPU half

def run_gpu(args) -> None:
    import torch

    from speculative_decoding_draft_04_gb300 import _lib, build, engine
    from speculative_decoding_draft_04_gb300 import workloads as W

    build.build()
    _lib.lib()
    _lib.spec_set_option(_lib.SPEC_OPT_FORCE_SIMT, 0)
    _lib.spec_set_option(_lib.SPEC_OPT_EPS_SCALE, 1.0)
    _lib.spec_set_option(_lib.SPEC_OPT_BIAS_PATH, 2)
    trials = parse_trials(args.trials)
    spec = W.config(args.config)

    def draw(trial):
        w = W.make_workload(spec, trial=trial)
        return trial, w, checksum(w)

    outs = {f: [] for f in OUTPUT_FIELDS}
    dst, vst, sums, done = [], [], [], []
    bufs = None
    t0 = time.time()
    with cf.ThreadPoolExecutor(max_workers=args.threads) as ex:
        pending = {}
        it = iter(trials)
        for tr in [next(it, None) for _ in range(args.threads + 2)]:
            if tr is not None:
                pending[tr] = ex.submit(draw, tr)
        for tr in trials:
            trial, w, cs = pending.pop(tr).result()
            nxt = next(it, None)
            if nxt is not None:
                pending[nxt] = ex.submit(draw, nxt)
            d = engine.DeviceWorkload.from_workload(w, "cuda")
            if bufs is None:
                bufs = engine.Buffers.for_workload(d, "cuda")
            engine.cycle(d, bufs)
            torch.cuda.synchronize()
            for f in OUTPUT_FIELDS:
                outs[f].append(getattr(bufs, f).cpu().numpy().copy())
            dst.append(engine.status_words(bufs.dstatus))
            vst.append(engine.status_words(bufs.vstatus))
            sums.append(cs)
            done.append(trial)
            del d, w
    os.makedirs(args.out, exist_ok=True)
    path = os.path.join(args.out, f"sweep_{args.config}_{trials[0]}_{trials[-1] + 1}.npz")
    np.savez_compressed(path, trials=np.array(done), checksums=np.array(sums),
                        dstatus=np.array(dst, np.int64), vstatus=np.array(vst, np.int64),
                        **{f: np.stack(v) for f, v in outs.items()})
    print(json.dumps({"config": args.config, "trials": len(done), "seconds": time.time() - t0,
                      "file": path}), flush=True)


# ----------------------------------------------------------------------------- CPU half

def _compare_one(task):
    name, trial, cs, g_arrays, dstatus, vstatus = task
    from parity import GpuResult, compare, oracle_cycle
    from speculative_decoding_draft_04_gb300 import workloads as W

    w = W.make_workload(W.config(name), trial=trial)
    if checksum(w) != cs:
        return dict(trial=trial, checksum_mismatch=True)
    g = GpuResult(*[g_arrays[f] for f in OUTPUT_FIELDS], list(dstatus), list(vstatus))
    res = oracle_cycle(w)
    rep = compare(w, g, res)
    near = [b for b in range(w.B) if res.row_dmin(b) < 1e-6]
    return dict(trial=trial, checksum_mismatch=False, rows=rep.rows, near=len(near),
                mismatched=[int(b) for b in rep.mismatched],
                far=[int(b) for b in rep.far_mismatched],
                q_err=rep.max_q_err, lse_err=rep.max_lse_err, alpha_err=rep.max_alpha_err,
                ptok_err=rep.max_ptok_err, redecided=int(dstatus[1]) + int(vstatus[1]),
                positions=int(w.verify_len.sum()))


def run_compare(args) -> None:
    files = sorted(f for f in os.listdir(args.dir) if f.startswith("sweep_") and f.endswith(".npz"))
    record = {}
    if os.path.exists(args.record) and not args.fresh:
        with open(args.record) as f:
            record = json.load(f)
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    for fn in files:
        name = fn.split("_")[1]
        z = np.load(os.path.join(args.dir, fn))
        tasks = []
        for i, trial in enumerate(z["trials"]):
            g_arrays = {f: z[f][i] for f in OUTPUT_FIELDS}
            tasks.append((name, int(trial), str(z["checksums"][i]), g_arrays, z["dstatus"][i],
                          z["vstatus"][i]))
        t0 = time.time()
        acc = dict(trials=0, rows=0, near=0, mismatched=0, far=0, checksum_mismatch=0,
                   q_err=0.0, lse_err=0.0, alpha_err=0.0, ptok_err=0.0, redecided=0,
                   positions=0, mismatched_rows=[], far_rows=[])
        with cf.ProcessPoolExecutor(max_workers=args.workers, mp_context=ctx) as ex:
            for r in ex.map(_compare_one, tasks, chunksize=1):
                if r["checksum_mismatch"]:
                    acc["checksum_mismatch"] += 1
                    continue
                acc["trials"] += 1
                for k in ("rows", "near", "redecided", "positions"):
                    acc[k] += r[k]
                acc["mismatched"] += len(r["mismatched"])
                acc["far"] += len(r["far"])
                acc["mismatched_rows"] += [[r["trial"], b] for b in r["mismatched"]]
                acc["far_rows"] += [[r["trial"], b] for b in r["far"]]
                for k in ("q_err", "lse_err", "alpha_err", "ptok_err"):
                    acc[k] = max(acc[k], r[k])
        acc["mismatch_rate"] = acc["mismatched"] / acc["rows"] if acc["rows"] else None
        acc["gate_met"] = bool(acc["rows"] and acc["far"] == 0 and acc["mismatched"] < 1e-4 * acc["rows"]
                               and acc["checksum_mismatch"] == 0
                               and max(acc["q_err"], acc["lse_err"], acc["alpha_err"], acc["ptok_err"]) <= 1e-5)
        acc["trial_range"] = [int(z["trials"][0]), int(z["trials"][-1]) + 1]
        acc["compare_seconds"] = round(time.time() - t0, 1)
        key = f"{name}:{acc['trial_range'][0]}-{acc['trial_range'][1]}"
        record[key] = acc
        print(key, json.dumps({k: v for k, v in acc.items() if not k.endswith("_rows")}), flush=True)
        with open(args.record, "w") as f:
            json.dump(record, f, indent=1, sort_keys=True)


def main() -> None:
    ap = argparse.ArgumentParser()
    sub = ap.add_subparsers(dest="cmd", required=True)
    g = sub.add_parser("gpu")
    g.add_argument("--config", required=True)
    g.add_argument("--trials", required=True, help="first:last+1")
    g.add_argument("--out", required=True)
    g.add_argument("--threads", type=int, default=12)
    c = sub.add_parser("compare")
    c.add_argument("--dir", required=True)
    c.add_argument("--record", required=True)
    c.add_argument("--workers", type=int, default=os.cpu_count() or 4)
    c.add_argument("--fresh", action="store_true")
    args = ap.parse_args()
    if args.cmd == "gpu":
        run_gpu(args)
    else:
        run_compare(args)


if __name__ == "__main__":
    main()
