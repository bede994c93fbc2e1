"""Benchmark of the fused verify step on GB300.

Default workload: the Qwen3.8-27B-shaped hybrid decoder (64 layers, 48 Gated
DeltaNet + 16 gated attention, hidden 5120, FFN 17408, vocab 248,320, Q4
weights ~ N(0, 0.02)), one sequence with 4,096 cached tokens in an fp16 KV
pool, T = 1 row per step. Inputs are seeded synthetic data.

Prints ONE JSON line. `value` = verified rows/s from device time of the single
cooperative launch per step (inputs resident in HBM; the 14.4 GB weight
stream is larger than L2, so no flush is needed); `e2e` = the same metric
through the public call mk_step with host row arrays and the host readback.

  python bench.py [--gpus N --steps K --warmup W --workload NAME --impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified rows/s & step µs on 1×GB300; achieved HBM GB/s vs ~8 TB/s peak"
UNIT = "rows/s"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def measured_traffic(algorithmic):
    """DRAM bytes per launch from the committed ncu capture (profiles/
    mk_persistent_traffic.json), scaled to this workload by the measured
    traffic/algorithmic ratio; None when the kernel sources changed since the
    capture (the counters would no longer describe this kernel)."""
    import glob
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "mk_persistent_traffic.json")) as f:
            rec = json.load(f)
        srcs = sorted(glob.glob(os.path.join(ROOT, "speculative_decode_persistent_gb300", "csrc", "*.cu")) +
                      glob.glob(os.path.join(ROOT, "speculative_decode_persistent_gb300", "csrc", "*.cuh")) +
                      [os.path.join(ROOT, "include", "mk.h")])
        h = hashlib.sha256()
        for fn in srcs:
            with open(fn, "rb") as f:
                h.update(f.read())
        if h.hexdigest() != rec["kernel_sources_sha256"]:
            return None
        return algorithmic * rec["traffic_over_algorithmic"]
    except Exception:
        return None


def algorithmic_bytes(model, kv_q8, seqs, n_draft=0):
    """Bytes the step must move: every streamed weight once, the embedding rows
    it gathers, each sequence's cached K/V once per attention layer plus the
    new rows, and the recurrent state read once and written once. With an MTP
    head, each of its n_draft sequential passes streams the head's weights and
    the lm_head rows of the draft vocabulary again, gathers embedding rows,
    and reads the head's KV layer."""
    from gen.configs import model_dims, tensor_inventory
    d = model_dims(model)
    R = sum(T for _c, T in seqs)
    H = model["hidden"]
    passes = n_draft if model.get("has_mtp") else 0
    w = 0.0
    for name, _tid, kind, shape in tensor_inventory(model):
        if kind != "q4":
            continue
        if name == "embed" and not model["tied"]:
            continue
        w += shape[0] * shape[1] * 0.5625 * (passes if name.startswith("mtp.") else 1)
    w += R * H * 0.5625
    w += passes * (model.get("draft_vocab", 0) * H + R * H) * 0.5625
    per_layer = model["hkv"] * model["dh"] * 2 * ((1 + 2 / 32) if kv_q8 else 2)
    per_tok = d["n_fa"] * per_layer
    kv = sum(c for c, _T in seqs) * per_tok + R * per_tok
    kv += passes * (sum(c for c, _T in seqs) + R) * per_layer
    nseq = len(seqs)
    state = nseq * 2 * d["n_gdn"] * model["hv"] * model["dv"] * model["dk"] * 4
    conv = nseq * 2 * d["n_gdn"] * (model["conv_w"] - 1) * d["conv_ch"] * 4
    return dict(weights=w, kv=kv, state=state + conv, total=w + kv + state + conv)


class Clocks:
    """nvidia-smi sampling while the timed region runs."""

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 7:
                self.samples.append(parts)

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4) if s[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v, device=None):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_oracle_sample(workload, budget_s=20.0):
    """The fp64 oracle as it stands, on this host's cores: full verify steps
    of the same workload (same seeds) until about budget_s of CPU time, or a
    single step if one step is longer. Returns rows/s and the sample."""
    from gen.workload import Workload
    from oracle import oracle as orc
    nthreads = os.cpu_count() or 1
    wl = Workload(workload, nthreads=nthreads)
    n_draft = int(wl.spec.get("n_draft", 0)) if wl.model.get("has_mtp") else 0
    o = orc.Oracle(wl.model, wl.weights, wl.pool, wl.kv_q8, wl.n_pages, wl.max_seqs, nthreads=nthreads,
                   n_draft=n_draft)
    for s, (cached, _T) in enumerate(wl.seqs):
        o.seq_set(s, cached, wl.tables[s], *wl.states[s])
    tok, pos, sid = wl.rows()
    steps, rows, el = 0, 0, 0.0
    while True:
        if steps:  # re-install the pre-step state (not timed)
            for s, (cached, _T) in enumerate(wl.seqs):
                o.seq_set(s, cached, wl.tables[s], *wl.states[s])
        t0 = time.perf_counter()
        o.step(tok, pos, sid, want_logits=False)
        el += time.perf_counter() - t0
        steps += 1
        rows += len(tok)
        if el >= budget_s or steps >= 1000:
            break
    return dict(value=rows / el, unit=UNIT, cores=nthreads, kind="oracle",
                sample=f"{steps} full fp64 verify step(s) of {workload} ({rows} rows) in {el:.1f} s")


def run_reference(args, world, rank):
    if rank != 0:
        return
    cb = cpu_oracle_sample(args.workload, budget_s=args.ref_budget)
    ms = 1000.0 * (1.0 / cb["value"]) * len_rows(args.workload)
    line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload}, "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def layer_override(args):
    """--layers N: the same widths with only the first N layers (profiling
    stand-in that fits an ncu capture; never a headline number)."""
    if not args.layers:
        return None
    from gen.configs import WORKLOADS
    m = dict(WORKLOADS[args.workload]["model"])
    m["kinds"] = list(m["kinds"])[: args.layers]
    m["n_layers"] = args.layers
    return dict(model=m)


def len_rows(workload):
    from gen.configs import WORKLOADS
    return sum(T for _c, T in WORKLOADS[workload]["seqs"])


def run_ours(args, world, rank, local):
    import torch
    from gen.workload import Workload
    from speculative_decode_persistent_gb300 import mk

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    t_setup = time.perf_counter()
    wl = Workload(args.workload, nthreads=os.cpu_count(), overrides=layer_override(args))
    n_draft = int(wl.spec.get("n_draft", 0)) if wl.model.get("has_mtp") else 0
    eng = mk.Engine(wl.model, wl.weights, wl.kv_q8, wl.n_pages, max_seqs=wl.max_seqs, device=f"cuda:{local}",
                    n_draft=n_draft)
    eng.load_pool(wl.pool)
    for s, (cached, _T) in enumerate(wl.seqs):
        eng.seq_set(s, cached, wl.tables[s], *wl.states[s])
    del wl.weights
    setup_s = time.perf_counter() - t_setup
    rng = np.random.default_rng(2)
    tok, pos, sid = wl.rows([list(rng.integers(0, wl.model["vocab"], T - 1)) for _c, T in wl.seqs])
    R = len(tok)
    stream = eng.stream

    # ---- device time: repeated launches of one prepared step (each launch
    # redoes the whole step; the step is idempotent until it is finished)
    eng.prepare(tok, pos, sid)
    for _ in range(args.warmup):
        eng.launch()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    per_launch = []
    barrier(world)
    torch.cuda.synchronize(dev)
    with Clocks(local) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            eng.launch()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    total_ms = e0.elapsed_time(e1)
    barrier(world)
    # per-launch durations (library events around each launch), for the roofline
    for _ in range(min(args.steps, 10)):
        eng.launch()
        torch.cuda.synchronize(dev)
        per_launch.append(eng.last_launch_ms())
    out_t, out_c = eng.finish()
    total_ms = max_over_ranks(world, total_ms, dev)
    ms = total_ms / args.steps

    # ---- end to end through mk_step (host rows in, accepted tokens out)
    def drafts():
        return eng.last_drafts(len(wl.seqs)) if n_draft else None

    for _ in range(2):
        out_t, out_c = eng.step(*next_rows(wl, tok, pos, sid, out_t, out_c, rng, drafts()))
        tok, pos, sid = last_rows
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    accepted = 0
    h2d = d2h = 0
    for _ in range(args.e2e_steps):
        rows = next_rows(wl, tok, pos, sid, out_t, out_c, rng, drafts())
        out_t, out_c = eng.step(*rows)
        tok, pos, sid = last_rows
        accepted += int(out_c.sum())
        hb, db = eng.io_bytes()
        h2d += hb + 3 * 4 * R
        d2h += db
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(world, e2e_s, dev)

    ab = algorithmic_bytes(wl.model, wl.kv_q8, wl.seqs, n_draft)
    peak, peak_kind = peaks()
    launch_ms = statistics.median(per_launch) if per_launch else ms
    achieved = ab["total"] / (launch_ms * 1e-3) / 1e9
    if rank == 0:
        line = {
            "metric": METRIC, "value": world * R / (ms * 1e-3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "q4-weights/f16-split-mma/f32",
            "data": "synthetic (seeded random-init weights and caches)",
            "config": {"workload": args.workload if not args.layers else f"{args.workload} (first {args.layers} layers: profiling stand-in)",
                       "rows_per_step": R, "sequences": len(wl.seqs),
                       "cached_tokens": [c for c, _T in wl.seqs], "kv": "q8" if wl.kv_q8 else "fp16",
                       "mtp": ({"n_draft": n_draft, "draft_vocab": wl.model["draft_vocab"],
                                "drafts": "next step's drafts are the head's (e2e loop)"} if n_draft else None),
                       "l2": "inputs larger than L2: 14.4 GB of weights streamed per step",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "step_us": ms * 1e3,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind, "traffic": measured_traffic(ab["total"]),
                         "algorithmic_bytes": ab["total"], "bytes_breakdown": ab,
                         "kernel": "mk_persistent (whole step, one cooperative launch)",
                         "frac_of_8TBs": achieved / 8000.0},
            "e2e": {"value": world * R * args.e2e_steps / e2e_s, "unit": UNIT,
                    "h2d_bytes_per_step": h2d // args.e2e_steps, "d2h_bytes_per_step": d2h // args.e2e_steps,
                    "accepted_tokens_per_s": accepted / e2e_s, "steps": args.e2e_steps},
            "gpu_launches": args.steps,
            "clocks": clk.summary(),
            "setup_s": setup_s,
        }
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_oracle_sample(args.workload, budget_s=args.ref_budget)
        print(json.dumps(line))
    eng.close()


last_rows = None


def next_rows(wl, tok, pos, sid, out_t, out_c, rng, drafts=None):
    """Next verify step of a greedy decode loop: each sequence's first row is
    its bonus token at the new length, the other rows the MTP head's drafts of
    the step before (drafts [sequence][n_draft]) or random tokens."""
    global last_rows
    new_tok, new_pos, new_sid = [], [], []
    at = 0
    for i, (_c, T) in enumerate(wl.seqs):
        c = int(out_c[i])
        bonus = int(out_t[at + c - 1])
        at += c
        base = int(np.asarray(pos)[np.asarray(sid) == i][0]) + c
        d = [] if drafts is None else [int(x) for x in drafts[i][: T - 1]]
        d += [int(x) for x in rng.integers(0, wl.model["vocab"], T - 1 - len(d))]
        new_tok += [bonus] + d
        new_pos += list(range(base, base + T))
        new_sid += [i] * T
    last_rows = (np.array(new_tok, np.int32), np.array(new_pos, np.int32), np.array(new_sid, np.int32))
    return last_rows


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--workload", default="qwen27-t1-4k-fp16")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-budget", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="profiling stand-in: keep only the first N layers")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
