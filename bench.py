"""Benchmark of the fused verify step on GB300.

Headline workload: the Qwen3.8-27B-shaped hybrid decoder (64 layers, 48 Gated
DeltaNet + 16 gated attention, hidden 5120, FFN 17408, vocab 248,320, Q4
weights ~ N(0, 0.02)) with 4 sequences x T = 3 rows per step, 23,000 cached
tokens each in a shared q8 paged KV pool (8,448 pages, shuffled page tables).
The same run also times the single-stream T = 1 and T = 5 steps over a 4,096-token
fp16 cache (per_workload), and reports T5 / T1. Inputs are seeded synthetic data.

Prints ONE JSON line. `value` = verified rows/s from device time of the single
cooperative launch per step (inputs resident in HBM; the 14.4 GB weight
stream is larger than L2, so no flush is needed); `e2e` = the same metric
through the public call mk_step with host row arrays and the host readback.
Drafts for T > 1 follow the engine's own greedy continuation (computed with
one-row steps before timing) with a seeded mismatch position per sequence
and step, so the accepted length is uniform over 0..T-1.

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


def workload_config(workload, layers=0):
    """The `config` object of a bench line (the same for both arms)."""
    from gen.configs import WORKLOADS
    w = WORKLOADS[workload]
    seqs = w["seqs"]
    m = w["model"]
    name = workload if not layers else f"{workload} (first {layers} layers: profiling stand-in)"
    return {"workload": name, "rows_per_step": sum(T for _c, T in seqs), "sequences": len(seqs),
            "cached_tokens": [c for c, _T in seqs], "kv": "q8" if w["kv_q8"] else "fp16",
            "mtp": ({"n_draft": w.get("n_draft"), "draft_vocab": m.get("draft_vocab")} if m.get("has_mtp") else None),
            "drafts": "greedy continuation, mismatch position uniform over 0..T-1 per sequence and step",
            "l2": "inputs larger than L2: 14.4 GB of weights streamed per step",
            "parallelism": "single GPU"}


def cpu_oracle_sample(workload, budget_s=20.0, steps=None, warmup=0):
    """The fp64 oracle as it stands, on this host's cores, over a bounded
    sample of the workload: one-row passes of its first sequence (at that
    sequence's cached context), `steps` of them timed after `warmup` untimed
    ones, or as many as fit in about budget_s when steps is None. Returns
    rows/s and the sample."""
    from gen.workload import Workload
    from oracle import oracle as orc
    nthreads = os.cpu_count() or 1
    wl = Workload(workload, nthreads=nthreads)
    n_draft = int(wl.spec.get("n_draft", 0)) if wl.model.get("has_mtp") else 0
    o = orc.Oracle(wl.model, wl.weights, wl.pool, wl.kv_q8, wl.n_pages, wl.max_seqs, nthreads=nthreads,
                   n_draft=n_draft)
    cached = wl.seqs[0][0]
    tok = [int(wl.first_tokens[0])]

    def one():
        o.seq_set(0, cached, wl.tables[0], *wl.states[0])  # the pre-step state (not timed)
        t0 = time.perf_counter()
        o.step(tok, [cached], [0], want_logits=False)
        return time.perf_counter() - t0

    for _ in range(warmup):
        one()
    n, el = 0, 0.0
    while True:
        el += one()
        n += 1
        if (steps is not None and n >= steps) or (steps is None and (el >= budget_s or n >= 1000)):
            break
    return dict(value=n / el, unit=UNIT, cores=nthreads, kind="oracle", steps=n, seconds=el,
                sample=f"{n} one-row fp64 passes of {workload}'s first sequence ({cached} cached tokens)"
                       f" in {el:.1f} s, after {warmup} untimed")


def run_reference(args, world, rank):
    if rank != 0:
        return
    cb = cpu_oracle_sample(args.workload, steps=args.steps, warmup=args.warmup)
    ms = 1000.0 * cb["seconds"] / cb["steps"]
    line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": 1,
            "steps": cb["steps"], "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args.workload),
            "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")},
            "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def layer_override(workload, layers):
    """--layers N: the same widths with only the first N layers (profiling
    stand-in that fits an ncu capture; never a headline number)."""
    if not layers:
        return None
    from gen.configs import WORKLOADS
    m = dict(WORKLOADS[workload]["model"])
    m["kinds"] = list(m["kinds"])[:layers]
    m["n_layers"] = layers
    return dict(model=m)


def greedy_trajectory(eng, wl, n):
    """The engine's own greedy continuation of every sequence: n one-row steps
    (one row per sequence, all in one launch) from the workload's cached
    state; every sequence is re-installed afterwards."""
    nseq = len(wl.seqs)
    toks = [int(t) for t in wl.first_tokens[:nseq]]
    base = [c for c, _T in wl.seqs]
    traj = [[] for _ in range(nseq)]
    sid = np.arange(nseq, dtype=np.int32)
    for j in range(n):
        out_t, _c = eng.step(np.array(toks, np.int32), np.array([b + j for b in base], np.int32), sid)
        for s in range(nseq):
            toks[s] = int(out_t[s])
            traj[s].append(toks[s])
    for s, (cached, _T) in enumerate(wl.seqs):
        eng.seq_reset(s)
        eng.seq_set(s, cached, wl.tables[s], *wl.states[s])
    return traj


class Drafter:
    """Rows of the next verify step: each sequence's row 0 is the token it
    last emitted, its drafts follow the greedy trajectory up to a seeded
    mismatch position m (uniform over 0..T-1), so m drafts are accepted."""

    def __init__(self, wl, traj, seed):
        self.wl, self.traj = wl, traj
        self.rng = np.random.default_rng(seed)
        self.off = [0] * len(wl.seqs)  # trajectory tokens already emitted
        self.last = [int(t) for t in wl.first_tokens[: len(wl.seqs)]]

    def rows(self):
        V = self.wl.model["vocab"]
        tok, pos, sid = [], [], []
        for s, (cached, T) in enumerate(self.wl.seqs):
            m = int(self.rng.integers(0, T))
            o, tr = self.off[s], self.traj[s]
            d = [tr[min(o + i, len(tr) - 1)] for i in range(T - 1)]
            if m < T - 1:
                d[m] = (d[m] + 1) % V
            tok += [self.last[s]] + d
            pos += list(range(cached + o, cached + o + T))
            sid += [s] * T
        return np.array(tok, np.int32), np.array(pos, np.int32), np.array(sid, np.int32)

    def advance(self, out_t, out_c):
        at = 0
        for s in range(len(self.wl.seqs)):
            c = int(out_c[s])
            self.off[s] += c
            self.last[s] = int(out_t[at + c - 1])
            at += c


def measure(args, eng, wl, workload, world, dev, torch, layers=0):
    """Device time, per-launch time, clocks and end-to-end rate of one
    workload on an engine whose sequences hold the workload's cached state."""
    from gen.configs import WORKLOADS
    n_draft = int(wl.spec.get("n_draft", 0)) if wl.model.get("has_mtp") else 0
    Tmax = max(T for _c, T in wl.seqs)
    traj = greedy_trajectory(eng, wl, (args.e2e_steps + 3) * Tmax + Tmax) if Tmax > 1 else None
    drafter = Drafter(wl, traj, 2) if traj else None
    if drafter:
        tok, pos, sid = drafter.rows()
    else:
        tok, pos, sid = wl.rows()
    R = len(tok)
    stream = eng.stream
    # ---- device time: repeated launches of one prepared step (each launch
    # redoes the whole step; the step is idempotent until it is finished)
    eng.prepare(tok, pos, sid)
    for _ in range(args.warmup):
        eng.launch()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    with Clocks(dev.index) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            eng.launch()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    total_ms = e0.elapsed_time(e1)
    barrier(world)
    per_launch = []
    for _ in range(min(args.steps, 10)):
        eng.launch()
        torch.cuda.synchronize(dev)
        per_launch.append(eng.last_launch_ms())
    timeline = phase_timeline(eng, wl, dev, torch) if args.timeline and not n_draft else None
    out_t, out_c = eng.finish()
    total_ms = max_over_ranks(world, total_ms, dev)
    ms = total_ms / args.steps
    # ---- end to end through mk_step (host rows in, accepted tokens out)
    for s, (cached, _T) in enumerate(wl.seqs):  # back to the cached state
        eng.seq_reset(s)
        eng.seq_set(s, cached, wl.tables[s], *wl.states[s])
    drafter = Drafter(wl, traj, 3) if traj else None
    rng = np.random.default_rng(5)

    def next_rows(out_t=None, out_c=None):
        if drafter:
            if out_t is not None:
                drafter.advance(out_t, out_c)
            return drafter.rows()
        if out_t is None:
            return wl.rows()
        return plain_next_rows(wl, last_rows_box, out_t, out_c, rng)

    last_rows_box = [wl.rows()]
    rows = next_rows()
    for _ in range(2):
        last_rows_box[0] = rows
        out_t, out_c = eng.step(*rows)
        rows = next_rows(out_t, out_c)
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    accepted = 0
    h2d = d2h = 0
    for _ in range(args.e2e_steps):
        last_rows_box[0] = rows
        out_t, out_c = eng.step(*rows)
        accepted += int(out_c.sum())
        hb, db = eng.io_bytes()
        h2d += hb + 3 * 4 * R
        d2h += db
        rows = next_rows(out_t, out_c)
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(world, e2e_s, dev)
    for s, (cached, _T) in enumerate(wl.seqs):  # leave the engine at the cached state
        eng.seq_reset(s)
        eng.seq_set(s, cached, wl.tables[s], *wl.states[s])
    ab = algorithmic_bytes(wl.model, wl.kv_q8, wl.seqs, n_draft)
    peak, peak_kind = peaks()
    launch_ms = statistics.median(per_launch) if per_launch else ms
    achieved = ab["total"] / (launch_ms * 1e-3) / 1e9
    return {
        "workload": workload, "value": world * R / (ms * 1e-3), "ms_per_step": ms, "step_us": ms * 1e3,
        "rows_per_step": R,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": measured_traffic(ab["total"]) if not layers else None,
                     "algorithmic_bytes": ab["total"], "bytes_breakdown": ab,
                     "launch_ms_median": launch_ms,
                     "kernel": "mk_persistent (whole step, one cooperative launch)",
                     "frac_of_8TBs": achieved / 8000.0},
        "e2e": {"value": world * R * args.e2e_steps / e2e_s, "unit": UNIT,
                "h2d_bytes_per_step": h2d // args.e2e_steps, "d2h_bytes_per_step": d2h // args.e2e_steps,
                "accepted_tokens_per_s": world * accepted / e2e_s,
                "accepted_per_step": accepted / args.e2e_steps, "steps": args.e2e_steps},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
        **({"timeline_us": timeline} if timeline else {}),
    }


def phase_timeline(eng, wl, dev, torch, launches=5):
    """Per-phase time of the prepared step (block 0's %globaltimer stamp at
    the start and at the end of every phase up to lm_head, through
    mk_debug_timeline), averaged over a few launches run after the timed ones:
    embed, then per layer the input projections, the mixer, o_proj, gate/up
    and down, then lm_head (GEMM and argmax; the verify phase is not stamped)."""
    nl = wl.model["n_layers"]
    stamps = torch.zeros(5 * nl + 8, dtype=torch.int64, device=dev)
    eng.timeline(stamps)
    acc = None
    for _ in range(launches):
        eng.launch()
        torch.cuda.synchronize(dev)
        d = np.diff(stamps.cpu().numpy()[: 5 * nl + 3].astype(np.float64)) / 1e3
        acc = d if acc is None else acc + d
    eng.timeline(None)
    names = ["embed"] + [f"L{l}.{p}" for l in range(nl) for p in ("in", "mix", "o", "gu", "down")] + ["lm_head"]
    return {n: round(float(v) / launches, 1) for n, v in zip(names, acc)}


def plain_next_rows(wl, box, out_t, out_c, rng):
    """Next step without a trajectory (T = 1, or an MTP head's own drafts):
    each sequence's first row is its bonus token at the new length."""
    tok, pos, sid = box[0]
    new_tok, new_pos, new_sid = [], [], []
    at = 0
    for i, (_c, T) in enumerate(wl.seqs):
        c = int(out_c[i])
        bonus = int(out_t[at + c - 1])
        at += c
        base = int(np.asarray(pos)[np.asarray(sid) == i][0]) + c
        new_tok += [bonus] + [int(x) for x in rng.integers(0, wl.model["vocab"], T - 1)]
        new_pos += list(range(base, base + T))
        new_sid += [i] * T
    return np.array(new_tok, np.int32), np.array(new_pos, np.int32), np.array(new_sid, np.int32)


def run_ours(args, world, rank, local):
    import torch
    from gen import synth
    from gen.workload import Workload
    from speculative_decode_persistent_gb300 import mk

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    t_setup = time.perf_counter()
    names = [args.workload] + [w for w in args.per_workload.split(",") if w and w != args.workload]
    if args.layers:
        names = [args.workload]
    results, engines, weights, setup = {}, {}, {}, {}
    for name in names:
        t0 = time.perf_counter()
        wl = Workload(name, nthreads=os.cpu_count(), overrides=layer_override(name, args.layers), weights=False)
        mkey = json.dumps(wl.model, sort_keys=True)
        if mkey not in weights:
            weights.clear()  # one model's weights on the host at a time
            weights[mkey] = synth.make_weights(wl.model, wl.spec.get("weight_seed", 0), 0.0, os.cpu_count())
        n_draft = int(wl.spec.get("n_draft", 0)) if wl.model.get("has_mtp") else 0
        ekey = (mkey, wl.kv_q8, wl.n_pages, n_draft)
        if ekey not in engines:
            for e in engines.values():
                e.close()
            engines.clear()
            engines[ekey] = mk.Engine(wl.model, weights[mkey], wl.kv_q8, wl.n_pages, max_seqs=wl.max_seqs,
                                      device=f"cuda:{local}", n_draft=n_draft)
            engines[ekey].load_pool(wl.pool)
        eng = engines[ekey]
        for s in range(8):
            eng.seq_reset(s)
        for s, (cached, _T) in enumerate(wl.seqs):
            eng.seq_set(s, cached, wl.tables[s], *wl.states[s])
        setup[name] = time.perf_counter() - t0
        results[name] = measure(args, eng, wl, name, world, dev, torch, args.layers)
        del wl
    for e in engines.values():
        e.close()
    head = results[args.workload]
    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "q4-weights/f16-split-mma/f32",
            "data": "synthetic (seeded random-init weights and caches)",
            "config": workload_config(args.workload, args.layers),
            "step_us": head["step_us"],
            "roofline": head["roofline"],
            "e2e": head["e2e"],
            "gpu_launches": head["gpu_launches"],
            "clocks": head["clocks"],
            **({"timeline_us": head["timeline_us"]} if "timeline_us" in head else {}),
            "setup_s": time.perf_counter() - t_setup,
        }
        others = {n: {k: r[k] for k in ("value", "ms_per_step", "step_us", "rows_per_step", "e2e", "clocks",
                                       "gpu_launches")} | {"roofline": {k: r["roofline"][k] for k in
                                                                        ("achieved", "peak", "frac", "unit",
                                                                         "algorithmic_bytes", "launch_ms_median")}}
                  for n, r in results.items() if n != args.workload}
        if others:
            line["per_workload"] = others
        t1, t5 = results.get("qwen27-t1-4k-fp16"), results.get("qwen27-t5-4k-fp16")
        if t1 and t5:
            line["t5_over_t1"] = t5["ms_per_step"] / t1["ms_per_step"]
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = {k: v for k, v in cpu_oracle_sample(args.workload, budget_s=args.ref_budget).items()
                                    if k in ("value", "unit", "cores", "kind", "sample")}
        print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--workload", default="qwen27-4x3-23k-q8")
    ap.add_argument("--per-workload", default="qwen27-t1-4k-fp16,qwen27-t5-4k-fp16",
                    help="comma-separated workloads timed in the same run (per_workload)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-budget", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="profiling stand-in: keep only the first N layers")
    ap.add_argument("--timeline", action="store_true",
                    help="add timeline_us: per-phase time of the step (block 0's stamps), after the timed launches")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
