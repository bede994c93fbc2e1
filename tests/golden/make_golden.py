"""Writes tests/golden/tiny_oracle_step.json: the oracle's output for one
seeded verify step of the tiny model, with and without the MTP draft head.

Calls only gen/ (the seeded inputs) and oracle/. The stored values are a
regression fixture for the oracle itself: a later change to its arithmetic
that moves them must say which passage of the pages justifies it and rerun
this script. (The pages print no worked example whose values could be stored
instead.)

    python tests/golden/make_golden.py
"""
from __future__ import annotations

import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from gen import configs  # noqa: E402
from gen.workload import Workload  # noqa: E402
from oracle import oracle as orc  # noqa: E402

OUT = os.path.join(HERE, "tiny_oracle_step.json")


def greedy_drafts(wl, model):
    """Drafts for the fixture step: the oracle's greedy continuation for two
    rows (one-row passes), then a wrong token, so two drafts are accepted."""
    o = orc.Oracle(wl.model, wl.weights, wl.pool, wl.kv_q8, wl.n_pages, wl.max_seqs, nthreads=2)
    o.seq_set(0, wl.seqs[0][0], wl.tables[0], *wl.states[0])
    tok, pos, out = int(wl.first_tokens[0]), wl.seqs[0][0], []
    for j in range(2):
        r = o.step([tok], [pos + j], [0], want_logits=False)
        o.commit([0], [1])
        tok = int(r["argmax"][0])
        out.append(tok)
    return out + [(out[-1] * 31 + 7) % model["vocab"]]


def run(model, n_draft):
    wl = Workload("tiny", norm_jitter=0.1, overrides=dict(model=model))
    o = orc.Oracle(wl.model, wl.weights, wl.pool, wl.kv_q8, wl.n_pages, wl.max_seqs, nthreads=2,
                   n_draft=n_draft)
    o.seq_set(0, wl.seqs[0][0], wl.tables[0], *wl.states[0])
    tok, pos, sid = wl.rows([greedy_drafts(wl, model)])
    r = o.step(tok, pos, sid, want_hidden=True)
    out = dict(tokens=[int(t) for t in tok], positions=[int(p) for p in pos],
               emitted=[int(t) for t in r["tokens"]], counts=[int(c) for c in r["counts"]],
               argmax=[int(a) for a in r["argmax"]], gap=[float(g) for g in r["gap"]],
               rms=[float(x) for x in r["rms"]],
               logits_head=[[float(x) for x in row[:8]] for row in r["logits"]],
               hidden_head=[[float(x) for x in row[:8]] for row in r["hidden"]])
    if n_draft:
        d = o.drafts(0)
        out["drafts"] = [int(x) for x in d["tokens"]]
        out["draft_gap"] = [float(x) for x in d["gap"]]
        out["draft_logits_head"] = [[float(x) for x in row[:8]] for row in d["logits"]]
    return out


def build():
    mtp = dict(configs.TINY, has_mtp=1, draft_vocab=1024)
    return {"tiny": run(configs.TINY, 0), "tiny_mtp": run(mtp, 3)}


if __name__ == "__main__":
    with open(OUT, "w") as f:
        json.dump(build(), f, indent=1)
    print("wrote", OUT)
