"""Full-size parity: the Qwen3.8-27B-shaped hybrid decoder (64 layers,
hidden 5120, FFN 17408, vocabulary 248,320, ~15 GB of Q4 weights) in the
launch configuration the benchmark times, verify steps against the fp64
oracle on identical seeded inputs: every row's logits and final hidden state,
the accepted tokens and counts, the committed recurrent state after the
accepted row, and the new KV entries.

Drafts are the oracle's greedy continuation with a chosen mismatch position,
so that a given number of drafts is accepted (the verify outcome the
workloads specify: accept lengths 0, 2 and 4 at T = 5; a seeded length per
sequence for 4 sequences x T = 3), and the state committed after a > 0
accepted rows is compared. Every test drives the CUDA path through the C ABI
(libmk.so via ctypes)."""
import os

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

from helpers import Pair, configs, drafts_with_mismatch  # noqa: E402

CASES = {
    # name: (workload, overrides, accept lengths: a list of steps, each a list per sequence)
    "t1-4k-fp16": ("qwen27-t1-4k-fp16", None, [[0]]),
    "t5-4k-fp16": ("qwen27-t5-4k-fp16", None, [[0], [2], [4]]),
    "4x3-23k-q8": ("qwen27-4x3-23k-q8", None, "seeded"),
    # T = 5 with the MTP draft head: four drafts per step over the first 32,768 tokens
    "t5-4k-fp16-mtp": ("qwen27-t5-4k-fp16-mtp", None, [[2]]),
    # the long-context stream: T = 5 over 96,000 cached tokens in a q8 pool
    "t5-96k-q8": ("qwen27-t5-96k-q8", None, [[3]]),
}


def _greedy(p, n):
    """The oracle's greedy continuation of every sequence (n one-row passes,
    one row per sequence), after which the oracle is put back to the cached
    state (positions past the cache are rewritten before they are read)."""
    wl = p.wl
    nseq = len(wl.seqs)
    toks = [int(t) for t in wl.first_tokens[:nseq]]
    out = [[] for _ in range(nseq)]
    sid = list(range(nseq))
    for j in range(n):
        r = p.oracle.step(toks, [c + j for c, _T in wl.seqs], sid, want_logits=False)
        p.oracle.commit(sid, [1] * nseq)
        toks = [int(a) for a in r["argmax"]]
        for s in range(nseq):
            out[s].append(toks[s])
    _reinstall(p)
    return out


def _reinstall(p):
    wl = p.wl
    for s, (cached, _T) in enumerate(wl.seqs):
        p.oracle.seq_set(s, cached, wl.tables[s], *wl.states[s])
        p.eng.seq_reset(s)
        p.eng.seq_set(s, cached, wl.tables[s], *wl.states[s])
    p.reset_flips()


@pytest.mark.parametrize("case", list(CASES))
def test_qwen27_full_step(cuda_ok, case):
    name, ov, accepts = CASES[case]
    p = Pair(name, overrides=ov, norm_jitter=0.0, nthreads=os.cpu_count())
    wl = p.wl
    V = wl.model["vocab"]
    nseq = len(wl.seqs)
    Tmax = max(T for _c, T in wl.seqs)
    if accepts == "seeded":  # accept lengths drawn per sequence (seed 9: 1, 2, 2, 0)
        rng = np.random.default_rng(9)
        accepts = [[int(rng.integers(0, wl.seqs[s][1])) for s in range(nseq)]]
    greedy = _greedy(p, Tmax - 1) if Tmax > 1 else [[] for _ in range(nseq)]
    seqs = list(range(nseq))
    n_fa = configs.model_dims(wl.model)["n_fa"]
    longest = 0
    for a_list in accepts:
        drafts = [drafts_with_mismatch(greedy[s], wl.seqs[s][1], a_list[s], V, salt=s) for s in seqs]
        tok, pos, sid = wl.rows(drafts)
        ro, rg = p.step(tok, pos, sid)
        excused, rep = p.compare_step(ro, rg, sid)
        co = [int(c) for c in ro["counts"]]
        cg = [int(c) for c in rg["counts"]]
        print(case, a_list, "counts oracle", co, "gpu", cg, rep)
        # the oracle's T-row pass equals its one-row passes, so it accepts exactly a
        assert co == [a + 1 for a in a_list], (co, a_list)
        longest = max(longest, max(cg))
        if p.n_draft:
            print(case, "drafts compared/excused", p.compare_drafts(seqs, [a == b for a, b in zip(co, cg)]))
            for s in seqs:
                if co[s] == cg[s]:
                    r0 = wl.seqs[s][0]
                    p.compare_kv(s, list(range(r0, r0 + co[s] + p.n_draft - 1)), layers=[n_fa])
        p.oracle.commit(seqs, co)
        p.eng.commit(seqs, cg)
        for s in seqs:
            mine = [int(x) for x, q in zip(pos, sid) if q == s]
            p.compare_kv(s, mine[: co[s]], layers=range(n_fa))
            if co[s] == cg[s]:  # a near-tie may legitimately change the accepted length
                p.compare_state(s)  # the state after the last accepted row
        _reinstall(p)
    if Tmax > 1 and max(max(a) for a in accepts) > 0:
        assert longest > 1, "no step accepted a draft"
