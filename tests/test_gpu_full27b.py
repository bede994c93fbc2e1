"""Full-size parity: the Qwen3.8-27B-shaped hybrid decoder (64 layers,
hidden 5120, FFN 17408, vocabulary 248,320, ~15 GB of Q4 weights) in the
launch configuration the benchmark times, one verify step against the fp64
oracle on identical seeded inputs: every row's logits and final hidden state,
the accepted tokens and counts, the committed recurrent state and the new KV
entries.

Every test drives the CUDA path through the C ABI (libmk.so via ctypes)."""
import os

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

from helpers import Pair, configs  # noqa: E402

CASES = {
    # name: (workload, overrides)
    "t1-4k-fp16": ("qwen27-t1-4k-fp16", None),
    "t5-4k-fp16": ("qwen27-t1-4k-fp16", dict(seqs=[(4096, 5)])),
    "4x3-23k-q8": ("qwen27-4x3-23k-q8", None),
    # T = 5 with the MTP draft head: four drafts per step over the first 32,768 tokens
    "t5-4k-fp16-mtp": ("qwen27-t5-4k-fp16-mtp", None),
}


@pytest.mark.parametrize("case", list(CASES))
def test_qwen27_full_step(cuda_ok, case):
    name, ov = CASES[case]
    p = Pair(name, overrides=ov, norm_jitter=0.0, nthreads=os.cpu_count())
    wl = p.wl
    rng = np.random.default_rng(7)
    tok, pos, sid = wl.rows([list(rng.integers(0, wl.model["vocab"], T - 1)) for (_c, T) in wl.seqs])
    ro, rg = p.step(tok, pos, sid)
    excused, rep = p.compare_step(ro, rg, sid)
    print(case, rep)
    co = [int(c) for c in ro["counts"]]
    cg = [int(c) for c in rg["counts"]]
    seqs = list(range(len(wl.seqs)))
    n_fa = configs.model_dims(wl.model)["n_fa"]
    if p.n_draft:
        print(case, "drafts compared/excused", p.compare_drafts(seqs, [a == b for a, b in zip(co, cg)]))
        for s in seqs:
            if co[s] == cg[s]:
                r0 = wl.seqs[s][0]
                p.compare_kv(s, list(range(r0, r0 + co[s] + p.n_draft - 1)), layers=[n_fa])
    p.oracle.commit(seqs, co)
    p.eng.commit(seqs, cg)
    for s in seqs:
        p.compare_kv(s, [int(x) for x, q in zip(pos, sid) if q == s], layers=range(n_fa))
        if co[s] == cg[s]:  # a near-tie may legitimately change the accepted length
            p.compare_state(s)
