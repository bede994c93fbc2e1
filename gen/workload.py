"""Synthetic workload set-up shared by tests, the smoke check and the benchmark.

Builds, from seeds only: the canonical weights, a filled KV pool, per-sequence
page tables (contiguous, or a seeded shuffle of the pool's pages) and
recurrent states, plus the first row tokens. No step arithmetic here.
"""
from __future__ import annotations

import numpy as np

from . import synth
from .configs import PAGE_TOKENS, WORKLOADS, model_dims


def page_tables(seqs, n_pages: int, shuffle_seed=None, reserve_free: bool = True):
    """Page ids for each sequence's cached tokens.

    Contiguous blocks by default; with shuffle_seed, the pages are taken in the
    order of a seeded permutation of the whole pool."""
    order = (np.arange(n_pages, dtype=np.int32) if shuffle_seed is None
             else synth.permutation(shuffle_seed, 70000, n_pages))
    tables, at = [], 0
    for cached, _rows in seqs:
        n = (cached + PAGE_TOKENS - 1) // PAGE_TOKENS
        if at + n > n_pages:
            raise ValueError("pool too small for the cached contexts")
        tables.append(np.ascontiguousarray(order[at:at + n]))
        at += n
    return tables


class Workload:
    """Everything both sides need to run one configuration."""

    def __init__(self, name: str | dict, weights: bool = True, norm_jitter: float = 0.0,
                 nthreads=None, overrides: dict | None = None, **kw):
        w = dict(WORKLOADS[name]) if isinstance(name, str) else dict(name)
        if overrides:
            w.update(overrides)
        w.update(kw)
        self.spec = w
        self.name = name if isinstance(name, str) else w.get("name", "custom")
        self.model = w["model"]
        self.dims = model_dims(self.model)
        self.kv_q8 = int(w["kv_q8"])
        self.n_pages = int(w["n_pages"])
        self.seqs = list(w["seqs"])
        self.max_seqs = max(8, len(self.seqs) + 1)
        self.weights = (synth.make_weights(self.model, w.get("weight_seed", 0), norm_jitter, nthreads)
                        if weights else None)
        self.pool = synth.make_pool(self.model, self.n_pages, self.kv_q8)
        synth.fill_pool(self.pool, w.get("cache_seed", 1), nthreads)
        self.tables = page_tables(self.seqs, self.n_pages, w.get("shuffle_seed"))
        self.states = [synth.make_seq_states(self.model, w.get("cache_seed", 1) + s, s, nthreads)
                       for s in range(len(self.seqs))]
        self.first_tokens = synth.uniform_tokens(w.get("draft_seed", 2), 80000, len(self.seqs),
                                                 self.model["vocab"])

    def rows(self, drafts=None):
        """Row arrays of one verify step: per sequence, row 0 is its first token
        at position = cached length, rows 1.. are drafts (zeros if not given)."""
        tokens, positions, seq_ids = [], [], []
        for s, (cached, T) in enumerate(self.seqs):
            d = drafts[s] if drafts is not None else [0] * (T - 1)
            row_tokens = [int(self.first_tokens[s])] + [int(x) for x in d]
            assert len(row_tokens) == T
            for j in range(T):
                tokens.append(row_tokens[j])
                positions.append(cached + j)
                seq_ids.append(s)
        return (np.array(tokens, np.int32), np.array(positions, np.int32),
                np.array(seq_ids, np.int32))
