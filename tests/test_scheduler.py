"""The multi-agent host scheduler (speculative_decode_persistent_gb300.scheduler)
on the CPU, over a toy engine with the library's step semantics: rows of a
sequence start at its committed length; verify rows accept drafts while they
equal the greedy token and return the accepted drafts plus the bonus; prompt
rows are committed at once (flag 2 on the last row returns the greedy token);
pages are taken lowest id first and a step that cannot get them is refused
before any change; commit keeps n rows of the pending step. The toy model's
next token depends on every cached token (read back from its pages) and on a
recurrent state kept per row, so a wrong page or state copy changes the text.

Checked: prompt-lookup drafts; every conversation's text equals running it
alone with plain greedy decoding (one token per step), with drafts, stacked
rows, chunked prompts, a shared prefix processed once, follow-up requests
in the same slot, max-token and stop truncation, and eviction when pages run
out; a pending prompt never stalls the decoding agents."""
import numpy as np
import pytest

from speculative_decode_persistent_gb300.mk import MK_MAX_DECODE_ROWS, MK_MAX_T, MkError
from speculative_decode_persistent_gb300.scheduler import AgentScheduler, prompt_lookup

V = 23  # toy vocabulary: small, so prompt-lookup drafts are often right


class ToyEngine:
    PT = 16

    def __init__(self, n_pages=64, max_seqs=8):
        self.n_pages, self.max_seqs = n_pages, max_seqs
        self.page_tok = np.full((n_pages, self.PT), -1, np.int64)
        self.free = set(range(n_pages))
        self.seqs = {}   # seq -> dict(len, pages, state)
        self.pending = {}  # seq -> dict(rows, states)
        self.rows_seen = []  # (seq, flag, n) per step and sequence

    # -- the toy model: next token after the cached prefix ending at `pos`
    def _next(self, s, pos, state):
        pages = self.seqs[s]["pages"]
        tok = lambda q: int(self.page_tok[pages[q // self.PT], q % self.PT])  # noqa: E731
        a = tok(pos)
        b = tok(pos - 1) if pos >= 1 else 0
        c = tok(pos // 2)
        return (7 * a + 3 * b + 5 * c + state + pos) % V

    @staticmethod
    def _state(state, t):
        return (3 * state + t + 1) % 97

    # -- the engine interface the scheduler uses
    def seq_new(self, s):
        self.seq_reset(s)
        self.seqs[s] = dict(len=0, pages=[], state=0)

    def seq_reset(self, s):
        self.pending.pop(s, None)
        if s in self.seqs:
            self.free.update(self.seqs[s]["pages"])
            del self.seqs[s]

    def seq_get(self, s):
        q = self.seqs[s]
        return dict(length=q["len"], pages=np.array(q["pages"], np.int32), slot=0)

    def clone_sequence(self, src, dst):
        self.seq_reset(dst)
        q = self.seqs[src]
        if len(self.free) < len(q["pages"]):
            raise MkError(-3, "clone")
        new = sorted(self.free)[: len(q["pages"])]
        for a, b in zip(q["pages"], new):
            self.page_tok[b] = self.page_tok[a]
        self.free -= set(new)
        self.seqs[dst] = dict(len=q["len"], pages=new, state=q["state"])

    def _commit(self, s, keep):
        p = self.pending.pop(s)
        q = self.seqs[s]
        q["len"] += keep
        q["state"] = p["states"][keep - 1]
        need = (q["len"] + self.PT - 1) // self.PT
        self.free.update(q["pages"][need:])
        q["pages"] = q["pages"][:need]

    def commit(self, seq_ids, n_keep):
        for s, k in zip(seq_ids, n_keep):
            assert 1 <= k <= self.pending[s]["count"], (s, k)
            self._commit(int(s), int(k))

    def step(self, tokens, positions, seq_ids, flags):
        tokens, positions, seq_ids, flags = map(list, (tokens, positions, seq_ids, flags))
        assert len(tokens) <= MK_MAX_DECODE_ROWS
        order = []
        for s in seq_ids:
            if s not in order:
                order.append(s)
        for s in order:  # a pending step is committed with every accepted row
            if s in self.pending:
                self._commit(s, self.pending[s]["count"])
        need = 0
        for s in order:
            idx = [i for i, x in enumerate(seq_ids) if x == s]
            assert idx == list(range(idx[0], idx[0] + len(idx))), "rows of a sequence are contiguous"
            assert len(idx) <= MK_MAX_T
            assert [positions[i] for i in idx] == list(range(self.seqs[s]["len"], self.seqs[s]["len"] + len(idx)))
            # one kind per sequence: verify rows (0), or prompt rows (1) of
            # which only the last may end the prompt (2)
            fs = [flags[i] for i in idx]
            assert fs == [0] * len(fs) or (set(fs[:-1]) <= {1} and fs[-1] in (1, 2)), fs
            end = self.seqs[s]["len"] + len(idx)
            need += max(0, (end + self.PT - 1) // self.PT - len(self.seqs[s]["pages"]))
        if need > len(self.free):
            raise MkError(-3, "mk_step")  # before any change
        out_t, out_c = [], []
        for s in order:
            idx = [i for i, x in enumerate(seq_ids) if x == s]
            q = self.seqs[s]
            state, states, greedy = q["state"], [], []
            for i in idx:
                pos = positions[i]
                if pos // self.PT >= len(q["pages"]):
                    pg = min(self.free)
                    self.free.remove(pg)
                    q["pages"].append(pg)
                self.page_tok[q["pages"][pos // self.PT], pos % self.PT] = tokens[i]
                state = self._state(state, tokens[i])
                states.append(state)
                greedy.append(self._next(s, pos, state))
            f = flags[idx[0]]
            self.rows_seen.append((s, f if f == 0 else 1, len(idx)))
            if f == 0:
                a = 0
                while a + 1 < len(idx) and tokens[idx[a + 1]] == greedy[a]:
                    a += 1
                out_t += [tokens[i] for i in idx[1:a + 1]] + [greedy[a]]
                out_c.append(a + 1)
                self.pending[s] = dict(count=a + 1, states=states)
            else:
                q["len"] += len(idx)
                q["state"] = state
                if flags[idx[-1]] == 2:
                    out_t.append(greedy[-1])
                    out_c.append(1)
                else:
                    out_c.append(0)
        return np.array(out_t, np.int32), np.array(out_c, np.int32)


def solo(tokens, max_new, stop=(), follow=()):
    """Plain greedy decoding of one conversation alone: the prompt, then one
    token per step; `follow`: (new tokens, max_new) requests after it."""
    e = ToyEngine(n_pages=256)
    e.seq_new(0)
    hist = list(tokens)
    outs = []
    cached = 0
    for req, mx in [(list(tokens), max_new)] + list(follow):
        if outs:
            hist += req
        new = []
        # prompt: every token not yet cached, the last one returning the greedy token
        for i in range(cached, len(hist)):
            f = 2 if (i == len(hist) - 1 and mx > 0) else 1
            t, c = e.step([hist[i]], [i], [0], [f])
            if f == 2:
                new.append(int(t[0]))
        cached = len(hist)
        while new and len(new) < mx and new[-1] not in stop:
            t, c = e.step([new[-1]], [cached], [0], [0])
            e.commit([0], [1])
            cached += 1
            new.append(int(t[0]))
        new = new[:mx]
        hist += new
        outs.append(new)
    return outs


def test_prompt_lookup():
    h = [1, 2, 3, 9, 1, 2, 3, 4, 5, 1, 2, 3]
    assert prompt_lookup(h, 2) == [4, 5]  # the most recent earlier "1 2 3"
    assert prompt_lookup(h, 5) == [4, 5, 1, 2, 3]
    assert prompt_lookup([5, 6, 7], 2) == []
    assert prompt_lookup([4, 8, 4], 2, max_ngram=3) == [8, 4]  # falls back to the 1-gram
    assert prompt_lookup(h, 0) == []
    assert prompt_lookup([], 3) == [] and prompt_lookup([1], 3) == []


def _prompts(rng, n, lo, hi):
    return [[int(x) for x in rng.integers(0, V, int(rng.integers(lo, hi)))] for _ in range(n)]


def test_agents_match_solo_greedy():
    rng = np.random.default_rng(3)
    prompts = _prompts(rng, 4, 5, 40)
    eng = ToyEngine()
    sch = AgentScheduler(eng, n_draft=2)
    for i, p in enumerate(prompts):
        sch.submit(i, p, 30)
    out = sch.run()
    for i, p in enumerate(prompts):
        assert out[i] == solo(p, 30)[0], i
    # rows were stacked: far fewer steps than the agents' tokens one by one
    assert sch.steps < sum(len(p) + 30 for p in prompts) / 3
    assert all(n <= MK_MAX_T for _s, _f, n in eng.rows_seen)


def test_shared_prefix_processed_once_and_followups_stay_in_slot():
    rng = np.random.default_rng(5)
    system = [int(x) for x in rng.integers(0, V, 37)]
    users = _prompts(rng, 3, 3, 12)
    eng = ToyEngine()
    sch = AgentScheduler(eng, n_draft=2)
    sch.register_prefix(system)
    prefix_rows = sum(n for _s, f, n in eng.rows_seen if f)
    assert prefix_rows == len(system)
    for i, u in enumerate(users):
        sch.submit(i, system + u, 12)
    first = sch.run()
    # only the users' own tokens were processed as prompts after the template
    prompt_rows = sum(n for _s, f, n in eng.rows_seen if f) - prefix_rows
    assert prompt_rows == sum(len(u) for u in users)
    slots = {i: sch.convs[i].slot for i in range(3)}
    more = _prompts(rng, 3, 2, 6)
    for i, m in enumerate(more):
        sch.submit(i, m, 9)
    second = sch.run()
    for i in range(3):
        want = solo(system + users[i], 12, follow=[(more[i], 9)])
        assert first[i] == want[0] and second[i] == want[1], i
        assert sch.convs[i].slot == slots[i]  # slot affinity


def test_prompt_does_not_stall_decoding():
    rng = np.random.default_rng(7)
    eng = ToyEngine()
    sch = AgentScheduler(eng, n_draft=2, min_prefill_rows=4)
    short = _prompts(rng, 4, 3, 6)
    for i, p in enumerate(short):
        sch.submit(i, p, 40)
    while not all(sch.convs[i].decoding() for i in range(4)):
        sch.step()
    long_prompt = [int(x) for x in rng.integers(0, V, 45)]
    sch.submit("new", long_prompt, 5)
    before = sch.convs["new"].cached
    steps = 0
    while sch.convs["new"].prefilling():
        got = sch.step()
        steps += 1
        for i in range(4):  # every decoding agent got tokens in every step
            if sch.convs[i].decoding() or i in got:
                assert i in got
        assert sch.convs["new"].cached - before >= 4 or not sch.convs["new"].prefilling()
        before = sch.convs["new"].cached
    assert steps <= (45 + 3) // 4
    out = sch.run()
    assert out["new"] == solo(long_prompt, 5)[0]
    for i, p in enumerate(short):
        assert out[i] == solo(p, 40)[0]


def test_max_tokens_and_stop():
    rng = np.random.default_rng(11)
    p = _prompts(rng, 1, 10, 20)[0]
    full = solo(p, 25)[0]
    stop_tok = full[7]
    eng = ToyEngine()
    sch = AgentScheduler(eng, n_draft=3)
    sch.submit("a", p, 25, stop=(stop_tok,))
    sch.submit("b", p, 4)
    out = sch.run()
    assert out["a"] == full[: full.index(stop_tok) + 1]
    assert out["b"] == full[:4]
    # the truncated conversations continue correctly in their slots
    sch.submit("b", [1, 2], 6)
    out = sch.run()
    assert out["b"] == solo(p, 4, follow=[([1, 2], 6)])[1]


def test_eviction_when_pages_run_out():
    rng = np.random.default_rng(13)
    eng = ToyEngine(n_pages=5)  # "a" keeps 3 pages, "b" needs 4
    sch = AgentScheduler(eng, n_draft=1, max_slots=3)
    a = _prompts(rng, 1, 30, 31)[0]
    sch.submit("a", a, 10)
    sch.run()
    b = _prompts(rng, 1, 40, 41)[0]
    sch.submit("b", b, 20)  # needs pages only the idle "a" holds
    out = sch.run()
    assert "a" not in sch.convs and out["b"] == solo(b, 20)[0]
    c = _prompts(rng, 1, 200, 201)[0]
    sch.submit("c", c, 5)
    with pytest.raises(MkError):
        sch.run()  # more pages than the pool, nothing idle to evict


class OracleEngine:
    """The fp64 oracle behind the engine calls the scheduler makes (no
    prefix templates: the oracle's state goes in through fp32)."""

    def __init__(self, orc):
        self.o = orc

    def seq_new(self, s):
        self.o.seq_set(s, 0, np.zeros(0, np.int32))

    def seq_reset(self, s):
        self.o.seq_set(s, 0, np.zeros(0, np.int32))

    def seq_get(self, s):
        g = self.o.seq_get(s)
        return dict(length=g["length"], pages=g["pages"], slot=0)

    def commit(self, seq_ids, n_keep):
        self.o.commit(seq_ids, n_keep)

    def step(self, tokens, positions, seq_ids, flags):
        r = self.o.step(tokens, positions, seq_ids, flags, want_logits=False)
        return r["tokens"], r["counts"]


def oracle_solo(make, prompt, max_new):
    """One conversation alone on a fresh oracle: prompt rows one by one, then
    one verify row per step."""
    e = OracleEngine(make())
    e.seq_new(0)
    for i, t in enumerate(prompt):
        tok, _c = e.step([t], [i], [0], [2 if i == len(prompt) - 1 else 1])
    new = [int(tok[0])]
    pos = len(prompt)
    while len(new) < max_new:
        tok, _c = e.step([new[-1]], [pos], [0], [0])
        e.commit([0], [1])
        pos += 1
        new.append(int(tok[0]))
    return new


def test_scheduler_on_the_oracle_tiny_model():
    from gen.workload import Workload
    from oracle import oracle as orc
    wl = Workload("tiny", nthreads=2)

    def make():
        return orc.Oracle(wl.model, wl.weights, {k: v.copy() for k, v in wl.pool.items()}, wl.kv_q8,
                          wl.n_pages, wl.max_seqs, nthreads=2)

    rng = np.random.default_rng(17)
    V_tiny = wl.model["vocab"]
    base = [int(x) for x in rng.integers(0, V_tiny, 6)]
    prompts = [base * 3 + [int(x) for x in rng.integers(0, V_tiny, n)] for n in (2, 9, 17)]
    sch = AgentScheduler(OracleEngine(make()), n_draft=2)
    for i, p in enumerate(prompts):
        sch.submit(i, p, 10)
    out = sch.run()
    for i, p in enumerate(prompts):
        assert out[i] == oracle_solo(make, p, 10), i


def test_prefix_copy_evicts_idle_and_prefix_can_be_dropped():
    rng = np.random.default_rng(23)
    system = [int(x) for x in rng.integers(0, V, 33)]  # 3 pages once processed
    eng = ToyEngine(n_pages=8)
    sch = AgentScheduler(eng, n_draft=1, max_slots=4)
    tid = sch.register_prefix(system)
    u1 = [int(x) for x in rng.integers(0, V, 5)]
    sch.submit("x", system + u1, 4)
    out = sch.run()
    assert out["x"] == solo(system + u1, 4)[0]
    # "x" (3 pages) is idle; a second copy of the prefix needs 3 of the 2 free pages
    u2 = [int(x) for x in rng.integers(0, V, 4)]
    sch.submit("y", system + u2, 3)
    assert "x" not in sch.convs
    assert sch.run()["y"] == solo(system + u2, 3)[0]
    sch.drop_prefix(tid)
    assert sch.templates[tid] is None and len(eng.free) == 8 - len(eng.seqs[sch.convs["y"].slot]["pages"])
    sch.submit("z", system + u1, 4)  # no template any more: the whole prompt is processed
    assert sch.run()["z"] == solo(system + u1, 4)[0]


@pytest.mark.parametrize("seed", range(6))
def test_random_mixes_match_solo(seed):
    """Random conversation mixes, row limits, draft depths and follow-ups:
    every step stays within the engine's limits (the toy engine asserts them)
    and every text equals the conversation decoded alone."""
    rng = np.random.default_rng(100 + seed)
    eng = ToyEngine(n_pages=96)
    sch = AgentScheduler(eng, n_draft=int(rng.integers(0, 5)), max_rows=int(rng.integers(6, 13)),
                         max_rows_per_seq=int(rng.integers(2, 9)), min_prefill_rows=int(rng.integers(1, 5)))
    n = int(rng.integers(2, 7))
    prompts = _prompts(rng, n, 1, 30)
    want_new = [int(rng.integers(1, 25)) for _ in range(n)]
    for i in range(n):
        sch.submit(i, prompts[i], want_new[i])
        if rng.random() < 0.5:
            sch.step()  # arrivals spread over steps
    first = sch.run()
    follow = {i: (_prompts(rng, 1, 1, 8)[0], int(rng.integers(1, 10))) for i in range(n) if rng.random() < 0.5}
    for i, (t, m) in follow.items():
        sch.submit(i, t, m)
    second = sch.run()
    for i in range(n):
        want = solo(prompts[i], want_new[i], follow=[follow[i]] if i in follow else [])
        assert first[i] == want[0], (seed, i)
        if i in follow:
            assert second[i] == want[1], (seed, i)
    assert sum(n_rows for _s, _f, n_rows in eng.rows_seen) == sch.rows_total
