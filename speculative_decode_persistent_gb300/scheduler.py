"""Host scheduler for several agents sharing one engine: every step stacks the
rows of all active conversations into ONE verify cycle, so the weights are
streamed once for all of them.

What it does, following the multi-agent mode of the pages (page "OpenJet's
CUDA megakernel runs 4 coding agents on one RTX 3090", sections "What
shipped" and "Why it matters"):
- up to `max_slots` conversations, one engine sequence slot each;
- each decoding agent contributes its next token plus up to `n_draft`
  prompt-lookup drafts (the tokens that followed the most recent earlier
  occurrence of the conversation's last n-gram);
- a new prompt does not stall the others: each step carries the next chunk
  of every pending prompt beside their rows (prompt rows, at most
  `max_rows_per_seq` per conversation and step); drafts are cut back so that
  at least `min_prefill_rows` rows of a step go to prompts while any wait;
- slot affinity: a follow-up request of a conversation returns to the slot
  that holds it, so only its new tokens are processed;
- prefix reuse: a registered prefix (say the system prompt and tool list
  common to all agents) is processed once into a template sequence; a
  conversation that starts with it is installed as a copy of the template
  (its KV pages and recurrent state) and processes only the rest.

The engine is any object with the mk.Engine calls used here: step, commit,
seq_get, seq_reset, seq_new (an empty sequence with a zero recurrent state)
and clone_sequence, for a model without an MTP head (the library takes no
prompt rows beside one). The scheduler commits the rows it keeps right after
each step, so no sequence is left pending between steps.
"""
from __future__ import annotations

from dataclasses import dataclass, field

from .mk import MK_MAX_DECODE_ROWS, MK_MAX_T, MkError

MK_ERR_NO_PAGES = -3  # mk_status of a step refused for lack of free pages


def prompt_lookup(history, n_draft: int, max_ngram: int = 3, min_ngram: int = 1) -> list:
    """Prompt-lookup drafts: for n from max_ngram down to min_ngram, find the
    most recent earlier occurrence of the last n tokens of `history` and
    return up to n_draft tokens that followed it; [] when none matches."""
    h = list(history)
    L = len(h)
    if n_draft <= 0:
        return []
    for n in range(min(max_ngram, L - 1), min_ngram - 1, -1):
        tail = h[L - n:]
        for i in range(L - n - 1, -1, -1):
            if h[i:i + n] == tail:
                return h[i + n:i + n + n_draft]
    return []


@dataclass
class _Conv:
    cid: object
    slot: int
    history: list = field(default_factory=list)  # every token: prompts and generated
    cached: int = 0           # tokens whose KV and recurrent state are in the engine
    emitted: bool = False     # the last token of history was generated and is not cached yet
    max_new: int = 0          # tokens to generate for the current request
    new: list = field(default_factory=list)  # tokens generated for the current request
    stop: tuple = ()
    last_used: int = 0

    def prefilling(self):
        return not self.emitted and self.cached < len(self.history)

    def decoding(self):
        stopped = bool(self.new) and self.new[-1] in self.stop
        return self.emitted and len(self.new) < self.max_new and not stopped

    def active(self):
        return self.prefilling() or self.decoding()


@dataclass
class _Template:
    tokens: list
    slot: int


class AgentScheduler:
    """Continuous multi-agent loop over one engine (see the module docstring)."""

    def __init__(self, engine, max_slots: int = 8, n_draft: int = 2, max_rows: int = MK_MAX_DECODE_ROWS,
                 max_rows_per_seq: int = MK_MAX_T, min_prefill_rows: int = 4, max_ngram: int = 3):
        if not 1 <= max_rows_per_seq <= MK_MAX_T or not 1 <= max_rows <= MK_MAX_DECODE_ROWS:
            raise ValueError("row limits beyond the engine's")
        self.eng = engine
        self.max_slots = max_slots
        self.n_draft = n_draft
        self.max_rows = max_rows
        self.max_rows_per_seq = max_rows_per_seq
        self.min_prefill_rows = min_prefill_rows
        self.max_ngram = max_ngram
        self.convs: dict = {}
        self.templates: list = []
        self.clock = 0
        self.steps = 0
        self.rows_total = 0

    # ------------------------------------------------------------- slots
    def _free_slot(self):
        used = {c.slot for c in self.convs.values()} | {t.slot for t in self.templates if t is not None}
        for s in range(self.max_slots):
            if s not in used:
                return s
        idle = [c for c in self.convs.values() if not c.active()]
        if not idle:
            raise RuntimeError("every slot holds an active conversation or a template")
        victim = min(idle, key=lambda c: c.last_used)  # least recently used
        self.release(victim.cid)
        return victim.slot

    # ------------------------------------------------------------ requests
    def register_prefix(self, tokens) -> int:
        """Process `tokens` once into a template sequence (prompt rows, in
        chunks of max_rows_per_seq); conversations that start with them are
        installed as its copy. Returns the template id."""
        tokens = [int(x) for x in tokens]
        slot = self._free_slot()
        self.eng.seq_new(slot)
        done = 0
        while done < len(tokens):
            n = min(self.max_rows_per_seq, len(tokens) - done)
            self.eng.step(tokens[done:done + n], list(range(done, done + n)), [slot] * n, [1] * n)
            self.steps += 1
            self.rows_total += n
            done += n
        self.templates.append(_Template(tokens, slot))
        return len(self.templates) - 1

    def submit(self, cid, tokens, max_new_tokens: int, stop=()):
        """Start conversation cid, or continue it in the slot that holds it,
        with new prompt tokens; ask for up to max_new_tokens generated tokens
        (ending early after a token in `stop`)."""
        tokens = [int(x) for x in tokens]
        self.clock += 1
        c = self.convs.get(cid)
        if c is None:
            if not tokens:
                raise ValueError("a new conversation needs at least one token")
            c = _Conv(cid, self._free_slot())
            tpl = self._template_for(tokens)
            if tpl is not None:
                while True:  # the copy needs free pages: idle conversations give theirs up
                    try:
                        self.eng.clone_sequence(tpl.slot, c.slot)
                        break
                    except MkError as e:
                        idle = [x for x in self.convs.values() if not x.active()]
                        if e.status != MK_ERR_NO_PAGES or not idle:
                            raise
                        self.release(min(idle, key=lambda x: x.last_used).cid)
                c.history, c.cached = list(tpl.tokens), len(tpl.tokens)
                tokens = tokens[len(tpl.tokens):]
            else:
                self.eng.seq_new(c.slot)
            self.convs[cid] = c
        c.history += tokens
        if tokens:
            c.emitted = False  # the new tokens (and the uncached last one) are a prompt
        c.max_new, c.new, c.stop, c.last_used = int(max_new_tokens), [], tuple(stop), self.clock

    def _template_for(self, tokens):
        best = None
        for t in self.templates:
            if t is None:
                continue
            n = len(t.tokens)
            if n < len(tokens) and tokens[:n] == t.tokens and (best is None or n > len(best.tokens)):
                best = t
        return best

    def release(self, cid):
        """Drop a conversation; its slot and pages return to the engine."""
        c = self.convs.pop(cid)
        self.eng.seq_reset(c.slot)

    def drop_prefix(self, tid: int):
        """Drop a registered prefix; its slot and pages return to the engine
        (conversations already copied from it keep their copies)."""
        t = self.templates[tid]
        if t is not None:
            self.eng.seq_reset(t.slot)
            self.templates[tid] = None

    def output(self, cid):
        return list(self.convs[cid].new)

    def busy(self):
        return any(c.active() for c in self.convs.values())

    # ---------------------------------------------------------------- step
    def _plan(self):
        """Rows of the next step: [(conversation, tokens, positions, flag)]."""
        dec = sorted((c for c in self.convs.values() if c.decoding()), key=lambda c: c.last_used)
        pre = sorted((c for c in self.convs.values() if c.prefilling()), key=lambda c: c.last_used)
        budget = self.max_rows - len(dec)
        if budget < 0:
            raise RuntimeError("more decoding conversations than rows in a step")
        draft_budget = budget - (min(self.min_prefill_rows, budget) if pre else 0)
        plan = []
        for c in dec:
            want = min(self.n_draft, self.max_rows_per_seq - 1, c.max_new - len(c.new) - 1, draft_budget)
            drafts = prompt_lookup(c.history, want, self.max_ngram) if want > 0 else []
            draft_budget -= len(drafts)
            toks = [c.history[-1]] + drafts
            plan.append((c, toks, list(range(c.cached, c.cached + len(toks))), 0))
        budget = self.max_rows - sum(len(p[1]) for p in plan)
        for c in pre:
            if budget <= 0:
                break
            n = min(len(c.history) - c.cached, self.max_rows_per_seq, budget)
            ends = c.cached + n == len(c.history) and c.max_new > 0
            plan.append((c, c.history[c.cached:c.cached + n], list(range(c.cached, c.cached + n)), 2 if ends else 1))
            budget -= n
        return plan

    def _launch(self, plan):
        while True:
            tok, pos, sid, fl = [], [], [], []
            for c, t, p, f in plan:
                tok += t
                pos += p
                sid += [c.slot] * len(t)
                fl += [f] * len(t) if f != 2 else [1] * (len(t) - 1) + [2]  # 2 marks the prompt's last row only
            try:
                return plan, self.eng.step(tok, pos, sid, fl), len(tok)
            except MkError as e:
                if e.status != MK_ERR_NO_PAGES:
                    raise
                idle = [c for c in self.convs.values() if not c.active()]
                if idle:
                    self.release(min(idle, key=lambda c: c.last_used).cid)
                elif any(p[3] for p in plan) and any(not p[3] for p in plan):
                    plan = [p for p in plan if not p[3]]  # prompts wait, decoding goes on
                else:
                    raise

    def step(self):
        """One engine step over every active conversation. Returns
        {conversation id: tokens generated this step}."""
        plan = self._plan()
        if not plan:
            return {}
        plan, (out_t, out_c), nrows = self._launch(plan)
        self.steps += 1
        self.rows_total += nrows
        generated, verified, keep = {}, [], []
        at = 0
        for (c, t, p, f), cnt in zip(plan, out_c):
            cnt = int(cnt)
            got = [int(x) for x in out_t[at:at + cnt]]
            at += cnt
            # keep what the request still wants, up to and including a stop token
            got = got[:c.max_new - len(c.new)]
            for i, x in enumerate(got):
                if x in c.stop:
                    got = got[:i + 1]
                    break
            if f == 0:
                # the first row and the accepted drafts that stay in the
                # history enter the cache: as many rows as tokens kept
                c.cached += len(got)
                verified.append(c.slot)
                keep.append(len(got))
            else:  # prompt rows are committed through their last row by the step
                c.cached += len(t)
            if got:
                c.history += got
                c.new += got
                c.emitted = True
                generated[c.cid] = got
            c.last_used = self.clock
        if verified:
            self.eng.commit(verified, keep)
        self.clock += 1
        return generated

    def run(self, max_steps: int = 100_000):
        """Step until no conversation is active; returns {id: generated tokens}."""
        for _ in range(max_steps):
            if not self.busy():
                break
            self.step()
        return {cid: list(c.new) for cid, c in self.convs.items()}
