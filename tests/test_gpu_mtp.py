"""The MTP draft head on the device against the fp64 oracle.

The head runs in the same persistent launch as the verify step. These tests
check the step's own outputs, the drafts for the next cycle, the KV entries
of the main attention layers and of the head's own KV layer, and the
committed state. Cases:
  - single sequences with every accept length;
  - a three-step speculative loop fed with the device's own drafts;
  - three sequences on a shuffled q8 pool;
  - draft positions that cross into a new page.

Every test drives the CUDA path through the C ABI (libmk.so via ctypes)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

from helpers import Pair, drafts_with_mismatch, greedy_continuation  # noqa: E402
from gen import configs  # noqa: E402

MTP_TINY = dict(configs.TINY, name="tiny-4L-h256-mtp", has_mtp=1, draft_vocab=1024)


def _pair(seqs, kv_q8=0, n_draft=3, shuffle=None):
    n_pages = sum((c + T + n_draft + 15) // 16 for c, T in seqs) + 8
    ov = dict(model=MTP_TINY, kv_q8=kv_q8, n_pages=n_pages, seqs=seqs, n_draft=n_draft)
    if shuffle is not None:
        ov["shuffle_seed"] = shuffle
    return Pair("tiny", overrides=ov)


def _check_step(p, tok, pos, sid):
    """One step on both sides; compares outputs, drafts and KV, then commits
    each side's own counts and compares the committed state. Returns the
    gpu drafts [n_seq][n_draft], both sides' counts and the gpu's emitted
    tokens."""
    ro, rg = p.step(tok, pos, sid)
    p.compare_step(ro, rg, sid)
    order = list(dict.fromkeys(int(s) for s in sid))
    co = [int(c) for c in ro["counts"]]
    cg = [int(c) for c in rg["counts"]]
    p.compare_drafts(order, [a == b for a, b in zip(co, cg)])
    n_fa = configs.model_dims(p.wl.model)["n_fa"]
    for i, s in enumerate(order):
        rows = [int(x) for x, q in zip(pos, sid) if q == s]
        p.compare_kv(s, rows, layers=range(n_fa))
        if co[i] == cg[i]:
            mtp_pos = list(range(rows[0], rows[0] + co[i] + p.n_draft - 1))
            p.compare_kv(s, mtp_pos, layers=[n_fa])
    drafts = p.eng.last_drafts(len(order))
    p.oracle.commit(order, co)
    p.eng.commit(order, cg)
    for i, s in enumerate(order):
        if co[i] == cg[i]:
            p.compare_state(s)
    return drafts, co, cg, rg["tokens"]


@pytest.mark.parametrize("kv_q8", [0, 1])
@pytest.mark.parametrize("accept", [0, 1, 2, 3])
def test_mtp_single_sequence(cuda_ok, kv_q8, accept):
    greedy = greedy_continuation("tiny", 4, overrides=dict(model=MTP_TINY, kv_q8=kv_q8, seqs=[(64, 4)]))
    p = _pair([(64, 4)], kv_q8=kv_q8)
    tok, pos, sid = p.wl.rows([drafts_with_mismatch(greedy, 4, accept, 2048)])
    _, co, cg, _ = _check_step(p, tok, pos, sid)
    assert co == cg == [accept + 1]


@pytest.mark.parametrize("kv_q8", [0, 1])
def test_mtp_speculative_loop(cuda_ok, kv_q8):
    """Three cycles where each step's drafts are the device's drafts from the
    step before; the head's KV layer carries over between cycles."""
    p = _pair([(64, 4)], kv_q8=kv_q8)
    tok, pos, sid = p.wl.rows([[1, 2, 3]])
    accepted = []
    for _ in range(3):
        drafts, co, cg, emitted = _check_step(p, tok, pos, sid)
        if co != cg:
            pytest.skip("near-tie changed the accepted length; the loops diverge")
        accepted.append(co[0] - 1)
        # next cycle: the bonus token (last emitted) at the new length, then the head's drafts
        start = int(p.eng.seq_get(0)["length"])
        tok = np.array([int(emitted[-1])] + [int(d) for d in drafts[0]], np.int32)
        pos = np.arange(start, start + 4, dtype=np.int32)
        sid = np.zeros(4, np.int32)
    print("accepted drafts per cycle:", accepted)


def test_mtp_three_sequences_q8_shuffled(cuda_ok):
    seqs = [(100, 4), (37, 4), (64, 4)]
    p = _pair(seqs, kv_q8=1, shuffle=5)
    drafts = []
    for s in range(3):
        g = greedy_continuation("tiny", 4, seq=s, overrides=dict(model=MTP_TINY, kv_q8=1, seqs=seqs, shuffle_seed=5,
                                                                  n_pages=p.wl.n_pages))
        drafts.append(drafts_with_mismatch(g, 4, s, 2048, salt=s))
    tok, pos, sid = p.wl.rows(drafts)
    _check_step(p, tok, pos, sid)


def test_mtp_draft_positions_cross_a_page(cuda_ok):
    """Rows at 60..63 end page 3; the draft passes write 64.. on a new page."""
    greedy = greedy_continuation("tiny", 4, overrides=dict(model=MTP_TINY, seqs=[(60, 4)]))
    p = _pair([(60, 4)])
    tok, pos, sid = p.wl.rows([drafts_with_mismatch(greedy, 4, 3, 2048)])
    _, co, cg, _ = _check_step(p, tok, pos, sid)
    assert co == cg == [4]
