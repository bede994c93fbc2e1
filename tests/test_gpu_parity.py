"""GPU verify step vs the fp64 CPU oracle on identical seeded inputs.

Every test drives the CUDA path through the C ABI (libmk.so via ctypes)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

from helpers import Pair, drafts_with_mismatch, greedy_continuation  # noqa: E402


@pytest.mark.parametrize("kv_q8", [0, 1])
@pytest.mark.parametrize("m", [0, 1, 2, 3])
def test_tiny_verify_accept_lengths(cuda_ok, kv_q8, m):
    """Tiny hybrid decoder, one sequence, 64 cached tokens, T = 1 + 3 rows,
    drafts = the oracle's greedy continuation with one mismatch at index m."""
    ov = dict(kv_q8=kv_q8)
    greedy = greedy_continuation("tiny", 4, overrides=ov)
    p = Pair("tiny", overrides=ov)
    wl = p.wl
    d = drafts_with_mismatch(greedy, 4, m, wl.model["vocab"], salt=m)
    tok, pos, sid = wl.rows([d])
    ro, rg = p.step(tok, pos, sid)
    excused, rep = p.compare_step(ro, rg, sid)
    assert excused == 0
    assert int(ro["counts"][0]) == m + 1
    # commit what was accepted; compare the committed recurrent state and the KV writes
    p.oracle.commit([0], [m + 1])
    p.eng.commit([0], [m + 1])
    p.compare_state(0)
    p.compare_kv(0, list(pos[: m + 1]))


@pytest.mark.parametrize("kv_q8", [0, 1])
def test_tiny_multi_seq_shuffled_pages_multi_step(cuda_ok, kv_q8):
    """Three sequences with different cached lengths and row counts on a
    shuffled page pool; several consecutive steps with auto-commit, then an
    explicit partial commit."""
    ov = dict(kv_q8=kv_q8, n_pages=96, seqs=[(37, 3), (64, 4), (5, 2)], shuffle_seed=3)
    p = Pair("tiny", overrides=ov)
    wl = p.wl
    rng = np.random.default_rng(11)
    tok, pos, sid = wl.rows([list(rng.integers(0, 2048, T - 1)) for (_c, T) in wl.seqs])
    for step in range(3):
        ro, rg = p.step(tok, pos, sid)
        p.compare_step(ro, rg, sid)
        for s in range(len(wl.seqs)):
            p.compare_kv(s, [int(x) for x, q in zip(pos, sid) if q == s])
        # next rows: bonus token of each sequence + random drafts
        new_tok, new_pos, new_sid = [], [], []
        at = 0
        for i, (cached, T) in enumerate(wl.seqs):
            c = int(ro["counts"][i])
            bonus = int(ro["tokens"][at + c - 1])
            at += c
            base = int(pos[np.asarray(sid) == i][0]) + c
            row_tokens = [bonus] + [int(x) for x in rng.integers(0, 2048, T - 1)]
            new_tok += row_tokens
            new_pos += list(range(base, base + T))
            new_sid += [i] * T
        tok, pos, sid = np.array(new_tok), np.array(new_pos), np.array(new_sid)
    ro, rg = p.step(tok, pos, sid)
    p.compare_step(ro, rg, sid)
    p.oracle.commit([0, 1, 2], [1, 1, 1])
    p.eng.commit([0, 1, 2], [1, 1, 1])
    for s in range(3):
        p.compare_state(s)


def test_tiny_repeated_launch_is_idempotent(cuda_ok):
    """Launching the same prepared step twice gives the same tokens (the
    benchmark times repeated launches of one prepared step)."""
    p = Pair("tiny")
    tok, pos, sid = p.wl.rows([[1, 2, 3]])
    p.eng.prepare(tok, pos, sid)
    p.eng.launch()
    p.eng.launch()
    t1, c1 = p.eng.finish()
    p2 = Pair("tiny")
    t2, c2 = p2.eng.step(tok, pos, sid)
    assert np.array_equal(t1, t2) and np.array_equal(c1, c2)
