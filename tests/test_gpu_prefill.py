"""Prompt (prefill) rows on the device against the fp64 oracle: rows taken as
given with no verification, the state committed through the last row, one
token emitted when the rows end the prompt. A longer prompt is fed as several
steps of up to MK_MAX_T rows. Every test drives the CUDA path through the C
ABI (libmk.so via ctypes)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

from helpers import Pair, drafts_with_mismatch, greedy_continuation  # noqa: E402
from gen import configs  # noqa: E402


def _prompt(n, vocab, seed=9):
    return [int(x) for x in np.random.default_rng(seed).integers(0, vocab, n)]


@pytest.mark.parametrize("kv_q8", [0, 1])
def test_prompt_chunks_then_verify(cuda_ok, kv_q8):
    """16 cached tokens, a 16-token prompt in two steps of 8 rows (the second
    ends the prompt and emits a token), then a verify step from that token."""
    p = Pair("tiny", overrides=dict(seqs=[(16, 4)], kv_q8=kv_q8, n_pages=64))
    V = p.wl.model["vocab"]
    prompt = _prompt(16, V)
    emitted = None
    for c in range(2):
        tok = np.array(prompt[8 * c:8 * c + 8], np.int32)
        pos = np.arange(16 + 8 * c, 24 + 8 * c, dtype=np.int32)
        sid = np.zeros(8, np.int32)
        flags = np.array([1] * 7 + [2 if c == 1 else 1], np.uint8)
        ro, rg = p.step(tok, pos, sid, flags)
        p.compare_step(ro, rg, sid, flags)
        assert list(rg["counts"]) == [1 if c == 1 else 0]
        p.compare_kv(0, pos.tolist())
        p.compare_state(0)  # committed through the last row by the step itself
        if c == 1:
            emitted = int(rg["tokens"][0])
            assert emitted == int(ro["argmax"][7])
    tok = np.array([emitted, 5, 6, 7], np.int32)
    pos = np.arange(32, 36, dtype=np.int32)
    sid = np.zeros(4, np.int32)
    ro, rg = p.step(tok, pos, sid)
    p.compare_step(ro, rg, sid)
    co, cg = int(ro["counts"][0]), int(rg["counts"][0])
    p.oracle.commit([0], [co])
    p.eng.commit([0], [cg])
    if co == cg:
        p.compare_state(0)


def test_prompt_rows_beside_verify_rows(cuda_ok):
    """One launch: a verified sequence (T = 4, two drafts accepted) and eight
    prompt rows of another sequence that end its prompt (12 rows)."""
    seqs = [(64, 4), (16, 8)]
    greedy = greedy_continuation("tiny", 4, overrides=dict(seqs=seqs, n_pages=64))
    p = Pair("tiny", overrides=dict(seqs=seqs, n_pages=64))
    V = p.wl.model["vocab"]
    d = drafts_with_mismatch(greedy, 4, 2, V)
    tok = np.array([int(p.wl.first_tokens[0])] + d + _prompt(8, V, seed=11), np.int32)
    pos = np.array(list(range(64, 68)) + list(range(16, 24)), np.int32)
    sid = np.array([0] * 4 + [1] * 8, np.int32)
    flags = np.array([0] * 4 + [1] * 7 + [2], np.uint8)
    ro, rg = p.step(tok, pos, sid, flags)
    p.compare_step(ro, rg, sid, flags)
    assert list(rg["counts"]) == [3, 1]
    p.compare_kv(0, list(range(64, 68)))
    p.compare_kv(1, list(range(16, 24)))
    p.compare_state(1)
    p.oracle.commit([0], [3])
    p.eng.commit([0], [3])
    p.compare_state(0)


def test_prompt_row_errors(cuda_ok):
    """Host-side checks, before any device work."""
    from speculative_decode_persistent_gb300 import mk
    p = Pair("tiny", overrides=dict(seqs=[(16, 4)], n_pages=64))
    tok = np.array([1, 2, 3, 4], np.int32)
    pos = np.arange(16, 20, dtype=np.int32)
    sid = np.zeros(4, np.int32)
    for flags in ([2, 1, 1, 1], [1, 0, 1, 1], [3, 3, 3, 3]):
        with pytest.raises(mk.MkError) as e:
            p.eng.step(tok, pos, sid, flags=np.array(flags, np.uint8))
        assert e.value.status == -1, flags
    model = dict(configs.TINY, has_mtp=1, draft_vocab=1024)
    q = Pair("tiny", overrides=dict(model=model, seqs=[(16, 4)], n_draft=3, n_pages=64))
    with pytest.raises(mk.MkError) as e:
        q.eng.step(tok, pos, sid, flags=np.array([1, 1, 1, 2], np.uint8))
    assert e.value.status == -8
    ro, rg = p.step(tok, pos, sid, np.array([1, 1, 1, 2], np.uint8))
    p.compare_step(ro, rg, sid, np.array([1, 1, 1, 2], np.uint8))
