"""The allocation-free step entry point (mk_step_static) against mk_step.

Some callers cannot allocate device memory at the moment they step (a server
whose memory pool owns the whole GPU, an allocator that must not grow while
requests are in flight, a latency-critical loop where cudaMalloc would stall
other streams); they use mk_step_static, whose scratch lives in a static
device array. It must give the same tokens, counts and logits (within the
parity tolerance of the other tests) as mk_step on the same inputs, two steps
in a row: the second reuses the shared scratch the first left behind.
Cases: the tiny model with an fp16 and a q8 KV pool, and a two-sequence step
that puts a sequence's prompt rows beside another's verify rows. A model with
an MTP head is refused with no change to any sequence.

Collected last (file name) so that a failure here comes after every other
test has run; each case builds its own contexts, so it also passes alone in
a fresh process."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

from helpers import LOGIT_TOL, Pair  # noqa: E402
from gen import configs  # noqa: E402


def _same(a, b, tok, pos, sid, flags=None):
    ta, ca = a.eng.step(tok, pos, sid, flags=flags)
    la = a.logits[: len(tok)].double().cpu().numpy()
    tb, cb = b.eng.step_static(tok, pos, sid, flags=flags)
    lb = b.logits[: len(tok)].double().cpu().numpy()
    assert np.array_equal(ca, cb), (ca, cb)
    assert np.array_equal(ta[: int(ca.sum())], tb[: int(cb.sum())])
    rms = np.sqrt(np.mean(la ** 2, axis=1))
    assert np.all(np.max(np.abs(la - lb), axis=1) <= LOGIT_TOL * rms)
    return ta, ca


@pytest.mark.parametrize("kv_q8", [0, 1])
def test_step_static_matches_step_twice(cuda_ok, kv_q8):
    ov = dict(kv_q8=kv_q8)
    a, b = Pair("tiny", overrides=ov), Pair("tiny", overrides=ov)
    tok, pos, sid = a.wl.rows([[7, 11, 13]])
    for _ in range(2):
        ta, ca = _same(a, b, tok, pos, sid)
        # next step: bonus token at the new length, fresh drafts
        c = int(ca[0])
        tok = np.array([int(ta[c - 1]), 3, 5, 8], np.int32)
        pos = np.arange(int(pos[0]) + c, int(pos[0]) + c + 4, dtype=np.int32)
    sa, sb = a.eng.seq_get(0), b.eng.seq_get(0)
    assert sa["length"] == sb["length"] and np.array_equal(sa["pages"], sb["pages"])


def test_step_static_prompt_rows_beside_verify_rows(cuda_ok):
    """Two sequences (more attention items, other partial offsets): verify rows
    of one beside eight prompt rows of the other, then a second step."""
    ov = dict(seqs=[(64, 4), (16, 8)], n_pages=64)
    a, b = Pair("tiny", overrides=ov), Pair("tiny", overrides=ov)
    V = a.wl.model["vocab"]
    prompt = [int(x) for x in np.random.default_rng(11).integers(0, V, 16)]
    tok = np.array([int(a.wl.first_tokens[0]), 7, 11, 13] + prompt[:8], np.int32)
    pos = np.array(list(range(64, 68)) + list(range(16, 24)), np.int32)
    sid = np.array([0] * 4 + [1] * 8, np.int32)
    flags = np.array([0] * 4 + [1] * 8, np.uint8)
    for step in range(2):
        ta, ca = _same(a, b, tok, pos, sid, flags)
        c0 = int(ca[0])
        base0 = int(pos[0]) + c0
        tok = np.array([int(ta[c0 - 1]), 3, 5, 8] + prompt[8:16], np.int32)
        pos = np.array(list(range(base0, base0 + 4)) + list(range(24, 32)), np.int32)
        flags = np.array([0] * 4 + [1] * 7 + [2], np.uint8)
        if step == 1:
            break
    for s in (0, 1):
        sa, sb = a.eng.seq_get(s), b.eng.seq_get(s)
        assert sa["length"] == sb["length"] and np.array_equal(sa["pages"], sb["pages"])


def test_step_static_refuses_mtp_head_unchanged(cuda_ok):
    model = dict(configs.TINY, has_mtp=1, draft_vocab=1024)
    p = Pair("tiny", overrides=dict(model=model, n_draft=3, n_pages=72))
    before = p.eng.seq_get(0)
    tok, pos, sid = p.wl.rows([[7, 11, 13]])
    from speculative_decode_persistent_gb300 import mk
    with pytest.raises(mk.MkError) as e:
        p.eng.step_static(tok, pos, sid)
    assert e.value.status == -8  # MK_ERR_UNSUPPORTED
    after = p.eng.seq_get(0)
    assert before["length"] == after["length"] and np.array_equal(before["pages"], after["pages"])
    assert before["slot"] == after["slot"]
