"""The allocation-free step entry point (mk_step_static) against mk_step.

Callers that cannot allocate device memory while they step use
mk_step_static; it must give the same tokens, counts and logits as mk_step on
the same inputs, two steps in a row (the second reuses the shared static
scratch left by the first). Collected last so that a failure here comes after
every other test has run."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

from helpers import LOGIT_TOL, Pair  # noqa: E402


def test_step_static_matches_step_twice(cuda_ok):
    a = Pair("tiny")
    b = Pair("tiny")
    tok, pos, sid = a.wl.rows([[7, 11, 13]])
    for _ in range(2):
        ta, ca = a.eng.step(tok, pos, sid)
        la = a.logits[: len(tok)].double().cpu().numpy()
        tb, cb = b.eng.step_static(tok, pos, sid)
        lb = b.logits[: len(tok)].double().cpu().numpy()
        assert np.array_equal(ta, tb) and np.array_equal(ca, cb)
        rms = np.sqrt(np.mean(la ** 2, axis=1))
        assert np.all(np.max(np.abs(la - lb), axis=1) <= LOGIT_TOL * rms)
        # next step: bonus token at the new length, fresh drafts
        c = int(ca[0])
        tok = np.array([int(ta[c - 1]), 3, 5, 8], np.int32)
        pos = np.arange(int(pos[0]) + c, int(pos[0]) + c + 4, dtype=np.int32)
    sa, sb = a.eng.seq_get(0), b.eng.seq_get(0)
    assert sa["length"] == sb["length"] and np.array_equal(sa["pages"], sb["pages"])
