"""Failure detection without a GPU fault: one block skips its arrival at a
grid barrier; every other block's bounded wait expires, the step returns
MK_ERR_BARRIER_TIMEOUT, no sequence becomes pending, and the next step on the
same context succeeds. Host-side faults return their status before any
device work."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

from helpers import Pair  # noqa: E402


def test_barrier_timeout_then_recovery(cuda_ok):
    from speculative_decode_persistent_gb300 import mk
    p = Pair("tiny")
    tok, pos, sid = p.wl.rows([[1, 2, 3]])
    p.eng.skip_arrival(block=3, barrier=5, timeout_ns=50_000_000)
    with pytest.raises(mk.MkError) as e:
        p.eng.step(tok, pos, sid)
    assert e.value.status == -4
    with pytest.raises(mk.MkError) as e:
        p.eng.commit([0], [1])
    assert e.value.status == -5  # nothing pending after a failed step
    p.eng.skip_arrival(-1, -1, 0)
    ro, rg = p.step(tok, pos, sid)
    p.compare_step(ro, rg, sid)


def test_host_side_errors(cuda_ok):
    from speculative_decode_persistent_gb300 import mk
    p = Pair("tiny", overrides=dict(n_pages=5))  # 64 cached tokens use 4 of 5 pages
    tok, pos, sid = p.wl.rows([[1, 2, 3]])
    with pytest.raises(mk.MkError) as e:  # wrong position
        p.eng.step(tok, pos + 1, sid)
    assert e.value.status == -1
    with pytest.raises(mk.MkError) as e:  # unknown sequence
        p.eng.step(tok, pos, np.array([5, 5, 5, 5]))
    assert e.value.status == -1
    # 64 + 20 rows would need 6 pages: refused before any device work
    long_tok = np.zeros(12, np.int32)
    with pytest.raises(mk.MkError):
        p.eng.step(long_tok, np.arange(64, 76), np.zeros(12, np.int32))
    ro, rg = p.step(tok, pos, sid)
    p.compare_step(ro, rg, sid)


@pytest.mark.parametrize("barrier", [26, 31, 35])
def test_barrier_timeout_inside_draft_passes(cuda_ok, barrier):
    """The same recovery when the skipped arrival falls inside the MTP head's
    passes. On the 4-layer model the main step uses barriers 0..22 (22 closes
    verify); each draft pass then has nine. 26 is pass 0's attention, 31 its
    draft phase, and 35 the attention of pass 1, which reads back earlier
    draft positions."""
    from speculative_decode_persistent_gb300 import mk
    from gen import configs
    model = dict(configs.TINY, has_mtp=1, draft_vocab=1024)
    p = Pair("tiny", overrides=dict(model=model, n_draft=3, n_pages=72))
    tok, pos, sid = p.wl.rows([[1, 2, 3]])
    p.eng.skip_arrival(block=3, barrier=barrier, timeout_ns=50_000_000)
    with pytest.raises(mk.MkError) as e:
        p.eng.step(tok, pos, sid)
    assert e.value.status == -4
    with pytest.raises(mk.MkError) as e:
        p.eng.last_drafts(1)
    assert e.value.status == -1  # no drafts from a failed step
    p.eng.skip_arrival(-1, -1, 0)
    ro, rg = p.step(tok, pos, sid)
    p.compare_step(ro, rg, sid)
    co, cg = int(ro["counts"][0]), int(rg["counts"][0])
    p.compare_drafts([0], [co == cg])
