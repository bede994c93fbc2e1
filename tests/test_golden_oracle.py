"""The oracle still reproduces its stored regression fixture
(tests/golden/tiny_oracle_step.json, written by tests/golden/make_golden.py
from gen/ and oracle/ only): tokens, counts and argmax exactly, floating
point to 1e-12 relative."""
import importlib.util
import json
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def _make_golden():
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(HERE, "golden", "make_golden.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def test_oracle_matches_stored_fixture():
    stored = json.load(open(os.path.join(HERE, "golden", "tiny_oracle_step.json")))
    now = _make_golden().build()
    assert stored.keys() == now.keys()
    for case in stored:
        a, b = stored[case], now[case]
        for k in ("tokens", "positions", "emitted", "counts", "argmax", "drafts"):
            assert a.get(k) == b.get(k), (case, k)
        for k in ("gap", "rms", "logits_head", "hidden_head", "draft_gap", "draft_logits_head"):
            if k in a:
                x, y = np.asarray(a[k]), np.asarray(b[k])
                assert np.allclose(x, y, rtol=1e-12, atol=1e-15), (case, k)
