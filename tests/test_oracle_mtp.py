"""Pins of the oracle's multi-token-prediction (MTP) draft head.

The drafts for the next cycle come from catch-up rows over the accepted rows
followed by chained one-row passes. This reading follows the "Fusing the whole
speculative-decoding cycle into one CUDA kernel" page, section "What shipped".
Each test pins one part of it to something other than the oracle's own code:
  - a closed form (the block made exactly the identity by zero output
    projections; the rest is numpy matmuls and the textbook RMSNorm);
  - invariance of the drafts and of the MTP KV layer under splitting the
    accepted rows over steps;
  - the exact set of KV positions written;
  - the main model's outputs being untouched by the head.
"""
import numpy as np
import pytest

from gen import configs
from gen.workload import Workload
from oracle import oracle as orc

MTP_TINY = dict(configs.TINY, name="tiny-4L-h256-mtp", has_mtp=1, draft_vocab=1024)
CACHED = 64


def _oracle(model=MTP_TINY, n_draft=3, kv_q8=0, seqs=None, edit=None, cached=CACHED):
    wl = Workload("tiny", norm_jitter=0.1,
                  overrides=dict(model=model, kv_q8=kv_q8, n_pages=64, seqs=seqs or [(cached, 1 + n_draft)]))
    if edit:
        edit(wl.weights)
    o = orc.Oracle(wl.model, wl.weights, wl.pool, wl.kv_q8, wl.n_pages, wl.max_seqs, nthreads=2,
                   n_draft=n_draft if model.get("has_mtp") else 0)
    for s in range(len(wl.seqs)):
        o.seq_set(s, wl.seqs[s][0], wl.tables[s], *wl.states[s])
    return wl, o


def _greedy(n, **kw):
    """Greedy continuation of sequence 0, one single-row step at a time."""
    wl, o = _oracle(**kw)
    toks = [int(wl.first_tokens[0])]
    for j in range(n):
        r = o.step([toks[-1]], [CACHED + j], [0])
        o.commit([0], [1])
        toks.append(int(r["argmax"][0]))
    return toks


def _rms(x, g, eps):
    return x / np.sqrt(np.mean(x * x) + eps) * g


def _zero_block_outputs(w):
    """Zero Q4 blocks decode to exactly 0: the block's attention and FFN then add
    exactly 0 to the residual stream and the block is the identity."""
    w["mtp.block.w_o"] = np.zeros_like(w["mtp.block.w_o"])
    w["mtp.block.w_down"] = np.zeros_like(w["mtp.block.w_down"])


def test_zero_q4_block_decodes_to_zero():
    assert not np.any(orc.q4_decode(np.zeros((3, 144), np.uint8)))


@pytest.mark.parametrize("n_draft,accept", [(3, 0), (3, 2), (1, 1), (3, 3)])
def test_identity_block_closed_form(n_draft, accept):
    """With the block the identity, draft j is argmax over the first draft_vocab
    rows of E RMSNorm_f(x_j), with x_1 = W_fc [RMSNorm_h(h_a); RMSNorm_e(E[g_a])]
    and x_{j+1} = W_fc [RMSNorm_h(x_j); RMSNorm_e(E[draft_j])]. Here h_a is the
    main model's final hidden state of the last accepted row (before the final
    norm) and g_a its greedy token."""
    T = 1 + n_draft
    greedy = _greedy(T, n_draft=n_draft, edit=_zero_block_outputs)
    drafts = greedy[1:1 + accept] + [(greedy[1 + accept] + 1) % 2048] + greedy[2 + accept:T]
    drafts = drafts[:n_draft]
    wl, o = _oracle(n_draft=n_draft, edit=_zero_block_outputs)
    r = o.step([greedy[0]] + drafts, list(range(CACHED, CACHED + T)), [0] * T, want_hidden=True)
    a = int(r["counts"][0]) - 1
    assert a == min(accept, n_draft)
    m, w = wl.model, wl.weights
    H, DV, eps = m["hidden"], m["draft_vocab"], m["eps"]
    E = orc.q4_decode(w["embed"]).reshape(m["vocab"], H)
    fc = orc.q4_decode(w["mtp.fc"]).reshape(H, 2 * H)
    nh, ne, nf = (w[k].astype(np.float64) for k in ("mtp.norm_h", "mtp.norm_e", "mtp.final_norm"))
    d = o.drafts(0)
    h, tok = r["hidden"][a], int(r["argmax"][a])
    for j in range(n_draft):
        x = fc @ np.concatenate([_rms(h, nh, eps), _rms(E[tok], ne, eps)])
        logits = E[:DV] @ _rms(x, nf, eps)
        assert np.max(np.abs(d["logits"][j] - logits)) <= 1e-12 * np.max(np.abs(logits))
        assert np.max(np.abs(d["hidden"][j] - x)) <= 1e-12 * np.max(np.abs(x))
        srt = np.sort(logits)
        assert srt[-1] - srt[-2] > 1e-9  # no tie to resolve
        assert int(d["tokens"][j]) == int(np.argmax(logits))
        h, tok = x, int(d["tokens"][j])


@pytest.mark.parametrize("kv_q8", [0, 1])
def test_drafts_invariant_to_step_partition(kv_q8):
    """Three accepted rows verified in one 4-row step (third draft wrong) leave
    the same drafts, draft logits and MTP KV layer as the same three tokens
    verified one row per step: catch-up runs over exactly the accepted rows, each
    with its next token, and the draft passes continue from the last one."""
    g = _greedy(4, kv_q8=kv_q8)
    wl, one = _oracle(kv_q8=kv_q8)
    r = one.step([g[0], g[1], g[2], (g[3] + 7) % 2048], [64, 65, 66, 67], [0] * 4)
    assert int(r["counts"][0]) == 3
    da = one.drafts(0)
    wl2, seq = _oracle(kv_q8=kv_q8)
    for j in range(3):
        rj = seq.step([g[j]], [64 + j], [0])
        assert rj["tokens"].tolist() == [g[j + 1]]
        if j < 2:
            seq.commit([0], [1])
    db = seq.drafts(0)
    assert da["tokens"].tolist() == db["tokens"].tolist()
    for j in range(3):
        assert np.max(np.abs(da["logits"][j] - db["logits"][j])) <= 1e-12 * np.max(np.abs(db["logits"][j]))
    mtp_layer = configs.model_dims(MTP_TINY)["n_fa"]
    for key in (("k", "v") if not kv_q8 else ("kq", "vq", "ks", "vs")):
        assert np.array_equal(wl.pool[key][mtp_layer], wl2.pool[key][mtp_layer]), key


@pytest.mark.parametrize("kv_q8", [0, 1])
def test_kv_write_set(kv_q8):
    """The main attention layer is written at the step's T positions; the MTP
    layer at the accepted positions p_0..p_a plus the draft passes' positions
    p_a+1..p_a+n_draft-1; nothing else changes."""
    g = _greedy(4, kv_q8=kv_q8)
    wl, o = _oracle(kv_q8=kv_q8)
    key = "k" if not kv_q8 else "kq"
    before = wl.pool[key].copy()
    r = o.step([g[0], g[1], (g[2] + 3) % 2048, 5], [64, 65, 66, 67], [0] * 4)
    a = int(r["counts"][0]) - 1
    assert a == 1
    changed = np.any(wl.pool[key] != before, axis=(2, 4))  # [layer][page][slot]
    pages = o.seq_get(0)["pages"]
    n_fa = configs.model_dims(MTP_TINY)["n_fa"]

    def slots(layer):
        out = set()
        for pi, page in enumerate(pages):
            for s in np.nonzero(changed[layer, page])[0]:
                out.add(pi * 16 + int(s))
        assert not np.any(np.delete(changed[layer], pages, axis=0))  # pages outside the table untouched
        return out

    assert slots(0) == {64, 65, 66, 67}
    assert slots(n_fa) == set(range(64, 64 + a + 3))


def test_main_outputs_unchanged_by_head():
    """The verify result, logits and committed state of a model with the head
    equal those of the same model without it."""
    g = _greedy(4)
    toks = [g[0], g[1], g[2], (g[3] + 11) % 2048]
    _, with_head = _oracle()
    _, without = _oracle(model=dict(MTP_TINY, has_mtp=0, draft_vocab=0))
    r1 = with_head.step(toks, [64, 65, 66, 67], [0] * 4, want_hidden=True)
    r2 = without.step(toks, [64, 65, 66, 67], [0] * 4, want_hidden=True)
    for k in ("tokens", "counts", "logits", "hidden", "argmax"):
        assert np.array_equal(r1[k], r2[k]), k
    c = int(r1["counts"][0])
    with_head.commit([0], [c])
    without.commit([0], [c])
    s1, s2 = with_head.seq_get(0), without.seq_get(0)
    for k in ("length", "pages"):
        assert np.array_equal(s1[k], s2[k]), k
    assert np.array_equal(s1["S"], s2["S"]) and np.array_equal(s1["conv"], s2["conv"])


def test_draft_pages_reserved_and_released():
    """Rows at 60..63 fill page 3; the draft passes may reach 63 + 2, so page 4
    is reserved for the step and freed by a commit that stays within page 3."""
    wl, o = _oracle(seqs=[(60, 4)], cached=60)
    assert o.seq_get(0)["pages"].tolist() == [0, 1, 2, 3]
    free0 = o.n_free_pages()
    r = o.step([int(wl.first_tokens[0]), 1, 2, 3], [60, 61, 62, 63], [0] * 4)
    assert o.seq_get(0)["pages"].tolist() == [0, 1, 2, 3, 4]
    assert o.n_free_pages() == free0 - 1
    o.commit([0], [int(r["counts"][0])])
    assert o.seq_get(0)["pages"].tolist() == [0, 1, 2, 3]
    assert o.n_free_pages() == free0


def test_rejects_bad_draft_vocab():
    with pytest.raises(ValueError):
        _oracle(model=dict(MTP_TINY, draft_vocab=4096))
