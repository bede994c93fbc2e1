"""Pins of the oracle's speculative SAMPLING verification (orc_sample_verify)
against what the mathematics fixes, not against its own formula:

- top_k = 1 is greedy verification (brute force: the longest prefix of
  drafts equal to each row's argmax, then that row's argmax), at any
  temperature and for any uniforms;
- the emitted text keeps the distribution of sampling without drafts (page
  "UPDATE: Qwen 3.8 27B 140 tok/s on single RTX 3090 Megakernel: KL
  divergence 0.0009 vs llama.cpp", section "Decode accuracy"): over seeded
  uniforms, the first emitted token follows the target distribution p_0 of
  row 0 (tempered softmax over its top_k logits, computed here with numpy),
  (first = d_0, second = y) follows p_0(d_0) p_1(y), and (d_0, d_1, z)
  follows p_0(d_0) p_1(d_1) p_2(z);
- no token outside a row's top_k is ever emitted;
- planted mistakes (the residual keeping the rejected draft; the bonus drawn
  from the wrong row) fail the distribution pin."""
import numpy as np
import pytest

from oracle import oracle as orc


def _target(row, temperature, k):
    order = np.argsort(-row, kind="stable")[:k]
    p = np.zeros_like(row)
    z = np.exp(row[order] / temperature - row[order[0]] / temperature)
    p[order] = z / z.sum()
    return p


def test_top1_is_greedy_verification():
    rng = np.random.default_rng(1)
    for trial in range(200):
        T, V = int(rng.integers(1, 6)), int(rng.integers(2, 40))
        lg = rng.standard_normal((T, V))
        g = [int(np.argmax(lg[i])) for i in range(T)]
        # drafts: the greedy token, up to a random mismatch
        cut = int(rng.integers(0, T))
        drafts = [g[i] if i < cut else int((g[i] + 1 + rng.integers(0, V - 1)) % V) for i in range(T - 1)]
        a = 0
        while a < T - 1 and drafts[a] == g[a]:
            a += 1
        want = drafts[:a] + [g[a]]
        for temperature in (0.05, 0.6, 3.0):
            got = orc.sample_verify(lg, drafts, temperature, 1, rng.random((T, 2)))
            assert got == want, (trial, temperature, got, want)


def _sample_many(lg, drafts, temperature, k, n, seed, library=None):
    rng = np.random.default_rng(seed)
    T = lg.shape[0]
    return [orc.sample_verify(lg, drafts, temperature, k, rng.random((T, 2)), library=library) for _ in range(n)]


LOGITS = np.array([[1.2, 0.3, -0.4, 2.0, 0.9, -1.5],
                   [0.1, 1.7, 0.5, -0.2, 1.1, 0.0],
                   [-0.6, 0.4, 1.9, 0.8, -1.0, 1.3]])
DRAFTS = [4, 1]  # row 0 proposes token 4 (neither its best nor its worst), row 1 proposes 1
TEMP, K, N = 0.6, 4, 120_000


def _check_distribution(outs):
    p0 = _target(LOGITS[0], TEMP, K)
    p1 = _target(LOGITS[1], TEMP, K)
    first = np.bincount([o[0] for o in outs], minlength=6) / len(outs)
    second = np.bincount([o[1] for o in outs if o[0] == DRAFTS[0] and len(o) > 1], minlength=6) / len(outs)
    tol = lambda p: 6 * np.sqrt(p * (1 - p) / len(outs)) + 1e-12  # noqa: E731
    assert np.all(np.abs(first - p0) <= tol(p0)), (first, p0)
    joint = p0[DRAFTS[0]] * p1
    assert np.all(np.abs(second - joint) <= tol(joint)), (second, joint)
    # both drafts accepted, then the bonus from row 2
    p2 = _target(LOGITS[2], TEMP, K)
    third = np.bincount([o[2] for o in outs if len(o) == 3], minlength=6) / len(outs)
    joint3 = p0[DRAFTS[0]] * p1[DRAFTS[1]] * p2
    assert np.all(np.abs(third - joint3) <= tol(joint3)), (third, joint3)


def test_sampling_keeps_the_target_distribution():
    outs = _sample_many(LOGITS, DRAFTS, TEMP, K, N, seed=2)
    _check_distribution(outs)
    # nothing outside a row's top_k
    allowed = [set(np.argsort(-LOGITS[i], kind="stable")[:K]) for i in range(3)]
    for o in outs:
        for j, x in enumerate(o):
            assert x in allowed[j], (o, j)


@pytest.mark.parametrize("mistake", ["residual_keeps_draft", "bonus_from_wrong_row"])
def test_planted_mistakes_fail_the_distribution_pin(tmp_path, mistake):
    subs = {
        "residual_keeps_draft": [("        p[d] = 0;\n", "")],
        "bonus_from_wrong_row": [("    topk_probs(logits + static_cast<size_t>(T - 1) * V, V, temperature, top_k, p);",
                                  "    topk_probs(logits, V, temperature, top_k, p);")],
    }[mistake]
    lib = orc.build_variant(subs, str(tmp_path))
    outs = _sample_many(LOGITS, DRAFTS, TEMP, K, N, seed=2, library=lib)
    with pytest.raises(AssertionError):
        _check_distribution(outs)
