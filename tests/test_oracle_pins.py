"""Pins of the CPU oracle to things other than itself.

Each test checks one oracle function against a closed form, a library routine
(numpy / torch fp64), an invariant, or brute force, chosen so that a dropped
term, a wrong sign or index, or a transposed operand fails one of them.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import gen
from gen import configs
from gen.workload import Workload
from oracle import oracle as orc

# ----------------------------------------------------------------- binary16


def test_half_round_matches_numpy():
    rng = np.random.default_rng(0)
    xs = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 5, 20000),
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                  2.0 ** -14, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, -1e9]),
    ])
    for x in xs:
        with np.errstate(over="ignore"):
            want = int(np.array(x, np.float64).astype(np.float16).view(np.uint16))
        assert orc.half_round(float(x)) == want, x


def test_half_value_all_finite_patterns():
    bits = np.arange(0, 0x7c00, dtype=np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.half_value(int(b)) for b in bits[::7]])
    assert np.array_equal(got, want[::7])
    assert orc.half_value(0x8001) == -(2.0 ** -24)


# ---------------------------------------------------------------------- Q4


def _hand_block(d_bits, dmin_bits, sc, mn, codes):
    """Pack one super-block straight from the format description: binary16 d
    and dmin, 6-bit scales at bit 6j and mins at bit 48+6j of a little-endian
    96-bit field, then sub-block j's 32 codes in 16 bytes (element i: low
    nibble of byte i for i < 16, high nibble of byte i-16 otherwise)."""
    blk = bytearray(144)
    blk[0:2] = int(d_bits).to_bytes(2, "little")
    blk[2:4] = int(dmin_bits).to_bytes(2, "little")
    field = 0
    for j in range(8):
        field |= (sc[j] & 63) << (6 * j)
        field |= (mn[j] & 63) << (48 + 6 * j)
    blk[4:16] = field.to_bytes(12, "little")
    for j in range(8):
        for i in range(32):
            q = codes[j][i] & 15
            if i < 16:
                blk[16 + 16 * j + i] |= q
            else:
                blk[16 + 16 * j + i - 16] |= q << 4
    return np.frombuffer(bytes(blk), np.uint8)


def test_q4_decode_known_codes():
    # d = 0.5 (0x3800), dmin = 0.25 (0x3400); distinct scales, mins and codes
    sc = [1, 2, 3, 5, 8, 13, 21, 63]
    mn = [0, 1, 4, 9, 16, 25, 36, 63]
    codes = [[(i * (j + 3) + j) % 16 for i in range(32)] for j in range(8)]
    blk = _hand_block(0x3800, 0x3400, sc, mn, codes)
    w = orc.q4_decode(blk)
    want = np.array([0.5 * sc[j] * codes[j][i] - 0.25 * mn[j] for j in range(8) for i in range(32)])
    assert np.array_equal(w, want)


def test_q4_decode_subnormal_scale():
    sc = [63] * 8
    mn = [0] * 8
    codes = [[15] * 32 for _ in range(8)]
    blk = _hand_block(0x0001, 0x0000, sc, mn, codes)  # d = 2^-24
    assert np.all(orc.q4_decode(blk) == 63 * 15 * 2.0 ** -24)


def test_q4_roundtrip_exact_codes():
    """Weights that are exactly representable with the chosen d, dmin, scales
    and codes quantise back to those same codes."""
    d, dmin = 2.0 ** -7, 2.0 ** -8
    sc = [63, 60, 62, 61, 63, 59, 63, 58]
    mn = [63, 63, 10, 0, 40, 63, 1, 5]
    rng = np.random.default_rng(3)
    codes = [[int(c) for c in rng.integers(0, 16, 32)] for _ in range(8)]
    for j in range(8):  # every sub-block spans its full range
        codes[j][0], codes[j][1] = 0, 15
    w = np.array([d * sc[j] * codes[j][i] - dmin * mn[j] for j in range(8) for i in range(32)])
    blk = orc.q4_encode(w)[0]
    dec = orc.q4_decode(blk)
    assert np.allclose(dec, w, atol=0.51 * d * 63)
    # sub-blocks whose step equals the super-block max step reproduce exactly
    for j in (0, 4, 6):
        assert np.array_equal(dec[32 * j:32 * j + 32], w[32 * j:32 * j + 32])


def test_q4_quantisation_error_bound():
    w = gen.normal_f64(0, 77, 256 * 64, sigma=0.02).reshape(-1, 256)
    blocks = orc.q4_encode(w)
    dec = orc.q4_decode(blocks).reshape(-1, 256)
    for b in range(w.shape[0]):
        steps = []
        for j in range(8):
            sub = w[b, 32 * j:32 * j + 32]
            steps.append((sub.max() - min(0.0, sub.min())) / 15)
        assert np.max(np.abs(dec[b] - w[b])) <= 1.05 * max(steps)


def test_q4_matvec_equals_numpy_matmul():
    rows, k = 40, 768
    W = gen.q4_matrix(1, 5, rows, k, 0.02)
    dense = orc.q4_decode(W).reshape(rows, k)
    u = np.random.default_rng(1).standard_normal(k)
    y = orc.q4_matvec(W, k, u, nthreads=3)
    want = dense @ u
    assert np.max(np.abs(y - want)) <= 1e-12 * np.max(np.abs(want))


# ---------------------------------------------------------------------- q8


def test_q8_known_codes():
    d16 = 0x2C00  # 1/16
    d = orc.half_value(d16)
    q = np.array(list(range(-15, 16)) + [127], np.int8)  # amax code 127
    x = d * q.astype(np.float64)
    # amax/127 = d exactly, so encode reproduces d and the codes
    cq, cd = orc.q8_encode(x)
    assert cd[0] == d16
    assert np.array_equal(cq[0], q)


def test_q8_zero_and_bounds():
    cq, cd = orc.q8_encode(np.zeros(32))
    assert cd[0] == 0 and not cq.any()
    x = np.random.default_rng(2).standard_normal((50, 32)) * 3
    cq, cd = orc.q8_encode(x)
    dv = np.array([orc.half_value(int(v)) for v in cd])
    assert np.all(np.abs(cq) <= 127)
    err = np.abs(x - dv[:, None] * cq)
    assert np.all(err <= dv[:, None] * 0.5 + np.abs(x).max(1, keepdims=True) * 2 ** -10)
    # the largest magnitude maps to +-127 up to the binary16 rounding of the scale
    assert np.all(np.abs(cq).max(1) >= 126)


# ------------------------------------------------------------------- small ops


def test_sigmoid_silu_closed_forms():
    assert orc.sigmoid(0.0) == 0.5
    assert orc.silu(0.0) == 0.0
    for v in (-3.0, -0.5, 0.7, 4.0):
        assert abs(orc.sigmoid(v) + orc.sigmoid(-v) - 1) < 1e-15
        assert abs(orc.silu(v) - v / (1 + math.exp(-v))) < 1e-15


def test_rmsnorm_closed_form():
    x = np.full(64, 3.0)
    g = np.linspace(0.5, 1.5, 64).astype(np.float32)
    y = orc.rmsnorm(x, g, 1e-6)
    assert np.allclose(y, 3.0 / math.sqrt(9.0 + 1e-6) * g.astype(np.float64), rtol=0, atol=1e-15)
    z = orc.rmsnorm(np.random.default_rng(0).standard_normal(100), None, 0.0)
    assert abs(np.mean(z ** 2) - 1) < 1e-12


def test_l2norm():
    x = np.array([3.0, 4.0])
    y = orc.l2norm(x, 0.0)
    assert np.allclose(y, [0.6, 0.8], atol=1e-16)
    y = orc.l2norm(x, 11.0)  # sqrt(25 + 11) = 6
    assert np.allclose(y, [0.5, 4 / 6], atol=1e-16)


def test_rope_closed_form_and_invariants():
    base = 1e7
    x = np.array([1.0, 0.0, 2.0, 1.0])  # dh = 4: pairs (0, 2) and (1, 3)
    p = 5
    y = orc.rope(x, p, base)
    t0, t1 = p * 1.0, p * base ** (-0.5)
    want = np.array([1 * math.cos(t0) - 2 * math.sin(t0), 0 * math.cos(t1) - 1 * math.sin(t1),
                     1 * math.sin(t0) + 2 * math.cos(t0), 0 * math.sin(t1) + 1 * math.cos(t1)])
    assert np.allclose(y, want, atol=1e-15)
    v = np.random.default_rng(4).standard_normal(64)
    assert np.array_equal(orc.rope(v, 0, base), v)
    assert abs(np.linalg.norm(orc.rope(v, 1234, base)) - np.linalg.norm(v)) < 1e-12
    q, k = v, np.random.default_rng(5).standard_normal(64)
    a = orc.rope(q, 40, base) @ orc.rope(k, 17, base)
    b = orc.rope(q, 23, base) @ k
    assert abs(a - b) < 1e-11


def test_attention_matches_torch_sdpa():
    rng = np.random.default_rng(6)
    n, dh = 37, 64
    q, K, V = rng.standard_normal(dh), rng.standard_normal((n, dh)), rng.standard_normal((n, dh))
    out = orc.attend(q, K, V)
    t = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None, None, None], torch.from_numpy(K)[None, None],
        torch.from_numpy(V)[None, None])[0, 0, 0].numpy()
    assert np.max(np.abs(out - t)) < 1e-13
    # one key: output is that value row; zero query: mean of the values
    assert np.allclose(orc.attend(q, K[:1], V[:1]), V[0], atol=1e-15)
    assert np.allclose(orc.attend(np.zeros(dh), K, V), V.mean(0), atol=1e-14)


# ---------------------------------------------------------------- delta rule


def _closed_form(S0, qs, ks, vs, alphas, betas):
    """S_T = S_0 prod_t A_t + sum_t beta_t v_t k_t^T prod_{s>t} A_s,
    A_t = alpha_t (I - beta_t k_t k_t^T)."""
    dk = S0.shape[1]
    A = [a * (np.eye(dk) - b * np.outer(k, k)) for a, b, k in zip(alphas, betas, ks)]
    T = len(ks)
    S = S0.copy()
    for t in range(T):
        S = S @ A[t]
    for t in range(T):
        term = betas[t] * np.outer(vs[t], ks[t])
        for s in range(t + 1, T):
            term = term @ A[s]
        S = S + term
    return S


@pytest.mark.parametrize("dk,dv,T", [(2, 2, 1), (3, 3, 2), (4, 4, 4), (3, 2, 3), (2, 4, 4)])
def test_gdn_unrolled_closed_form(dk, dv, T):
    rng = np.random.default_rng(dk * 10 + T)
    S0 = rng.standard_normal((dv, dk))
    ks = [v / np.linalg.norm(v) for v in rng.standard_normal((T, dk))]
    qs = [v / np.linalg.norm(v) for v in rng.standard_normal((T, dk))]
    vs = list(rng.standard_normal((T, dv)))
    al = list(rng.uniform(0.2, 1.0, T))
    be = list(rng.uniform(0.0, 1.0, T))
    S = S0
    for t in range(T):
        S, o = orc.gdn_update(S, qs[t], ks[t], vs[t], al[t], be[t])
        assert np.allclose(o, S @ qs[t], atol=1e-14)
    assert np.allclose(S, _closed_form(S0, qs, ks, vs, al, be), atol=1e-13)


def test_gdn_invariants():
    rng = np.random.default_rng(9)
    S0 = rng.standard_normal((4, 4))
    k = rng.standard_normal(4)
    k /= np.linalg.norm(k)
    q, v = rng.standard_normal(4), rng.standard_normal(4)
    S, _ = orc.gdn_update(S0, q, k, v, 1.0, 0.0)
    assert np.array_equal(S, S0)
    S, _ = orc.gdn_update(S0, q, k, v, 0.37, 1.0)
    assert np.allclose(S @ k, v, atol=1e-14)
    S, _ = orc.gdn_update(S0, q, k, v, 0.0, 1.0)
    assert np.allclose(S, np.outer(v, k), atol=1e-15)


# ---------------------------------------------------------------- the step


def _tiny_oracle(model=None, kv_q8=0, norm_jitter=0.1, n_pages=64, seqs=None):
    wl = Workload("tiny", norm_jitter=norm_jitter,
                  overrides=dict(model=model or configs.TINY, kv_q8=kv_q8, n_pages=n_pages,
                                 seqs=seqs or [(64, 4)]))
    o = orc.Oracle(wl.model, wl.weights, wl.pool, wl.kv_q8, wl.n_pages, wl.max_seqs, nthreads=2)
    for s in range(len(wl.seqs)):
        o.seq_set(s, wl.seqs[s][0], wl.tables[s], *wl.states[s])
    return wl, o


@pytest.mark.parametrize("kv_q8", [0, 1])
def test_T_row_pass_equals_sequential(kv_q8):
    """(a) a T-row pass equals T sequential single-row passes: the greedy
    continuation is produced one row at a time, then the same four tokens go
    through one 4-row pass, which must accept all of them with the same logits
    and leave the same committed state."""
    wl, seq = _tiny_oracle(kv_q8=kv_q8)
    toks = [int(wl.first_tokens[0])]
    seq_logits = []
    for j in range(4):
        rj = seq.step([toks[j]], [64 + j], [0])
        seq.commit([0], [1])
        seq_logits.append(rj["logits"][0])
        toks.append(int(rj["argmax"][0]))
    _, one = _tiny_oracle(kv_q8=kv_q8)
    r = one.step(toks[:4], [64, 65, 66, 67], [0] * 4)
    assert r["counts"].tolist() == [4]
    assert r["tokens"].tolist() == toks[1:5]
    for j in range(4):
        assert np.max(np.abs(seq_logits[j] - r["logits"][j])) <= 1e-12 * np.max(np.abs(r["logits"][j]))
    one.commit([0], [4])
    s1, s2 = one.seq_get(0), seq.seq_get(0)
    assert s1["length"] == s2["length"] == 68
    assert np.max(np.abs(s1["S"] - s2["S"])) <= 1e-12 * np.max(np.abs(s2["S"]))
    assert np.max(np.abs(s1["conv"] - s2["conv"])) <= 1e-12 * np.max(np.abs(s2["conv"]))


def test_replay_of_accepted_prefix_gives_committed_state():
    """(c) committing a+1 rows of a T-row step equals replaying rows 0..a."""
    wl, o1 = _tiny_oracle()
    r0 = o1.step([int(wl.first_tokens[0])], [64], [0])
    g0 = int(r0["argmax"][0])
    _, o1 = _tiny_oracle()
    toks = [int(wl.first_tokens[0]), g0, 3, 4]  # accept at least the first draft
    r = o1.step(toks, [64, 65, 66, 67], [0] * 4)
    keep = int(r["counts"][0])
    assert keep >= 2
    o1.commit([0], [keep])
    _, o2 = _tiny_oracle()
    o2.step(toks[:keep], list(range(64, 64 + keep)), [0] * keep)
    o2.commit([0], [keep])
    s1, s2 = o1.seq_get(0), o2.seq_get(0)
    assert s1["length"] == s2["length"] == 64 + keep
    assert np.array_equal(s1["S"], s2["S"])
    assert np.array_equal(s1["conv"], s2["conv"])
    assert np.array_equal(s1["pages"], s2["pages"])


def _vocab16_model(kind):
    m = dict(configs.TINY)
    m.update(name="vocab16", n_layers=1, kinds=[kind], vocab=16)
    return m


@pytest.mark.parametrize("kind", [configs.GDN, configs.FA])
def test_acceptance_equals_brute_force(kind):
    """(d) on a 16-token vocabulary, the accepted count and emitted tokens of a
    3-row step equal the brute-force reading of per-position greedy argmax,
    for every one of the 256 draft pairs."""
    model = _vocab16_model(kind)
    wl, o = _tiny_oracle(model=model, seqs=[(20, 3)])
    t0 = int(wl.first_tokens[0]) % 16
    g0 = int(o.step([t0], [20], [0])["argmax"][0])
    wl, o = _tiny_oracle(model=model, seqs=[(20, 3)])
    o.step([t0], [20], [0])
    o.commit([0], [1])
    g1 = int(o.step([g0], [21], [0])["argmax"][0])
    for d1, d2 in itertools.product(range(16), range(16)):
        wl, o = _tiny_oracle(model=model, seqs=[(20, 3)])
        r = o.step([t0, d1, d2], [20, 21, 22], [0, 0, 0])
        if d1 != g0:
            want = [g0]
        elif d2 != g1:
            want = [d1, g1]
        else:
            g2 = int(r["argmax"][2])
            want = [d1, d2, g2]
        assert r["counts"][0] == len(want)
        assert r["tokens"].tolist() == want


def test_page_allocator_rule():
    """Lowest free page id in row order; pages wholly beyond the length freed."""
    wl, o = _tiny_oracle(n_pages=8, seqs=[(20, 4), (5, 2)])
    # re-install: seq 0 on pages [3, 5] (positions 0..31), seq 1 on page [1]
    o.seq_set(0, 20, [3, 5], *wl.states[0])
    o.seq_set(1, 5, [1], *wl.states[1])
    assert o.n_free_pages() == 5
    toks = [1, 2, 3, 4]
    # seq 0: positions 20..23 inside page index 1 (16..31): no allocation
    r = o.step(toks, [20, 21, 22, 23], [0] * 4)
    assert o.seq_get(0)["pages"].tolist() == [3, 5]
    o.commit([0], [1])
    o.seq_set(0, 30, [3, 5], *wl.states[0])
    # seq 0 rows at 30..33 need page index 2 -> lowest free id 0; seq 1 rows 5,6 none
    r = o.step([1, 2, 3, 4, 7, 8], [30, 31, 32, 33, 5, 6], [0, 0, 0, 0, 1, 1])
    assert o.seq_get(0)["pages"].tolist() == [3, 5, 0]
    c0 = int(r["counts"][0])
    o.commit([0, 1], [1, 1])
    # seq 0 keeps 1 row -> length 31 -> 2 pages, page 0 is freed
    assert o.seq_get(0)["pages"].tolist() == [3, 5]
    assert o.seq_get(0)["length"] == 31
    assert o.n_free_pages() == 8 - 3
    assert c0 >= 1


def test_prefill_rows_commit_and_emit():
    wl, o = _tiny_oracle(seqs=[(16, 1)])
    toks = [3, 9, 27, 81]
    r = o.step(toks, [16, 17, 18, 19], [0] * 4, flags=[1, 1, 1, 1])
    assert r["counts"].tolist() == [0] and len(r["tokens"]) == 0
    assert o.seq_get(0)["length"] == 20
    r = o.step([5, 6], [20, 21], [0, 0], flags=[1, 2])
    assert r["counts"].tolist() == [1]
    assert r["tokens"].tolist() == [int(r["argmax"][1])]
    assert o.seq_get(0)["length"] == 22


def test_prompt_rows_invariant_to_chunking_and_batching():
    """Prompt rows (the page's chunked prefill riding along with decode rows)
    give the same committed state and emitted token whether the prompt comes
    as one 8-row step, as two 4-row steps, or beside another sequence's
    verify rows: rows of different sequences never interact, and the
    recurrence runs row by row."""
    prompt = [5, 77, 901, 13, 1500, 2, 640, 333]
    flags = [1] * 7 + [2]
    wl, one = _tiny_oracle(seqs=[(64, 4), (16, 8)], n_pages=32)
    r1 = one.step(prompt, list(range(16, 24)), [1] * 8, flags=flags)
    wl, two = _tiny_oracle(seqs=[(64, 4), (16, 8)], n_pages=32)
    two.step(prompt[:4], list(range(16, 20)), [1] * 4, flags=[1] * 4)
    r2 = two.step(prompt[4:], list(range(20, 24)), [1] * 4, flags=[1, 1, 1, 2])
    wl, mixed = _tiny_oracle(seqs=[(64, 4), (16, 8)], n_pages=32)
    r3 = mixed.step([1, 2, 3, 4] + prompt, list(range(64, 68)) + list(range(16, 24)), [0] * 4 + [1] * 8,
                    flags=[0] * 4 + flags)
    assert r1["tokens"].tolist() == r2["tokens"].tolist() == [int(r3["tokens"][-1])]
    s1, s2, s3 = one.seq_get(1), two.seq_get(1), mixed.seq_get(1)
    assert s1["length"] == s2["length"] == s3["length"] == 24
    for k in ("S", "conv"):
        assert np.max(np.abs(s1[k] - s2[k])) <= 1e-12 * np.max(np.abs(s1[k]))
        assert np.array_equal(s1[k], s3[k])
    assert np.max(np.abs(r1["logits"][7] - r2["logits"][3])) <= 1e-12 * np.max(np.abs(r1["logits"][7]))
