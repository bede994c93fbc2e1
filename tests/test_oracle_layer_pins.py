"""Pins of the oracle's layer composition to the mathematics.

The oracle's building blocks (binary16, Q4/q8 codecs, RMSNorm, L2 norm, RoPE,
single-head attention, the delta rule) are pinned one by one elsewhere. These
tests pin how a layer puts them together, with models built so that the
answer follows from a definition and can be computed here with numpy from
the inputs alone:

* the Gated DeltaNet short causal conv: with one-hot taps (tap i = 1, the
  others 0) the conv output of a row is SiLU of the input 3 - i rows back,
  and the stored history after a row is (x_{t-2}, x_{t-1}, x_t), oldest first
  (the layout the C header documents for conv_state);
* the Gated DeltaNet head grouping: from a zero state, one row leaves each
  v-head h with the rank-one state beta_h v_h k_g^T, g = h div (hv / hk)
  (the delta rule on S = 0, with the per-row projections and the conv above);
* the gated-attention head grouping: q head h reads kv head h div (hq / hkv)
  (a kv head whose values are all zero silences exactly its own q heads), and
  the gated attention output equals torch's fp64 scaled-dot-product attention
  over the stored cache with the kv heads repeated per group;
* the Gated DeltaNet output gate: out_h = RMSNorm(o_h) w (.) SiLU(z_h): z = 0
  gives exactly 0; out / SiLU(z) does not depend on z; its per-head RMS
  (divided by the gain) is 1;
* the paged KV index: a new row's K and V sit at [layer][page][head][slot][:]
  of the pool, as the C header documents, equal to the binary16 rounding of
  RoPE(W_k u) and of W_v u.

Each pin is also run against a copy of the oracle with one mistake planted
(reversed conv taps; the history shifted the other way; GDN heads grouped by
h mod hk; attention heads grouped by h mod hkv; the gate applied before the
norm; SiLU replaced by a sigmoid in the gate; head and slot swapped in the KV
index), and must fail on it (tests named *_catches_*).

Models: the tiny widths (hidden 256 = hq * dh = hv * dv), two layers, with
the second layer made silent (zero Q4 output projections decode to exactly
0), W_o the identity and zero FFN weights, so that the final hidden state is
the embedding plus exactly the first layer's mixer output.
"""
import math

import numpy as np
import pytest
import torch

from gen import configs, synth
from oracle import oracle as orc

GDN, FA = configs.GDN, configs.FA
EPS = 1e-6

# ---------------------------------------------------------------- builders


def _identity_q4(n):
    """n x n identity in the Q4 format: per row one super-block holds the 1 as
    d = 1.0, scale 1 and code 1 in its sub-block, every other scale 0."""
    nsb = n // 256
    out = np.zeros((n, nsb * 144), np.uint8)
    for r in range(n):
        sb, kk = divmod(r, 256)
        j, i = divmod(kk, 32)
        blk = out[r, sb * 144:(sb + 1) * 144]
        blk[0:2] = np.frombuffer((0x3C00).to_bytes(2, "little"), np.uint8)  # d = 1.0
        field = 1 << (6 * j)  # scale 1 for sub-block j, every min 0
        blk[4:16] = np.frombuffer(field.to_bytes(12, "little"), np.uint8)
        if i < 16:
            blk[16 + 16 * j + i] = 1
        else:
            blk[16 + 16 * j + i - 16] = 1 << 4
    return out


def _deq(m):
    """fp64 dequantised Q4 matrix (the decoder is pinned on hand-built blocks)."""
    rows = m.shape[0]
    return orc.q4_decode(m).reshape(rows, -1)


def _rms(x, g):
    return x / math.sqrt(float(np.mean(x * x)) + EPS) * g


def _l2(x):
    return x / math.sqrt(float(np.sum(x * x)) + EPS)


def _silu(x):
    return x / (1.0 + np.exp(-x))


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _model(kinds, **kw):
    m = dict(configs.TINY)
    m.update(name="pin", n_layers=len(kinds), kinds=list(kinds), vocab=64, hkv=2)
    m.update(kw)
    return m


def _silence(w, li):
    """Zero layer li's mixer output projection and FFN: it adds exactly 0."""
    w[f"layers.{li}.w_o"] = np.zeros_like(w[f"layers.{li}.w_o"])
    for n in ("w_gate", "w_up", "w_down"):
        w[f"layers.{li}.{n}"] = np.zeros_like(w[f"layers.{li}.{n}"])


def _setup(kinds, seed=5, kv_q8=0, cached=40, jitter=0.1, **kw):
    m = _model(kinds, **kw)
    w = synth.make_weights(m, seed, jitter, nthreads=2)
    for li in range(len(kinds)):
        _silence(w, li)
    w["layers.0.w_o"] = _identity_q4(m["hidden"])
    n_pages = 8
    pool = synth.make_pool(m, n_pages, kv_q8)
    synth.fill_pool(pool, seed + 1)
    S, conv = synth.make_seq_states(m, seed + 2, 0)
    pages = np.array([3, 6, 1], np.int32)[: (cached + 15) // 16 + 1]
    return m, w, pool, S, conv, pages


def _run(m, w, pool, S, conv, pages, cached, token, kv_q8=0, library=None):
    o = orc.Oracle(m, w, pool, kv_q8, 8, 2, nthreads=1, library=library)
    o.seq_set(0, cached, pages[: (cached + 15) // 16], S, conv)
    r = o.step([token], [cached], [0], want_logits=False, want_hidden=True)
    o.commit([0], [1])
    st = o.seq_get(0)
    return r["hidden"][0], st


def _u(m, w, token, layer=0):
    x0 = _deq(w["embed"][token:token + 1])[0]
    return x0, _rms(x0, w[f"layers.{layer}.attn_norm"].astype(np.float64))


# ------------------------------------------------------ GDN conv and grouping


def check_gdn_conv_and_grouping(tap, library=None):
    kinds = [GDN, FA]
    m, w, pool, S, conv, pages = _setup(kinds)
    d = configs.model_dims(m)
    C, hk, hv, dk, dv = d["conv_ch"], m["hk"], m["hv"], m["dk"], m["dv"]
    qk = hk * dk
    taps = np.zeros((C, 4), np.float32)
    taps[:, tap] = 1.0
    w["layers.0.conv_w"] = taps
    S0 = np.zeros_like(S)
    rng = np.random.default_rng(17)
    H0 = rng.standard_normal(conv.shape).astype(np.float32)
    token, cached = 9, 40
    _h, st = _run(m, w, pool, S0, H0, pages, cached, token, library=library)
    _x0, u = _u(m, w, token)
    pre = _deq(w["layers.0.w_qkv"]) @ u
    window = [H0[0, 0].astype(np.float64), H0[0, 1].astype(np.float64), H0[0, 2].astype(np.float64), pre]
    c = _silu(window[tap])  # one-hot tap `tap` selects the input 3 - tap rows back
    beta = _sigmoid(_deq(w["layers.0.w_b"]) @ u)
    per = hv // hk
    for h in range(hv):
        g = h // per
        k = _l2(c[qk + g * dk: qk + (g + 1) * dk])
        v = c[2 * qk + h * dv: 2 * qk + (h + 1) * dv]
        want = beta[h] * np.outer(v, k)
        got = st["S"][0, h]
        assert np.max(np.abs(got - want)) <= 1e-12 * max(1.0, np.max(np.abs(want))), f"v-head {h}"
    hist = st["conv"][0]
    want_hist = np.stack([window[1], window[2], pre])
    assert np.max(np.abs(hist - want_hist)) <= 1e-12 * np.max(np.abs(want_hist)), "conv history"


@pytest.mark.parametrize("tap", [0, 1, 2, 3])
def test_gdn_conv_taps_history_and_grouping(tap):
    check_gdn_conv_and_grouping(tap)


_REVERSED_TAPS = [
    ("acc += lw.conv_w[ch * cw + t] * hist[t * conv_ch + ch];",
     "acc += lw.conv_w[ch * cw + (cw - 1 - t)] * hist[t * conv_ch + ch];"),
    ("acc += lw.conv_w[ch * cw + cw - 1] * pre[ch];", "acc += lw.conv_w[ch * cw + 0] * pre[ch];"),
]
_HISTORY_NEWEST_FIRST = [
    ("for (int t = 0; t < cw - 1; ++t) acc += lw.conv_w[ch * cw + t] * hist[t * conv_ch + ch];",
     "for (int t = 0; t < cw - 1; ++t) acc += lw.conv_w[ch * cw + t] * hist[(cw - 2 - t) * conv_ch + ch];"),
    ("for (int t = 0; t + 1 < cw - 1; ++t) hist[t * conv_ch + ch] = hist[(t + 1) * conv_ch + ch];\n"
     "                    hist[(cw - 2) * conv_ch + ch] = pre[ch];",
     "for (int t = cw - 2; t > 0; --t) hist[t * conv_ch + ch] = hist[(t - 1) * conv_ch + ch];\n"
     "                    hist[0 * conv_ch + ch] = pre[ch];"),
]
_GDN_MOD_GROUPING = [("const int g = h / per;", "const int g = h % L.hk;")]


def test_gdn_pin_catches_reversed_taps(tmp_path):
    lib = orc.build_variant(_REVERSED_TAPS, str(tmp_path))
    with pytest.raises(AssertionError):
        check_gdn_conv_and_grouping(0, library=lib)


def test_gdn_pin_catches_history_kept_newest_first(tmp_path):
    """Reading and writing the history newest-first is self-consistent (every
    T-row and replay check passes), but the stored order is not the
    documented one."""
    lib = orc.build_variant(_HISTORY_NEWEST_FIRST, str(tmp_path))
    with pytest.raises(AssertionError):
        check_gdn_conv_and_grouping(2, library=lib)


def test_gdn_pin_catches_mod_grouping(tmp_path):
    lib = orc.build_variant(_GDN_MOD_GROUPING, str(tmp_path))
    with pytest.raises(AssertionError):
        check_gdn_conv_and_grouping(3, library=lib)


# ------------------------------------------------------------ GDN output gate


def check_gdn_output_gate(library=None):
    kinds = [GDN, FA]
    m, w, pool, S, conv, pages = _setup(kinds)
    hv, dv = m["hv"], m["dv"]
    token, cached = 21, 40
    x0, u = _u(m, w, token)
    # z = 0 (zero W_z): SiLU(0) = 0 silences the whole mixer, exactly
    w0 = dict(w)
    w0["layers.0.w_z"] = np.zeros_like(w["layers.0.w_z"])
    h0, _ = _run(m, w0, pool, S, conv, pages, cached, token, library=library)
    assert np.array_equal(h0, x0), "z = 0 must give exactly zero mixer output"
    # two different W_z: out / SiLU(z) is RMSNorm(o) w, the same for both
    ratios = []
    for seed in (101, 202):
        wz = synth.q4_matrix(seed, 7, hv * dv, m["hidden"], 0.05)
        ww = dict(w)
        ww["layers.0.w_z"] = wz
        h, _ = _run(m, ww, pool, S, conv, pages, cached, token, library=library)
        out = h - x0
        z = _deq(wz) @ u
        gate = _silu(z)
        keep = np.abs(gate) > 1e-3 * np.max(np.abs(gate))
        ratios.append((out, gate, keep))
    (o1, g1, k1), (o2, g2, k2) = ratios
    both = k1 & k2
    r1, r2 = o1[both] / g1[both], o2[both] / g2[both]
    assert np.max(np.abs(r1 - r2)) <= 1e-9 * np.max(np.abs(r1)), "out / SiLU(z) depends on z"
    # per head, RMSNorm(o) has unit RMS (up to eps): out / (SiLU(z) w), taking
    # each element from whichever W_z gives it the larger gate
    gain = w["layers.0.o_norm"].astype(np.float64)
    full = np.where(np.abs(g1) >= np.abs(g2), o1 / g1, o2 / g2) / np.tile(gain, hv)  # one gain per head dim
    assert np.min(np.maximum(np.abs(g1), np.abs(g2))) > 1e-6
    for h in range(hv):
        seg = full[h * dv:(h + 1) * dv]
        assert abs(math.sqrt(float(np.mean(seg * seg))) - 1.0) <= 1e-4, f"head {h} norm"


def test_gdn_output_gate():
    check_gdn_output_gate()


_GATE_BEFORE_NORM = [
    ("rmsnorm(&o[h * L.dv], lw.o_norm, L.dv, L.eps, &on[h * L.dv]);\n"
     "                    for (int i = 0; i < L.dv; ++i) on[h * L.dv + i] *= silu(z[h * L.dv + i]);",
     "for (int i = 0; i < L.dv; ++i) o[h * L.dv + i] *= silu(z[h * L.dv + i]);\n"
     "                    rmsnorm(&o[h * L.dv], lw.o_norm, L.dv, L.eps, &on[h * L.dv]);"),
]
_SIGMOID_GATE = [("on[h * L.dv + i] *= silu(z[h * L.dv + i]);", "on[h * L.dv + i] *= sigmoid(z[h * L.dv + i]);")]


def test_gate_pin_catches_gate_before_norm(tmp_path):
    lib = orc.build_variant(_GATE_BEFORE_NORM, str(tmp_path))
    with pytest.raises(AssertionError):
        check_gdn_output_gate(library=lib)


def test_gate_pin_catches_sigmoid_gate(tmp_path):
    lib = orc.build_variant(_SIGMOID_GATE, str(tmp_path))
    with pytest.raises(AssertionError):
        check_gdn_output_gate(library=lib)


# ------------------------------------------------- attention head grouping


def _rope(x, pos, base):
    """Rotate-half RoPE over the whole head: pairs (i, i + dh/2), angle
    pos * base^(-2i/dh)."""
    dh = x.shape[-1]
    i = np.arange(dh // 2)
    th = pos * base ** (-2.0 * i / dh)
    a, b = x[..., : dh // 2], x[..., dh // 2:]
    return np.concatenate([a * np.cos(th) - b * np.sin(th), a * np.sin(th) + b * np.cos(th)], axis=-1)


def check_attention_grouping(library=None):
    kinds = [FA, GDN]
    m, w, pool, S, conv, pages = _setup(kinds)
    hq, hkv, dh, H = m["hq"], m["hkv"], m["dh"], m["hidden"]
    grp = hq // hkv
    # kv head 0 holds zero values: cached V and this row's W_v rows
    pool["v"][0, :, 0] = 0
    wv = w["layers.0.w_v"].copy()
    wv[:dh] = 0
    w["layers.0.w_v"] = wv
    token, cached = 33, 40
    snapshot = {k: v.copy() for k, v in pool.items()}
    h, st = _run(m, w, pool, S, conv, pages, cached, token, library=library)
    x0, u = _u(m, w, token)
    out = (h - x0).reshape(hq, dh)
    for qh in range(hq):
        silent = qh // grp == 0
        if silent:
            assert np.all(out[qh] == 0.0), f"q head {qh} reads a nonzero kv head"
        else:
            assert np.max(np.abs(out[qh])) > 1e-6, f"q head {qh} reads the zero kv head"
    # the whole gated output against torch SDPA with repeated kv heads
    q = (_deq(w["layers.0.w_q"]) @ u).reshape(hq, dh)
    gate = _sigmoid(_deq(w["layers.0.w_g"]) @ u).reshape(hq, dh)
    k_new = (_deq(w["layers.0.w_k"]) @ u).reshape(hkv, dh)
    v_new = (_deq(w["layers.0.w_v"]) @ u).reshape(hkv, dh)
    base = m["rope_base"]
    qr = _rope(q, cached, base)
    kr = _rope(k_new, cached, base)
    K = np.zeros((hkv, cached + 1, dh))
    V = np.zeros((hkv, cached + 1, dh))
    for p in range(cached):
        pg, sl = pages[p // 16], p % 16
        K[:, p] = snapshot["k"][0, pg, :, sl].view(np.float16).astype(np.float64)
        V[:, p] = snapshot["v"][0, pg, :, sl].view(np.float16).astype(np.float64)
    K[:, cached] = kr.astype(np.float16).astype(np.float64)
    V[:, cached] = v_new.astype(np.float16).astype(np.float64)
    Kr = torch.from_numpy(np.repeat(K, grp, axis=0))  # kv head of q head h: h div grp
    Vr = torch.from_numpy(np.repeat(V, grp, axis=0))
    att = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(qr)[:, None, :], Kr, Vr)
    want = att[:, 0, :].numpy() * gate
    assert np.max(np.abs(out - want)) <= 1e-9 * max(1.0, np.max(np.abs(want))), "gated attention output"


def test_attention_head_grouping():
    check_attention_grouping()


_ATTN_MOD_GROUPING = [("for (int h = kh * group; h < (kh + 1) * group; ++h)",
                       "for (int h = kh; h < L.hq; h += L.hkv)")]


def test_attention_pin_catches_mod_grouping(tmp_path):
    lib = orc.build_variant(_ATTN_MOD_GROUPING, str(tmp_path))
    with pytest.raises(AssertionError):
        check_attention_grouping(library=lib)


# --------------------------------------------------------------- KV index


def check_kv_index(kv_q8, library=None):
    kinds = [FA, GDN]
    m, w, pool, S, conv, pages = _setup(kinds, kv_q8=kv_q8)
    hkv, dh = m["hkv"], m["dh"]
    token, cached = 45, 37  # position 37: page index 2, slot 5
    _run(m, w, pool, S, conv, pages, cached, token, kv_q8=kv_q8, library=library)
    _x0, u = _u(m, w, token)
    k = _rope((_deq(w["layers.0.w_k"]) @ u).reshape(hkv, dh), cached, m["rope_base"])
    v = (_deq(w["layers.0.w_v"]) @ u).reshape(hkv, dh)
    pg, sl = pages[cached // 16], cached % 16
    for head in range(hkv):
        for name, want in (("k", k[head]), ("v", v[head])):
            if not kv_q8:
                got = pool[name][0, pg, head, sl].view(np.float16).astype(np.float64)
                assert np.max(np.abs(got - want)) <= 2.0 ** -11 * np.max(np.abs(want)), f"{name} head {head}"
            else:
                codes = pool[name + "q"][0, pg, head, sl].astype(np.float64)
                sc = pool[name + "s"][0, pg, head, sl].view(np.float16).astype(np.float64)
                got = codes * np.repeat(sc, 32)
                assert np.all(np.abs(got - want) <= 0.5 * np.repeat(sc, 32) * 1.001 + 1e-12), f"{name} head {head}"


@pytest.mark.parametrize("kv_q8", [0, 1])
def test_kv_index_matches_documented_layout(kv_q8):
    check_kv_index(kv_q8)


_KV_HEAD_SLOT_SWAPPED = [
    ("return ((((static_cast<size_t>(kvl) * L.n_pages + page) * L.hkv + head) * L.page_tokens + slot) * L.dh) + d;",
     "return ((((static_cast<size_t>(kvl) * L.n_pages + page) * L.page_tokens + slot) * L.hkv + head) * L.dh) + d;"),
]


def test_kv_pin_catches_head_slot_swap(tmp_path):
    lib = orc.build_variant(_KV_HEAD_SLOT_SWAPPED, str(tmp_path))
    with pytest.raises(AssertionError):
        check_kv_index(0, library=lib)
