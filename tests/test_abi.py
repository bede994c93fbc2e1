"""The C-ABI library loads, exports every symbol include/mk.h declares, and
its host-only size queries agree with the documented buffer layouts. No
compute call here needs a GPU."""
import ctypes
import os
import re

import pytest

from gen import configs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mk():
    from speculative_decode_persistent_gb300 import build as b
    b.build()
    from speculative_decode_persistent_gb300 import mk as m
    return m


def _declared():
    src = open(os.path.join(ROOT, "include", "mk.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mk_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(mk):
    names = _declared()
    assert len(names) >= 18
    for n in names:
        assert hasattr(mk.lib, n), n
        assert n in mk.EXPORTS, n


def test_size_queries_tiny(mk):
    m = configs.TINY
    L = mk.make_layout(m, kv_q8=0, n_pages=64, max_seqs=8)
    p = ctypes.byref(L)
    d = configs.model_dims(m)
    assert mk.lib.mk_kv_bytes(p) == d["n_fa"] * 64 * m["hkv"] * 16 * m["dh"] * 2
    assert mk.lib.mk_kv_scale_bytes(p) == 0
    assert mk.lib.mk_gdn_state_bytes(p) == 8 * 9 * d["n_gdn"] * m["hv"] * m["dv"] * m["dk"] * 4
    assert mk.lib.mk_conv_state_bytes(p) == 8 * 9 * d["n_gdn"] * 3 * d["conv_ch"] * 4
    # packed weights: every streamed matrix in 4608-byte units of 32 rows
    # (rows padded to 32) plus the embedding copy and the fp32 parameters
    assert mk.lib.mk_packed_bytes(p) > 0
    Lq = mk.make_layout(m, kv_q8=1, n_pages=64, max_seqs=8)
    assert mk.lib.mk_kv_bytes(ctypes.byref(Lq)) == d["n_fa"] * 64 * m["hkv"] * 16 * m["dh"]
    assert mk.lib.mk_kv_scale_bytes(ctypes.byref(Lq)) == d["n_fa"] * 64 * m["hkv"] * 16 * (m["dh"] // 32) * 2


def test_packed_bytes_27b_close_to_q4_size(mk):
    m = configs.QWEN27
    L = mk.make_layout(m, kv_q8=0, n_pages=320, max_seqs=1)
    n = mk.lib.mk_packed_bytes(ctypes.byref(L))
    streamed = 0
    for name, _tid, kind, shape in configs.tensor_inventory(m):
        if kind == "q4" and name != "embed":
            streamed += shape[0] * shape[1] * 0.5625
    embed = m["vocab"] * m["hidden"] * 0.5625
    assert streamed + embed <= n <= (streamed + embed) * 1.01


def test_layout_rejections(mk):
    for key, bad in [("hidden", 300), ("dh", 48), ("dk", 96), ("conv_w", 3)]:
        m = dict(configs.TINY)
        m[key] = bad
        if key == "dk":
            m["dv"] = 64
        L = mk.make_layout(m, kv_q8=0, n_pages=64)
        assert mk.lib.mk_packed_bytes(ctypes.byref(L)) == 0, key
    L = mk.make_layout(configs.TINY, kv_q8=0, n_pages=64, max_seqs=9)
    assert mk.lib.mk_packed_bytes(ctypes.byref(L)) == 0


def test_status_strings(mk):
    for code in mk.STATUS:
        assert mk.lib.mk_status_str(code)


def test_mtp_layout_sizes_and_rejections(mk):
    """With an MTP head the pool gains one KV layer and the packed buffer the
    head's matrices (W_fc 2H->H and one gated-attention layer); n_draft and
    draft_vocab are range-checked."""
    m = dict(configs.QWEN27, has_mtp=1, draft_vocab=32768)
    base = mk.make_layout(configs.QWEN27, kv_q8=0, n_pages=320, max_seqs=1)
    L = mk.make_layout(m, kv_q8=0, n_pages=320, max_seqs=1, n_draft=4)
    d = configs.model_dims(m)
    assert mk.lib.mk_kv_bytes(ctypes.byref(L)) == (d["n_fa"] + 1) * 320 * m["hkv"] * 16 * m["dh"] * 2
    H, F = m["hidden"], m["ffn"]
    head = (H * 2 * H + (2 * d["fa_q"] + 2 * d["fa_kv"]) * H + H * d["fa_q"] + 3 * F * H) * 0.5625
    extra = mk.lib.mk_packed_bytes(ctypes.byref(L)) - mk.lib.mk_packed_bytes(ctypes.byref(base))
    assert head <= extra <= head * 1.01
    for kw in (dict(n_draft=0), dict(n_draft=mk.MK_MAX_T)):
        bad = mk.make_layout(m, kv_q8=0, n_pages=320, max_seqs=1, **kw)
        assert mk.lib.mk_packed_bytes(ctypes.byref(bad)) == 0, kw
    bad = mk.make_layout(dict(m, draft_vocab=m["vocab"] + 1), kv_q8=0, n_pages=320, max_seqs=1, n_draft=4)
    assert mk.lib.mk_packed_bytes(ctypes.byref(bad)) == 0


def test_engine_refuses_q8_head_dim_192():
    from gen import configs
    from speculative_decode_persistent_gb300 import mk
    model = dict(configs.TINY, dh=192, hq=2, hkv=1)
    with pytest.raises(mk.MkError) as e:
        mk.Engine(model, {}, 1, 64)
    assert e.value.status == -8
